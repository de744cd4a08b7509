// Per-sequence decisions from the streaming pass's per-warp partials.
//
// Sources: "Speculative decoding: guess a few tokens first - why the answer
// stays the same", section "What happens in one round" step 3 (accept x_i
// with probability min(1, p_i(x_i)/q_i(x_i)), left to right, the first
// rejection voiding the rest) and its greedy paragraph (accept while the
// draft equals the target argmax); "AdaPLD: adaptive retrieval and reuse for
// efficient model-free speculative decoding", section 3.3 and Algorithm 1
// (VerifyAndAccept over the draft tree).
//
// A decision is taken by a group of NT threads (a whole CTA: 256 threads, 512
// for sampling, 1024 for greedy chains and trees) synchronised on named
// barrier 1; gt is the thread's index in the group.
// Each runs in its own kernel, one CTA per sequence (sv_argmax.cu for greedy
// chains and trees, sv_sample.cu for sampling).
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr int kGroup = kThreads;                 // 256
constexpr int kMaxGamma = 256;                   // sampling: rows per sequence <= 513
constexpr int kMaxNodes = 1024;                  // greedy chains and trees: rows <= 1024

enum : int { kModeSample = 0, kModeGreedy = 1, kModeTree = 2,
             kModeTopK2 = 3, kModeTopK4 = 4, kModeTopK8 = 5,
             kModeLazy = 6 };     // sampling statistics of one position group (lazy pass)

// List length of a top-K streaming mode (0 for the other modes).
__host__ __device__ constexpr int topk_of(int mode) {
    return mode == kModeTopK2 ? 2 : mode == kModeTopK4 ? 4 : mode == kModeTopK8 ? 8 : 0;
}

// Row-statistics partials take their exponent arguments as z s - fl(m s)
// while |fl(m s)| < kFmaArgLimit (2^24: the rounding residual of m s is then
// at most 1 in magnitude), else as (z - m) s.
constexpr float kFmaArgLimit = 16777216.f;

// The residual m s - fl(m s) that a partial with maximum m carries in every
// exponent (0 for partials past the limit).
__device__ __forceinline__ float partial_residual(float m, float s) {
    const float ms = m * s;
    return fabsf(ms) < kFmaArgLimit ? fmaf(m, s, -ms) : 0.f;
}

struct VerifyArgs {
    const char* zt;            // target logits
    const char* zd;            // draft logits (sampling)
    const int32_t* x;          // draft tokens (chains) / node tokens (trees)
    const int32_t* par;        // parents (trees)
    const float* u;            // uniforms (sampling)
    float T, invT, s, s_lo;    // temperature, 1/T, log2(e)/T as a float-float pair (s, s_lo)
    int gamma;                 // drafts per sequence (chains)
    int rows_per_seq;          // 2*gamma+1 (sampling), gamma+1 (greedy), N (tree)
    int V, nseg;
    long long total_chunks;
    int B;
    int C;                     // sampling: final-pass chunks per row
    int early_inputs;          // sampling: the decide kernel follows this call's own stream, so it
                               // may load the call's inputs before griddepcontrol.wait
    float2* parts;             // per-warp-chunk partials
    unsigned long long* desc;  // sampling: [B] SampleDescs as kDescWords tagged words
    unsigned long long epoch;  // sampling: this call's launch tag (kClaimTagBits bits, nonzero)
    uint32_t ptag;             // sampling: this call's tag for tagged words (nonzero)
    int poll_parts;            // sampling: the decide step runs beside the stream and waits for
                               // each sequence's tagged partials instead of the whole stream
    unsigned long long* tick;  // sampling: per-sequence count of finished final-pass chunks,
                               // (epoch << kClaimIdxBits) | count
    unsigned long long* sums;  // sampling: [B, C, 8] segments' sums as kSumWords tagged words:
                               // Za, Zb (float-float), and after a rejection the residual sum W
                               // at the desc's ratio rt (float-float) and its slope D
    int* err;
    int32_t* out_tok;
    int32_t* out_acc;
    float* out_lp;             // sampling, nullable
    int32_t* out_nodes;        // trees
    // Lazy sampling, one position group per stream + decide pair: target rows
    // of positions [lz_lo, lz_lo + lz_nt) and draft rows of [lz_lo, lz_lo + lz_nd)
    // of the sequences in lz_list[0 .. *lz_count) (every sequence, in order,
    // when lz_list is null); the decide step appends the sequences that accept
    // every draft of the group to lz_next_list / lz_next_count.  The first
    // group's stream zeroes the lz_nzero counts at lz_zero.
    int lz_lo, lz_nt, lz_nd, lz_nzero;
    const int* lz_list;
    const int* lz_count;
    int* lz_next_list;
    int* lz_next_count;
    int* lz_zero;
    // Polls of a bounded wait on a ring barrier before it reports
    // SPEC_DEVERR_TIMEOUT (kWaitLimit unless a test lowers it); the wait for a
    // CTA's own copies in flight before it exits always takes kWaitLimit.
    uint32_t wait_limit;
    // Ring streams: the workspace's claim counter and this launch's tag,
    // already shifted into place (tag << kClaimIdxBits); set by launch_stream.
    unsigned long long* claim;
    unsigned long long claim_tag;
};

// Partial i of a row-statistics stream: sampling stores them as tagged
// 64-bit word pairs (the float in each word's low half), the other modes as
// float2.
template <bool TAGGED>
__device__ __forceinline__ float2 load_part(const VerifyArgs& a, size_t i) {
    if constexpr (TAGGED) {
        const ulonglong2 q = __ldcg(reinterpret_cast<const ulonglong2*>(a.parts) + i);
        return make_float2(__uint_as_float((uint32_t)q.x), __uint_as_float((uint32_t)q.y));
    } else {
        return __ldcg(a.parts + i);
    }
}

__device__ __forceinline__ void group_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// The same barrier for a group of NT threads.
template <int NT>
__device__ __forceinline__ void group_sync_n() { asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory"); }

// Row r of sequence b of a sampling batch: r <= gamma is target row r, r > gamma
// is draft row r-gamma-1.
__device__ __forceinline__ const char* sample_row(const VerifyArgs& a, int b, int r, size_t rowbytes) {
    return r <= a.gamma ? a.zt + ((size_t)b * (a.gamma + 1) + r) * rowbytes
                        : a.zd + ((size_t)b * a.gamma + (r - a.gamma - 1)) * rowbytes;
}

// ---------------------------------------------------------------- sampling
struct SampleDecideSmem {
    float M[2 * kMaxGamma + 1];       // row max
    float lnZ[2 * kMaxGamma + 1];     // ln sum exp((z - M)/T)
    float lp[kMaxGamma], lq[kMaxGamma];
    int bad, k;
};

// Rows r[0..RB) of sequence b from their warp partials (one warp, every lane
// gets the results; rows at or past rows_per_seq are skipped): M = max m_p and
// lnZ = ln sum_p Z_p 2^((m_p - M) s - r_p), with r_p = partial_residual(m_p)
// (float-float sum).  Each lane holds up to KH partials of each row in
// registers, all rows' loads in flight together, and adds a row's partials in
// increasing p whatever RB and KH are, so every row's result is bit-identical
// across batch shapes.  lnZ is 0 for a row without a finite logit.
template <int RB, int KH, bool TAGGED = false>
__device__ __forceinline__ void merge_rows_stats(const VerifyArgs& a, int b, const int (&r)[RB], int lane,
                                                 float (&Mout)[RB], float (&lnZout)[RB]) {
    const int P = a.nseg * kWarps;
    float2 q[RB][KH];
#pragma unroll
    for (int j = 0; j < RB; ++j) {
        const size_t pr = ((size_t)b * a.rows_per_seq + r[j]) * P;
#pragma unroll
        for (int h = 0; h < KH; ++h) {
            const int p = lane + 32 * h;
            q[j][h] = (r[j] < a.rows_per_seq && p < P) ? load_part<TAGGED>(a, pr + p) : make_float2(kNegInf, 0.f);
        }
    }
#pragma unroll
    for (int j = 0; j < RB; ++j) {
        if (r[j] >= a.rows_per_seq) continue;             // warp-uniform
        const size_t pr = ((size_t)b * a.rows_per_seq + r[j]) * P;
        float m = kNegInf;
#pragma unroll
        for (int h = 0; h < KH; ++h) m = fmaxf(m, q[j][h].x);
        for (int p = lane + 32 * KH; p < P; p += 32) m = fmaxf(m, load_part<TAGGED>(a, pr + p).x);
        m = warp_max(m);
        FF z{0.f, 0.f};
        if (m != kNegInf) {
#pragma unroll
            for (int h = 0; h < KH; ++h)
                if (q[j][h].x != kNegInf)
                    ff_add(z, q[j][h].y * ex2_approx(fmaf(q[j][h].x - m, a.s, -partial_residual(q[j][h].x, a.s))));
            for (int p = lane + 32 * KH; p < P; p += 32) {
                const float2 t = load_part<TAGGED>(a, pr + p);
                if (t.x != kNegInf)
                    ff_add(z, t.y * ex2_approx(fmaf(t.x - m, a.s, -partial_residual(t.x, a.s))));
            }
        }
        z = ff_norm(warp_sum_ff(z));
        Mout[j] = m;
        lnZout[j] = m == kNegInf ? 0.f : logf(z.hi) + z.lo / z.hi;
    }
}

// One row, eight partials per lane in registers: the same sums as
// merge_rows_stats, written out for the sampling decide (a template-built
// version of this one-row merge measured 4 us slower in the chained
// chain-b64 step, with the same registers and shared memory).
template <bool TAGGED = false>
__device__ __forceinline__ void merge_row_stats(const VerifyArgs& a, int b, int r, int lane,
                                                float* Mout, float* lnZout) {
    constexpr int kHeld = 8;
    const int P = a.nseg * kWarps;
    const size_t pr = ((size_t)b * a.rows_per_seq + r) * P;
    float2 q[kHeld];
#pragma unroll
    for (int h = 0; h < kHeld; ++h) {
        const int p = lane + 32 * h;
        q[h] = p < P ? load_part<TAGGED>(a, pr + p) : make_float2(kNegInf, 0.f);
    }
    float m = kNegInf;
#pragma unroll
    for (int h = 0; h < kHeld; ++h) m = fmaxf(m, q[h].x);
    for (int p = lane + 32 * kHeld; p < P; p += 32) m = fmaxf(m, load_part<TAGGED>(a, pr + p).x);
    m = warp_max(m);
    FF z{0.f, 0.f};
    if (m != kNegInf) {
#pragma unroll
        for (int h = 0; h < kHeld; ++h)
            if (q[h].x != kNegInf)
                ff_add(z, q[h].y * ex2_approx(fmaf(q[h].x - m, a.s, -partial_residual(q[h].x, a.s))));
        for (int p = lane + 32 * kHeld; p < P; p += 32) {
            const float2 t = load_part<TAGGED>(a, pr + p);
            if (t.x != kNegInf)
                ff_add(z, t.y * ex2_approx(fmaf(t.x - m, a.s, -partial_residual(t.x, a.s))));
        }
    }
    z = ff_norm(warp_sum_ff(z));
    *Mout = m;
    *lnZout = m == kNegInf ? 0.f : logf(z.hi) + z.lo / z.hi;
}

// Rows [0, n) of sequence b given by row(q), the warps of an NT-thread group
// sharing them: a row per warp and round while they fit, else four rows per
// warp and round.  Stores (M, lnZ) of row q at M[q], lnZ[q].
template <int NT, typename RowOf>
__device__ __forceinline__ void merge_rows_group(const VerifyArgs& a, int b, int n, RowOf row, int gt,
                                                 float* M, float* lnZ) {
    constexpr int NW = NT / 32;
    const int lane = gt & 31, gw = gt >> 5;
    if (n <= NW) {
        if (gw < n) {
            float m, l;
            merge_row_stats(a, b, row(gw), lane, &m, &l);
            if (lane == 0) { M[gw] = m; lnZ[gw] = l; }
        }
        return;
    }
    constexpr int RB = 4;
    for (int q0 = gw; q0 < n; q0 += NW * RB) {
        int rr[RB];
#pragma unroll
        for (int j = 0; j < RB; ++j) rr[j] = q0 + NW * j < n ? row(q0 + NW * j) : a.rows_per_seq;
        float m[RB], l[RB];
        merge_rows_stats<RB, 4>(a, b, rr, lane, m, l);
        if (lane == 0)
#pragma unroll
            for (int j = 0; j < RB; ++j)
                if (q0 + NW * j < n) { M[q0 + NW * j] = m[j]; lnZ[q0 + NW * j] = l[j]; }
    }
}

// ln p(x) = (z_x - M)/T - lnZ for a row with max M and normaliser lnZ.
__device__ __forceinline__ float row_log_prob(float zx, float M, float lnZ, const VerifyArgs& a) {
    return (zx - M) / a.T - lnZ;
}

// The accept test u < p(x)/q(x) from the two log-probabilities (p = 0
// rejects, q = 0 with p > 0 accepts).
__device__ __forceinline__ bool accept_draft(float lp, float lq, float u) {
    float r;
    if (lp == kNegInf) r = 0.f;
    else if (lq == kNegInf) r = CUDART_INF_F;
    else r = expf(lp - lq);
    return u < r;
}

// Sampling call whose decide kernel runs beside the stream: wait (bounded)
// until every partial of sequence b carries this call's tag.  One thread
// first polls the partial the stream reaches last for this sequence (the
// last warp of its last chunk: the stream advances through the chunks in
// index order), then every thread checks its share and the check repeats
// until no partial is stale.  The whole CTA (NT threads) takes part.
template <int NT>
__device__ void wait_seq_parts(const VerifyArgs& a, int b, int gt) {
    const size_t n = (size_t)a.rows_per_seq * a.nseg * kWarps;
    const unsigned long long* base = reinterpret_cast<const unsigned long long*>(a.parts) + 2 * (size_t)b * n;
    const unsigned long long tag = (unsigned long long)a.ptag;
    auto fresh = [&](size_t i) {
        unsigned long long x, y;
        asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(x), "=l"(y) : "l"(base + 2 * i) : "memory");
        return (x >> 32) == tag && (y >> 32) == tag;
    };
    if (gt == 0)
        for (uint32_t i = 0; !fresh(n - 1); ++i) {
            if (i >= a.wait_limit) {
                atomicOr(a.err, SPEC_DEVERR_TIMEOUT);
                break;
            }
            __nanosleep(200);
        }
    __syncthreads();
    for (uint32_t round = 0;; ++round) {
        int stale = 0;
        for (size_t i = gt; i < n; i += NT) stale |= !fresh(i);
        if (!__syncthreads_or(stale)) break;
        if (round >= a.wait_limit) {
            if (gt == 0) atomicOr(a.err, SPEC_DEVERR_TIMEOUT);
            break;
        }
        __nanosleep(200);
    }
}

// Row statistics from the partials (M = max m_p, Z = sum Z_p 2^((m_p - M) s),
// float-float) and the accept decisions u_i < p_i(x_i)/q_i(x_i) in single
// precision (GB300's double-precision rate is a small fraction of its float
// rate): ln p_i(x_i) and ln q_i(x_i) carry errors of ~1e-6, far inside the
// 1e-4 decision margin and the 1e-5 bar on returned probabilities.  Every
// position's test runs on its own thread; the first rejection is the smallest
// rejected index.  Returns the rejection index k (gamma when every draft is
// accepted, -1 for bad input) in every thread and leaves the row statistics
// in sm.
template <int ELT, int NT>
__device__ int decide_sample(const VerifyArgs& a, int b, int gt, SampleDecideSmem& sm) {
    const size_t rowbytes = (size_t)a.V * ELT;
    if (!a.early_inputs) pdl_wait();   // first kernel of the call: the kernel before may write the inputs
    // Issue the gathers of z[x_i] first: their latency overlaps the merges.
    int xi = -1;
    float ztx = 0.f, zdx = 0.f;
    if (gt < a.gamma) {
        xi = a.x[(size_t)b * a.gamma + gt];
        if (xi >= 0 && xi < a.V) {
            ztx = load_logit<ELT>(sample_row(a, b, gt, rowbytes), xi);
            zdx = load_logit<ELT>(sample_row(a, b, a.gamma + 1 + gt, rowbytes), xi);
        }
    }
    const float ui = gt < a.gamma ? a.u[(size_t)b * (a.gamma + 1) + gt] : 0.f;
    if (gt == 0) {
        sm.bad = 0;
        sm.k = a.gamma;
    }
    // Everything above reads inputs only; the partials below come from the
    // stream, which may still be running.
    if (a.poll_parts) wait_seq_parts<NT>(a, b, gt);
    else pdl_wait();
    group_sync_n<NT>();
    // two rows per warp and round, both rows' loads in flight together
    constexpr int NW = NT / 32;
    for (int r0 = (gt >> 5); r0 < a.rows_per_seq; r0 += 2 * NW) {
        const int rr[2] = {r0, r0 + NW};
        float M[2], lnZ[2];
        merge_rows_stats<2, 4, true>(a, b, rr, gt & 31, M, lnZ);
        if ((gt & 31) == 0)
#pragma unroll
            for (int j = 0; j < 2; ++j)
                if (rr[j] < a.rows_per_seq) {
                    sm.M[rr[j]] = M[j];
                    sm.lnZ[rr[j]] = lnZ[j];
                }
    }
    group_sync_n<NT>();
    for (int i = gt; i < a.gamma; i += NT) {
        if (i != gt) {                                     // gamma > NT: late gathers
            xi = a.x[(size_t)b * a.gamma + i];
            if (xi >= 0 && xi < a.V) {
                ztx = load_logit<ELT>(sample_row(a, b, i, rowbytes), xi);
                zdx = load_logit<ELT>(sample_row(a, b, a.gamma + 1 + i, rowbytes), xi);
            }
        }
        if (xi < 0 || xi >= a.V) {
            atomicOr(&sm.bad, SPEC_DEVERR_TOKEN_RANGE);
            sm.lp[i] = sm.lq[i] = 0.f;
        } else {
            const float lp = row_log_prob(ztx, sm.M[i], sm.lnZ[i], a);
            const float lq = row_log_prob(zdx, sm.M[a.gamma + 1 + i], sm.lnZ[a.gamma + 1 + i], a);
            sm.lp[i] = lp;
            sm.lq[i] = lq;
            const float u = i == gt ? ui : a.u[(size_t)b * (a.gamma + 1) + i];
            if (!accept_draft(lp, lq, u)) atomicMin(&sm.k, i);
        }
    }
    for (int r = gt; r < a.rows_per_seq; r += NT)
        if (sm.M[r] == kNegInf) atomicOr(&sm.bad, SPEC_DEVERR_EMPTY_ROW);
    group_sync_n<NT>();
    return sm.bad ? -1 : sm.k;
}

// The SampleDesc of sequence b as this call's tagged words: the final pass,
// which may already run, starts on the sequence when it reads them.
__device__ __forceinline__ void publish_desc(const VerifyArgs& a, int b, const SampleDesc& d) {
    unsigned long long* p = a.desc + (size_t)kDescWords * b;
    st_tagged2(p, (uint32_t)d.k, __float_as_uint(d.mt), a.ptag);
    st_tagged2(p + 2, __float_as_uint(d.md), __float_as_uint(d.rt), a.ptag);
}

// Waits (bounded) for this call's SampleDesc of sequence b; k = -1 after a
// timeout (SPEC_DEVERR_TIMEOUT set).  One thread.
__device__ __forceinline__ SampleDesc wait_desc(const VerifyArgs& a, int b) {
    const unsigned long long* p = a.desc + (size_t)kDescWords * b;
    SampleDesc d;
    uint32_t k, mt, md, rt;
    for (uint32_t i = 0;; ++i) {
        const bool h0 = ld_tagged2(p, a.ptag, &k, &mt);
        const bool h1 = ld_tagged2(p + 2, a.ptag, &md, &rt);
        if (h0 && h1) break;
        if (i >= a.wait_limit) {
            atomicOr(a.err, SPEC_DEVERR_TIMEOUT);
            k = 0xffffffffu;
            break;
        }
        __nanosleep(100);
    }
    d.k = (int)k;
    d.mt = __uint_as_float(mt);
    d.md = __uint_as_float(md);
    d.rt = __uint_as_float(rt);
    return d;
}

// Every output of the sampling decision but the final token, and the
// SampleDesc the final-sample kernels read.
template <int NT>
static __device__ void write_sample_decision(const VerifyArgs& a, int b, int gt, int k,
                                             const SampleDecideSmem& sm) {
    if (gt == 0) {
        if (sm.bad) atomicOr(a.err, sm.bad);
        a.out_acc[b] = k;
        SampleDesc d;
        d.k = k;
        d.mt = k >= 0 ? sm.M[k] : 0.f;
        d.md = (k >= 0 && k < a.gamma) ? sm.M[a.gamma + 1 + k] : 0.f;
        d.rt = (k >= 0 && k < a.gamma) ? expf(sm.lnZ[k] - sm.lnZ[a.gamma + 1 + k]) : 0.f;
        publish_desc(a, b, d);
    }
    // accepted drafts and padding; slot k belongs to the final-pass search
    for (int i = gt; i <= a.gamma; i += NT)
        if (k < 0 || i != k)
            a.out_tok[(size_t)b * (a.gamma + 1) + i] = (k >= 0 && i < k) ? a.x[(size_t)b * a.gamma + i] : -1;
    if (a.out_lp)
        for (int i = gt; i < a.gamma; i += NT) {
            float* o = a.out_lp + ((size_t)b * a.gamma + i) * 2;
            o[0] = k >= 0 ? sm.lp[i] : CUDART_NAN_F;
            o[1] = k >= 0 ? sm.lq[i] : CUDART_NAN_F;
        }
}

// ---------------------------------------------------------- greedy and trees
struct ArgmaxDecideSmem {
    int g[kMaxNodes];                 // row argmax
    int x[kMaxNodes];                 // draft tokens (chains) / node tokens (trees)
    int par[kMaxNodes];               // trees: parents
    int k, len, bad, last;
};

// The tree walk's per-node state.
struct TreeWalkSmem {
    int up[kMaxNodes];                // ancestor pointers being doubled
    int acc[kMaxNodes];               // accepted (every node to the root matched)
    int dep[kMaxNodes];               // depth below the root
    int sub[kMaxNodes];               // deepest accepted depth in the subtree
    int key[kMaxNodes];               // (sub, lowest id) of the best child
};

// The sequence's tokens (and parents) into shared memory.  They are inputs,
// so a decide kernel loads them before waiting for the stream's partials;
// the merge that follows ends with a group barrier that publishes them.
template <int NT>
__device__ __forceinline__ void prefetch_tokens(const VerifyArgs& a, int b, int gt, bool tree,
                                                ArgmaxDecideSmem& sm) {
    const int n = tree ? a.rows_per_seq : a.gamma;
    for (int i = gt; i < n; i += NT) {
        sm.x[i] = a.x[(size_t)b * n + i];
        if (tree) sm.par[i] = a.par[(size_t)b * n + i];
    }
}

// Argmax of every row of sequence b from the (value, index) partials (every
// slot of a row is written, those past the row's end as (-inf, INT_MAX)).
// Rows of at most 32 partials share a warp: aligned groups of G lanes (G the
// power of two at or above the row's partial count), one row per group,
// reduced by xor shuffles inside the group.  Longer rows take a warp each,
// kRows rows' loads in flight at once when a warp has several rows.
template <int NT, bool MANY_ROWS = false>
__device__ __forceinline__ void merge_argmax_rows(const VerifyArgs& a, int b, int gt, int* g) {
    const int lane = gt & 31, gw = gt >> 5;
    constexpr int NW = NT / 32;
    const int P = a.nseg * kWarps, np = P;              // row stride and partials
    const int R = a.rows_per_seq;
    const size_t base = (size_t)b * R * P;                // the row partials, tagged pairs
    if (np <= 32) {
        int G = 1;
        while (G < np) G <<= 1;
        const int per = 32 / G, grp = lane / G, li = lane - grp * G;
        for (int r0 = gw * per; r0 < R; r0 += NW * per) {
            const int r = r0 + grp;
            float bv = kNegInf;
            int bi = 0x7fffffff;
            if (r < R && li < np) {
                const float2 q = load_part<true>(a, base + (size_t)r * P + li);
                bv = q.x;
                bi = __float_as_int(q.y);
            }
            for (int o = G >> 1; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (am_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
            }
            if (li == 0 && r < R) g[r] = bi;
        }
    } else if (!MANY_ROWS || R <= NW) {                   // a row per warp and round
        for (int r = gw; r < R; r += NW) {
            const size_t pr = base + (size_t)r * P;
            float bv = kNegInf;
            int bi = 0x7fffffff;
            constexpr int kHeld = 4;                       // loads in flight per lane
            for (int p0 = lane; p0 < np; p0 += 32 * kHeld) {
                float2 q[kHeld];
#pragma unroll
                for (int h = 0; h < kHeld; ++h) {
                    const int p = p0 + 32 * h;
                    q[h] = p < np ? load_part<true>(a, pr + p) : make_float2(kNegInf, __int_as_float(0x7fffffff));
                }
#pragma unroll
                for (int h = 0; h < kHeld; ++h) {
                    const int qi = __float_as_int(q[h].y);
                    if (am_better(q[h].x, qi, bv, bi)) { bv = q[h].x; bi = qi; }
                }
            }
            warp_argmax(bv, bi);
            if (lane == 0) g[r] = bi;
        }
    } else if constexpr (MANY_ROWS) {
        constexpr int kRows = 4, kHeld = 4;              // rows and loads per lane in flight
        for (int r0 = gw; r0 < R; r0 += NW * kRows) {
            float bv[kRows];
            int bi[kRows];
#pragma unroll
            for (int j = 0; j < kRows; ++j) { bv[j] = kNegInf; bi[j] = 0x7fffffff; }
            for (int p0 = lane; p0 < np; p0 += 32 * kHeld) {
                float2 q[kRows][kHeld];
#pragma unroll
                for (int j = 0; j < kRows; ++j)
#pragma unroll
                    for (int h = 0; h < kHeld; ++h) {
                        const int r = r0 + NW * j, p = p0 + 32 * h;
                        q[j][h] = (r < R && p < np) ? load_part<true>(a, base + (size_t)r * P + p)
                                                    : make_float2(kNegInf, __int_as_float(0x7fffffff));
                    }
#pragma unroll
                for (int j = 0; j < kRows; ++j)
#pragma unroll
                    for (int h = 0; h < kHeld; ++h) {
                        const int qi = __float_as_int(q[j][h].y);
                        if (am_better(q[j][h].x, qi, bv[j], bi[j])) { bv[j] = q[j][h].x; bi[j] = qi; }
                    }
            }
#pragma unroll
            for (int j = 0; j < kRows; ++j) {
                warp_argmax(bv[j], bi[j]);
                if (lane == 0 && r0 + NW * j < R) g[r0 + NW * j] = bi[j];
            }
        }
    }
    group_sync_n<NT>();
}

// Greedy chain: k = first i with x_i != argmax of row i, else gamma; output
// x_0..x_{k-1} then the target argmax of row k.
template <int NT>
static __device__ void decide_greedy(const VerifyArgs& a, int b, int gt, ArgmaxDecideSmem& sm) {
    const int G = a.gamma;
    merge_argmax_rows<NT>(a, b, gt, sm.g);
    if (gt == 0) {
        int bad = 0;
        for (int i = 0; i < G; ++i) {
            const int xi = sm.x[i];
            if (xi < 0 || xi >= a.V) bad = 1;
        }
        int k = G;
        if (bad) {
            atomicOr(a.err, SPEC_DEVERR_TOKEN_RANGE);
            k = -1;
        } else {
            for (int i = 0; i < G; ++i)
                if (sm.x[i] != sm.g[i]) { k = i; break; }
        }
        sm.k = k;
        a.out_acc[b] = k;
    }
    group_sync_n<NT>();
    const int k = sm.k;
    for (int i = gt; i <= G; i += NT) {
        int v = -1;
        if (k >= 0) v = i < k ? sm.x[i] : (i == k ? sm.g[k] : -1);
        a.out_tok[(size_t)b * (G + 1) + i] = v;
    }
}

// Draft tree: a node is accepted when its parent is and its token is the
// argmax of the parent's row; output the longest accepted root path (ties:
// lowest node ids) and the argmax of the path's last node.
//
// Trees of fewer than kTreeParallelNodes nodes take one thread's sweep over
// the nodes in descending id order (children have larger ids than their
// parent, so a node is final before its parent reads it; on equal length the
// lower child id wins), then the walk from the root.  Larger trees take one
// thread per node (N <= NT), in O(log depth) rounds of pointer doubling:
//   1. acceptance and depth: each node follows a pointer that doubles its
//      reach every round, AND-ing the matches and adding the depths of the
//      segments it jumps;
//   2. sub(n), the deepest accepted depth in n's subtree: every accepted node
//      pushes its value (atomic max) to the ancestor its pointer reaches, the
//      pointer doubling each round, so after round k a node holds the values
//      of its descendants up to 2^(k+1) - 1 below it (concurrent pushes only
//      add descendants' depths, which a max tolerates);
//   3. each accepted node offers (sub, lowest id) to its parent (atomic max):
//      the parent's chosen child continues the longest path, the lowest id
//      among equals -- the rule of a sweep that walks from the root;
//   4. a node is on the path when every link from it to the root is a chosen
//      one (pointer doubling again); its output slot is its depth - 1, and
//      the path has sub(root) nodes.
constexpr int kTreeParallelNodes = 64;

template <int NT>
static __device__ void decide_tree(const VerifyArgs& a, int b, int gt, ArgmaxDecideSmem& sm,
                                   TreeWalkSmem& tw) {
    const int N = a.rows_per_seq;                          // <= NT
    const int* tok = sm.x;                                 // prefetched
    const int* par = sm.par;
    if (gt == 0) sm.bad = 0;
    merge_argmax_rows<NT, true>(a, b, gt, sm.g);           // ends with group_sync
    const int n = gt;
    const bool own = n < N;
    if (own) {
        const int p = par[n];
        if (n == 0 ? p != -1 : (p < 0 || p >= n)) atomicOr(&sm.bad, SPEC_DEVERR_TREE_PARENT);
        if (n > 0) {
            const int t = tok[n];
            if (t < 0 || t >= a.V) atomicOr(&sm.bad, SPEC_DEVERR_TOKEN_RANGE);
        }
    }
    group_sync_n<NT>();
    int32_t* on = a.out_nodes + (size_t)b * N;
    int32_t* ot = a.out_tok + (size_t)b * N;
    const int bad = sm.bad;
    int len = -1;
    if (!bad && N < kTreeParallelNodes) {
        // the sweep: sm.sub holds a node's longest accepted continuation, sm.key its child
        if (own) { tw.sub[n] = 0; tw.key[n] = -1; }
        __syncthreads();
        if (gt == 0) {
            for (int m = N - 1; m >= 1; --m) {
                const int p = par[m];
                if (tok[m] != sm.g[p]) continue;
                if (1 + tw.sub[m] >= tw.sub[p]) { tw.sub[p] = 1 + tw.sub[m]; tw.key[p] = m; }
            }
            int l = 0, cur = 0;
            while (tw.key[cur] >= 0) {
                cur = tw.key[cur];
                on[l] = cur;
                ot[l] = tok[cur];
                ++l;
            }
            ot[l] = sm.g[cur];
            sm.len = l;
        }
        __syncthreads();
        len = sm.len;
    } else if (!bad) {
        // 1. acceptance and depth
        int u = own && n > 0 ? par[n] : -1;
        int ac = own && (n == 0 || tok[n] == sm.g[par[n]]) ? 1 : 0;
        int d = own && n > 0 ? 1 : 0;
        if (own) { tw.up[n] = u; tw.acc[n] = ac; tw.dep[n] = d; }
        while (__syncthreads_or(u >= 0)) {
            int nu = -1;
            if (u >= 0) { ac &= tw.acc[u]; d += tw.dep[u]; nu = tw.up[u]; }
            __syncthreads();
            u = nu;
            if (own) { tw.up[n] = u; tw.acc[n] = ac; tw.dep[n] = d; }
        }
        // 2. deepest accepted depth of every subtree
        int w = own && n > 0 ? par[n] : -1;
        if (own) { tw.sub[n] = ac ? d : -1; tw.up[n] = w; tw.key[n] = -1; }
        while (__syncthreads_or(w >= 0)) {
            const int v = own ? tw.sub[n] : -1;
            if (w >= 0 && v >= 0) atomicMax(&tw.sub[w], v);
            const int nw = w >= 0 ? tw.up[w] : -1;
            __syncthreads();
            w = nw;
            if (own) tw.up[n] = w;
        }
        // 3. the chosen child of every node: longest continuation, lowest id
        if (own && n > 0 && ac) atomicMax(&tw.key[par[n]], (tw.sub[n] << 11) | (2047 - n));
        __syncthreads();
        // 4. the path: nodes whose every link to the root is a chosen one
        auto chosen = [&](int p) { const int k = tw.key[p]; return k >= 0 ? 2047 - (k & 2047) : -1; };
        int v2 = own && n > 0 ? par[n] : -1;
        int ok = own && (n == 0 || chosen(par[n]) == n) ? 1 : 0;
        if (own) { tw.up[n] = v2; tw.acc[n] = ok; }
        while (__syncthreads_or(v2 >= 0)) {
            int nv = -1;
            if (v2 >= 0) { ok &= tw.acc[v2]; nv = tw.up[v2]; }
            __syncthreads();
            v2 = nv;
            if (own) { tw.up[n] = v2; tw.acc[n] = ok; }
        }
        len = tw.sub[0];                                   // the root is accepted: depth 0 or more
        if (gt == 0) sm.last = 0;
        __syncthreads();
        if (own && n > 0 && ok) {
            on[d - 1] = n;
            ot[d - 1] = tok[n];
            if (d == len) sm.last = n;
        }
        __syncthreads();
        if (gt == 0) ot[len] = sm.g[sm.last];
    }
    if (gt == 0) {
        if (bad) atomicOr(a.err, bad);
        a.out_acc[b] = len;
    }
    for (int m = gt; m < N; m += NT) {
        if (len < 0 || m >= len) on[m] = -1;
        if (len < 0 || m > len) ot[m] = -1;
    }
}

// The contiguous range of block chunks [*c0, *c1) that CTA `cta` of `ncta`
// streams, balanced to within one chunk.
__device__ __forceinline__ void cta_range(unsigned total, unsigned cta, unsigned ncta, unsigned* c0,
                                          unsigned* c1) {
    const unsigned q = total / ncta, r = total % ncta;
    *c0 = cta * q + min(cta, r);
    *c1 = *c0 + q + (cta < r ? 1u : 0u);
}

}  // namespace sv
