// Stochastic verification: the kernels behind spec_verify_sample.
//
// Source: "Speculative decoding: guess a few tokens first - why the answer
// stays the same", section "What happens in one round" (steps 1-4) and section
// "Why fixing wrong guesses does not leave the target distribution" (residual
// p'(x) = norm(max(0, p(x) - q(x)))).
//
// Pass 1 streams every logit once (sv_stream.cuh): each warp chunk of each of
// the 2*gamma+1 rows of every sequence becomes a partial (max m, sum
// 2^((z - m) log2(e)/T)).
//
// Pass 2 takes the accept decisions (sv_decide.cuh) and draws the final token
// of every sequence from the single row pair it comes from -- target and
// draft row k after a rejection at k (weights max(0, p_k - q_k)), target row
// gamma when every draft was accepted (weights p_gamma) -- by inverse CDF in
// index order.  Two kernels, launched with programmatic dependent launch,
// keep every sequence in flight at once; in a whole sampling call both start
// with the pass-1 stream and work beside it, each on a sequence as soon as
// that sequence's data carries the call's tag (tagged words, sv_common.cuh):
//   sample_decide_kernel  one CTA per sequence: row statistics from the
//                         partials, the accept decisions, every output but
//                         the final token, and the approximate normaliser
//                         ratio rt = Z_t/Z_d of row k from those statistics,
//                         published in the tagged SampleDesc;
//   sample_final_kernel   one CTA per 8192-element chunk of row k, one warp
//                         per 1024-element segment: sums of the exponentials
//                         of the target and draft segment and, after a
//                         rejection, the residual sum at ratio rt with its
//                         slope, stored as tagged words.  The sequence's
//                         chunk CTA that takes the last ticket (a tagged
//                         count) then runs the search: the exact ratio R
//                         from the exponential sums, the segment residual
//                         sums moved from rt to R to first order, prefix over
//                         them, the owning segment, its 1024 weights
//                         recomputed at R and scanned, the owning element.
// The weights are formed from the very exponentials whose sums normalise them
// (the same arithmetic in every kernel), and all sums are float-float (about
// 48 bits): the CDF each sequence samples from stays within ~1e-9 of the
// exact one, which matters because the long tail of a 150K-token vocabulary
// puts CDF boundaries ~1e-7 apart.
#include <stdlib.h>

#include <atomic>

#include "sv_final.cuh"

namespace sv {


// One CTA per sequence: the accept decisions and every output but the final
// token, and the SampleDesc the chunk kernels read.  In a whole sampling call
// this kernel starts with the stream and runs beside it (8 warps of at most
// 48 registers: two stream CTAs, one of these and a final-pass CTA fill an
// SM's 64K registers exactly): each CTA takes its sequence's
// decision once that sequence's partials are in, and the last CTA waits for
// the stream to complete before exiting, so that this kernel's completion
// covers the stream's for the kernels after it.
constexpr int kSampleDecideThreads = 256;

template <int ELT>
__global__ void __launch_bounds__(kSampleDecideThreads, 5) sample_decide_kernel(const VerifyArgs a) {
    __shared__ SampleDecideSmem dsm;
    pdl_trigger();
    const int k = decide_sample<ELT, kSampleDecideThreads>(a, blockIdx.x, threadIdx.x, dsm);  // waits for its partials
    write_sample_decision<kSampleDecideThreads>(a, blockIdx.x, threadIdx.x, k, dsm);
    if (a.poll_parts && blockIdx.x == gridDim.x - 1) pdl_wait();
}

// Per (chunk, sequence): the sums of the exponentials of target row k and
// (after a rejection) draft row k over each of the chunk's segments, and the
// residual sums at the approximate ratio with their slopes; then, in the
// last of the sequence's C chunk CTAs to take a ticket, the search.  Each CTA
// starts once its sequence's SampleDesc of this call is published (by the
// decide kernel or the lazy pass).
template <int ELT, bool VEC>
__global__ void __launch_bounds__(kCT, 4) sample_final_kernel(const VerifyArgs a) {
    __shared__ FinalSmem sm;
    const int b = blockIdx.x / a.C, c = blockIdx.x - b * a.C;   // chunks of a sequence adjacent
    pdl_trigger();
    // The last CTA waits for the decide kernel to complete, so that this
    // kernel's completion covers it; the others start on their sequence as
    // soon as its SampleDesc of this call is published.
    if (blockIdx.x == gridDim.x - 1) pdl_wait();
    if (threadIdx.x == 0) sm.desc = wait_desc(a, b);
    __syncthreads();
    const SampleDesc d = sm.desc;
    if (d.k < 0) return;
    // the final token's uniform, loaded now so that its latency is not the search's
    const float u = a.u[(size_t)b * (a.gamma + 1) + a.gamma];
    {
        const FinalRows f = final_rows<ELT>(a, b, d);
        segment_sums_global<ELT, VEC>(a, f, b, c * kCW + (threadIdx.x >> 5), d.rt, threadIdx.x & 31);
    }
    // The last of the sequence's chunk CTAs to take a ticket runs the
    // search; it waits there for any other chunk's tagged sums still on
    // their way.
    __syncthreads();
    if (threadIdx.x == 0) sm.mine = take_ticket(a, b) == (unsigned)(a.C - 1);
    __syncthreads();
    if (!sm.mine) return;
    search_sequence<ELT, VEC>(a, b, d, u, sm, threadIdx.x);
}

// ------------------------------------------------ lazy (early-exit) pass 1
// Source: "Speculative decoding: guess a few tokens first - why the answer
// stays the same", section "What happens in one round", step 3: drafts are
// checked left to right and the first rejection discards every later draft,
// so a position's rows are only needed while every earlier draft was
// accepted.
//
// The positions go in groups of doubling size -- [0, 2), [2, 6), [6, 14), ...,
// the last group ending with target row gamma -- and each group is one pass
// over the whole GPU: the bulk-copy stream of sv_stream.cuh (kModeLazy) over
// the group's target and draft rows of the sequences still undecided, then
// lazy_decide_kernel, one CTA per such sequence, which merges those rows'
// partials and takes the group's accept decisions in order.  A sequence
// that rejects a draft (or reaches the bonus row) is finished there -- every
// output but the final token, and the SampleDesc of the final sample -- and
// the others go on the next group's survivor list.  The partials are the full
// pass's bit for bit (same block chunks, same arithmetic, same merge), so
// every decision and log-probability is too.
//
// A rejection at k lies in a group [lo, hi) with hi <= 2 k + 2, so the rows
// read are at most those of positions 0..2k+1, twice the exact early exit,
// in O(log gamma) passes: one pass per position would pay a kernel boundary
// per position, and one cluster of CTAs per sequence that streams and
// decides position by position is bound by that chain's latency.

// Positions per group: at most 128 (gamma <= 256).
constexpr int kLazyMaxGroup = kMaxGamma / 2;

struct LazyDecideSmem {
    float M[2 * kLazyMaxGroup], lnZ[2 * kLazyMaxGroup];   // group rows: target, then draft
    float lp[kLazyMaxGroup], lq[kLazyMaxGroup];
    float u[kLazyMaxGroup], zt[kLazyMaxGroup], zd[kLazyMaxGroup];
    int bad, k;
};

// 16 warps: the 13 rows of a [2, 8) group are merged in one round of loads.
constexpr int kLazyDecideThreads = 512;

// One CTA per sequence of the group's list (every sequence for the first
// group).  k is the rejection index, gamma when the group holds the bonus row
// and every draft was accepted, -1 for bad input, -2 for "undecided: next
// group".
template <int ELT>
__global__ void __launch_bounds__(kLazyDecideThreads) lazy_decide_kernel(const VerifyArgs a) {
    __shared__ LazyDecideSmem sm;
    const int gt = threadIdx.x;
    const int lo = a.lz_lo, nt = a.lz_nt, nd = a.lz_nd;
    const size_t rowbytes = (size_t)a.V * ELT;
    const bool first = a.lz_list == nullptr;
    pdl_trigger();
    auto gather = [&](int b) {
        for (int q = gt; q < nd; q += kLazyDecideThreads) {
            const int p = lo + q;
            const int xi = a.x[(size_t)b * a.gamma + p];
            const bool in = xi >= 0 && xi < a.V;
            sm.zt[q] = in ? load_logit<ELT>(sample_row(a, b, p, rowbytes), xi) : 0.f;
            sm.zd[q] = in ? load_logit<ELT>(sample_row(a, b, a.gamma + 1 + p, rowbytes), xi) : 0.f;
            sm.u[q] = a.u[(size_t)b * (a.gamma + 1) + p];
        }
    };
    int b = blockIdx.x, bad = 0;
    if (first) {
        // Inputs only: this group's stream waited for the kernel before the
        // call, so they are final.  Every draft token of the sequence is
        // checked here, as the full pass's decision does.
        gather(b);
        for (int i = gt; i < a.gamma; i += kLazyDecideThreads) {
            const int xi = a.x[(size_t)b * a.gamma + i];
            if (xi < 0 || xi >= a.V) bad = 1;
        }
    }
    pdl_wait();                                           // the group's partials and list
    if (!first) {
        if ((int)blockIdx.x >= __ldcg(a.lz_count)) return;   // the whole CTA
        b = __ldcg(a.lz_list + blockIdx.x);
        gather(b);
    }
    merge_rows_group<kLazyDecideThreads>(
        a, b, nt + nd, [&](int q) { return q < nt ? lo + q : a.gamma + 1 + lo + (q - nt); }, gt, sm.M, sm.lnZ);
    bad = __syncthreads_or(bad);
    if (gt == 0) {
        int k = -2, bits = bad ? SPEC_DEVERR_TOKEN_RANGE : 0;
        for (int q = 0; !bits && q < nt; ++q) {
            if (sm.M[q] == kNegInf || (q < nd && sm.M[nt + q] == kNegInf)) {
                bits = SPEC_DEVERR_EMPTY_ROW;
                break;
            }
            if (q == nd) { k = a.gamma; break; }          // target row gamma: every draft accepted
            sm.lp[q] = row_log_prob(sm.zt[q], sm.M[q], sm.lnZ[q], a);
            sm.lq[q] = row_log_prob(sm.zd[q], sm.M[nt + q], sm.lnZ[nt + q], a);
            if (!accept_draft(sm.lp[q], sm.lq[q], sm.u[q])) { k = lo + q; break; }
        }
        sm.bad = bits;
        sm.k = bits ? -1 : k;
    }
    __syncthreads();
    const int k = sm.k;
    if (a.out_lp && k != -1)                              // the positions decided here
        for (int q = gt; q < nd; q += kLazyDecideThreads)
            if (k == -2 || lo + q <= k) {
                float* o = a.out_lp + ((size_t)b * a.gamma + lo + q) * 2;
                o[0] = sm.lp[q];
                o[1] = sm.lq[q];
            }
    if (k == -2) {
        if (gt == 0) a.lz_next_list[atomicAdd(a.lz_next_count, 1)] = b;
        return;
    }
    if (gt == 0) {
        if (sm.bad) atomicOr(a.err, sm.bad);
        a.out_acc[b] = k;
        SampleDesc d;
        d.k = k;
        d.mt = k >= 0 ? sm.M[k - lo] : 0.f;
        d.md = (k >= 0 && k < a.gamma) ? sm.M[nt + k - lo] : 0.f;
        d.rt = (k >= 0 && k < a.gamma) ? expf(sm.lnZ[k - lo] - sm.lnZ[nt + k - lo]) : 0.f;   // as the decide step
        publish_desc(a, b, d);
    }
    // accepted drafts and padding; slot k belongs to the final-pass search
    for (int i = gt; i <= a.gamma; i += kLazyDecideThreads)
        if (k < 0 || i != k)
            a.out_tok[(size_t)b * (a.gamma + 1) + i] = (k >= 0 && i < k) ? a.x[(size_t)b * a.gamma + i] : -1;
    if (a.out_lp)                                         // positions never decided
        for (int i = gt; i < a.gamma; i += kLazyDecideThreads)
            if (k < 0 || i > k) {
                float* o = a.out_lp + ((size_t)b * a.gamma + i) * 2;
                o[0] = CUDART_NAN_F;
                o[1] = CUDART_NAN_F;
            }
}

// Rows that are not a multiple of 16 bytes take the full pass in lazy mode;
// this clears the log-probabilities of the positions a lazy pass does not read.
__global__ void lazy_mask_logprobs_kernel(const VerifyArgs a) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= a.B) return;
    const int k = a.out_acc[b];
    for (int i = 0; i < a.gamma; ++i)
        if (k < 0 || i > k) {
            a.out_lp[((size_t)b * a.gamma + i) * 2] = CUDART_NAN_F;
            a.out_lp[((size_t)b * a.gamma + i) * 2 + 1] = CUDART_NAN_F;
        }
}

// A group boundary costs a pass: a stream and a decide kernel, about 7 us of
// ramp and latency on GB300.  It pays when the sequences that stop before it
// skip more HBM time than that; with half of them stopping, when the rows
// after the boundary (for every sequence) hold at least 2 x 7 us x 6.7 TB/s,
// about 96 MB.  Below that the group runs on to the end.  The environment
// variable SPEC_VERIFY_LAZY_SPLIT_BYTES, read once per process, and
// spec_verify_set_lazy_split_bytes override the figure (0: always split);
// outputs do not depend on it.
constexpr double kLazySplitBytes = 96.0 * (1 << 20);

// The initial figure: the environment variable, read once per process (at the
// first lazy call or groups query), else kLazySplitBytes.
static double lazy_split_from_env() {
    const char* e = getenv("SPEC_VERIFY_LAZY_SPLIT_BYTES");
    if (!e || !*e) return kLazySplitBytes;
    char* end = nullptr;
    const double v = strtod(e, &end);
    return (end && *end == '\0' && v >= 0.0) ? v : kLazySplitBytes;
}

// The current figure; spec_verify_set_lazy_split_bytes changes it.  A negative
// value in the slot means "not yet read".
static std::atomic<double> g_lazy_split{-1.0};

static double lazy_split_bytes() {
    double v = g_lazy_split.load(std::memory_order_relaxed);
    if (v < 0.0) {
        static const double from_env = lazy_split_from_env();   // thread-safe, once
        double expect = v;
        g_lazy_split.compare_exchange_strong(expect, from_env, std::memory_order_relaxed);
        v = g_lazy_split.load(std::memory_order_relaxed);
    }
    return v;
}

void set_lazy_split_bytes(double bytes) {
    g_lazy_split.store(bytes >= 0.0 ? bytes : kLazySplitBytes, std::memory_order_relaxed);
}

// Upper ends of the lazy position groups: sizes doubling from 2, a group
// running on to the end (at most kLazyMaxGroup positions) when the rows after
// it are too few to be worth a pass.  Every group has at least the doubling
// size, so gamma <= 256 takes at most kLazyGroups of them.  Returns the count.
static int lazy_group_ends(int B, int gamma, size_t rowbytes, int (&hi)[kLazyGroups]) {
    const double split = lazy_split_bytes();
    int ng = 0;
    for (int lo = 0, n = 2; lo <= gamma && ng < kLazyGroups; n *= 2) {
        int h = min(lo + min(n, kLazyMaxGroup), gamma + 1);
        const double rest = (double)B * (double)rowbytes *
                            (double)((gamma + 1 - h) + (gamma - min(h, gamma)));
        if (rest < split) h = min(lo + kLazyMaxGroup, gamma + 1);
        hi[ng++] = h;
        lo = h;
    }
    return ng;
}

int lazy_groups_host(int B, int gamma, size_t rowbytes, int* ends) {
    int hi[kLazyGroups];
    const int n = lazy_group_ends(B, gamma, rowbytes, hi);
    for (int g = 0; g < n; ++g) ends[g] = hi[g];
    return n;
}

// The lazy pass: per position group a stream and a decide kernel, chained
// with programmatic dependent launch; the first group's stream zeroes the
// later groups' survivor counts.
template <int ELT>
static cudaError_t launch_lazy(VerifyArgs a, const DeviceInfo& di, cudaStream_t st, char* lz) {
    int* counts = reinterpret_cast<int*>(lz);
    int* lists = reinterpret_cast<int*>(lz + 256);
    int ends[kLazyGroups];
    const int ngroups = lazy_group_ends(a.B, a.gamma, (size_t)a.V * ELT, ends);
    for (int g = 0, lo = 0; g < ngroups; lo = ends[g], ++g) {
        const int hi = ends[g];
        a.lz_lo = lo;
        a.lz_nt = hi - lo;
        a.lz_nd = min(hi, a.gamma) - lo;
        a.lz_list = g > 0 ? lists + (size_t)g * a.B : nullptr;
        a.lz_count = g > 0 ? counts + g : nullptr;
        a.lz_next_list = g + 1 < ngroups ? lists + (size_t)(g + 1) * a.B : nullptr;
        a.lz_next_count = g + 1 < ngroups ? counts + g + 1 : nullptr;
        a.lz_zero = counts + 1;
        a.lz_nzero = g == 0 ? ngroups - 1 : 0;
        a.total_chunks = (long long)a.B * (a.lz_nt + a.lz_nd) * a.nseg;   // at most
        cudaError_t e = launch_stream<ELT, kModeLazy>(a, di, st);
        if (e != cudaSuccess) return e;
        e = launch_pdl(lazy_decide_kernel<ELT>, dim3((unsigned)a.B), kLazyDecideThreads, 0, st, a);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// ---------------------------------------------------------------- launch
// The decide and final-pass kernels prefer the whole carveout as shared
// memory, as the ring stream does: SMs that hold stream CTAs can then take
// theirs too (an SM runs CTAs of several kernels only under one carveout).
template <typename K>
static cudaError_t prefer_max_shared(K kfn, DeviceSlots& slots) {
    int unused = 0;
    return device_once(slots, &unused, [&](int, int* o) {
        *o = 1;
        return cudaFuncSetAttribute(kfn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                    cudaSharedmemCarveoutMaxShared);
    });
}

template <int ELT, bool VEC>
static cudaError_t launch_final_t(const VerifyArgs& a, cudaStream_t st, bool decide = true) {
    cudaError_t e = cudaSuccess;
    if (decide) {
        static DeviceSlots dslots = {};
        e = prefer_max_shared(sample_decide_kernel<ELT>, dslots);
        if (e != cudaSuccess) return e;
        e = launch_pdl(sample_decide_kernel<ELT>, dim3(a.B), kSampleDecideThreads, 0, st, a);
        if (e != cudaSuccess) return e;
    }
    static DeviceSlots fslots = {};
    e = prefer_max_shared(sample_final_kernel<ELT, VEC>, fslots);
    if (e != cudaSuccess) return e;
    return launch_pdl(sample_final_kernel<ELT, VEC>, dim3((unsigned)a.C * (unsigned)a.B), kCT, 0, st,
                      a);
}

cudaError_t launch_sample(const void* zt, const void* zd, spec_dtype_t dt, const int32_t* x,
                          const float* u, float T, int B, int gamma, int V, int32_t* out_tok,
                          int32_t* out_acc, float* out_lp, void* ws, cudaStream_t st, int parts) {
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int elt = elt_size(dt);
    const bool vec = ((size_t)V * elt) % 16 == 0;
    const WsLayout L = ws_layout(B, gamma, V);
    char* w = static_cast<char*>(ws);

    VerifyArgs a = {};
    a.wait_limit = ring_wait_limit();
    a.zt = static_cast<const char*>(zt);
    a.zd = static_cast<const char*>(zd);
    a.x = x;
    a.u = u;
    a.T = T;
    a.invT = 1.0f / T;
    const double sd = 1.4426950408889634 / (double)T;
    a.s = (float)sd;
    a.s_lo = (float)(sd - (double)a.s);

    a.gamma = gamma;
    a.rows_per_seq = 2 * gamma + 1;
    a.V = V;
    a.nseg = nseg(V, elt);
    a.total_chunks = (long long)B * a.rows_per_seq * a.nseg;
    a.B = B;
    a.C = final_chunks(V);
    a.parts = reinterpret_cast<float2*>(w + L.part_off);
    a.desc = reinterpret_cast<unsigned long long*>(w + L.desc_off);
    a.epoch = next_launch_tag();
    a.ptag = (uint32_t)a.epoch ? (uint32_t)a.epoch : 1u;
    a.tick = reinterpret_cast<unsigned long long*>(w + L.tick_off);
    a.sums = reinterpret_cast<unsigned long long*>(w + L.sum_off);
    a.err = reinterpret_cast<int*>(w + L.err_off);
    a.out_tok = out_tok;
    a.out_acc = out_acc;
    a.out_lp = out_lp;

    a.early_inputs = (parts & kSampleStats) ? 1 : 0;
    bool mask_lp = false;
    if (parts & kSampleLazy) {
        if (vec) {
            char* lz = w + L.lz_off;
            e = elt == 2 ? launch_lazy<2>(a, di, st, lz) : launch_lazy<4>(a, di, st, lz);
            if (e != cudaSuccess) return e;
            return elt == 2 ? launch_final_t<2, true>(a, st, false) : launch_final_t<4, true>(a, st, false);
        }
        parts = kSampleStats | kSampleFinish;             // full pass, then unread positions cleared
        a.early_inputs = 1;
        mask_lp = out_lp != nullptr;
    }
    // A whole call on 16-byte rows: the decide kernel runs beside the ring
    // stream and waits for each sequence's tagged partials.
    a.poll_parts = (parts & kSampleStats) && (parts & kSampleFinish) && vec ? 1 : 0;
    if (parts & kSampleStats) {
        e = elt == 2 ? launch_stream<2, kModeSample>(a, di, st) : launch_stream<4, kModeSample>(a, di, st);
        if (e != cudaSuccess) return e;
    }
    if (parts & kSampleFinish) {
        if (elt == 2) e = vec ? launch_final_t<2, true>(a, st) : launch_final_t<2, false>(a, st);
        else e = vec ? launch_final_t<4, true>(a, st) : launch_final_t<4, false>(a, st);
        if (e != cudaSuccess) return e;
    }
    if (mask_lp) {
        lazy_mask_logprobs_kernel<<<(B + 127) / 128, 128, 0, st>>>(a);
        e = cudaGetLastError();
    }
    return e;
}

bool sample_supported_vocab(int V) {
    // the search kernel scans all chunk totals of a row in one CTA
    return final_chunks(V) <= kFinalChunkThreads;
}

}  // namespace sv
