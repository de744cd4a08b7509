// Stochastic verification: the kernels behind spec_verify_sample.
//
// Source: "Speculative decoding: guess a few tokens first - why the answer
// stays the same", section "What happens in one round" (steps 1-4) and section
// "Why fixing wrong guesses does not leave the target distribution" (residual
// p'(x) = norm(max(0, p(x) - q(x)))).
//
// Pass 1 streams every logit once (ring_stream_kernel in sv_stream.cuh for
// 16-byte rows, sample_rowstats_kernel below otherwise): each warp chunk of
// each of the 2*gamma+1 rows of every sequence becomes a partial (max m,
// sum 2^((z - m) log2(e)/T)).
//
// Pass 2 draws the final token of every sequence from the single row pair it
// comes from -- target and draft row k after a rejection at k (weights
// max(0, p_k - q_k)), target row gamma when every draft was accepted (weights
// p_gamma) -- by inverse CDF in index order.  Four small kernels, chained with
// programmatic dependent launch, keep every sequence in flight at once:
//   sample_decide_kernel  one CTA per sequence: row statistics from the
//                         partials, accept decisions u_i < p_i(x_i)/q_i(x_i)
//                         left to right, all outputs but the final token;
//   sample_zsum_kernel    one CTA per 8192-element chunk of row k: sums of the
//                         exponentials of the target and draft chunk;
//   sample_wsum_kernel    one CTA per chunk (rejections only): the ratio of the
//                         two row normalisers from all chunk sums, then the
//                         chunk's residual weight total;
//   sample_search_kernel  one CTA per sequence: prefix over the chunk totals,
//                         the owning chunk, its weights recomputed and scanned,
//                         the owning element.
// The weights are formed from the very exponentials whose sums normalise them,
// all sums are float-float (about 48 bits), and a chunk's total and the scan
// that later searches inside it come from the same block-scan code, so the
// intervals of chunks, threads and elements tile [0, S) exactly.
#include "sv_common.cuh"
#include "sv_stream.cuh"

namespace sv {

#ifndef SV_FINAL_EXACT_EXP
#define SV_FINAL_EXACT_EXP 1
#endif

constexpr int kMaxGamma = 256;                 // rows per sequence <= 2*256+1
constexpr int kDecideThreadsS = 512;

struct StatsArgs {
    const char* zt;
    const char* zd;
    float s;            // log2(e) / T
    int gamma, V;
    int nseg;           // block chunks per row
    int rows_per_seq;   // 2 * gamma + 1
    long long total_chunks;
    float2* parts;
};

struct FinalArgs {
    const char* zt;
    const char* zd;
    const int32_t* x;
    const float* u;
    float T, invT, s;
    int B, gamma, V;
    int nseg, rows_per_seq;
    int C;              // 2048-element chunks per row
    const float2* parts;
    SampleDesc* desc;
    float4* zsum;       // [B, C]: (Za.hi, Za.lo, Zb.hi, Zb.lo) of each chunk
    float2* wsum;       // [B, C]: residual weight total of each chunk
    int32_t* out_tok;
    int32_t* out_acc;
    float* out_lp;
    int* err;
};

// Row r of sequence b: r <= gamma is target row r, r > gamma is draft row r-gamma-1.
__device__ __forceinline__ const char* seq_row(const char* zt, const char* zd, int gamma, int b,
                                               int r, size_t rowbytes) {
    return r <= gamma ? zt + ((size_t)b * (gamma + 1) + r) * rowbytes
                      : zd + ((size_t)b * gamma + (r - gamma - 1)) * rowbytes;
}

template <int ELT, bool VEC>
__global__ void __launch_bounds__(kThreads) sample_rowstats_kernel(const StatsArgs a) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int WE = 32 * kLaneBytes / ELT;              // elements per warp chunk
    const int P = a.nseg * kWarps;
    const size_t rowbytes = (size_t)a.V * ELT;

    for (long long c = blockIdx.x; c < a.total_chunks; c += gridDim.x) {
        if (c + gridDim.x >= a.total_chunks) pdl_trigger();
        const int seg = (int)(c % a.nseg);
        const long long rr = c / a.nseg;
        const int b = (int)(rr / a.rows_per_seq);
        const int r = (int)(rr % a.rows_per_seq);
        const char* row = seq_row(a.zt, a.zd, a.gamma, b, r, rowbytes);
        const int base = (seg * kWarps + warp) * WE;

        float m = kNegInf, z = 0.f;
        if (base < a.V) {
            LaneChunk<ELT, VEC> ch;
            ch.load(row, a.V, base, lane);
#pragma unroll
            for (int i = 0; i < LaneChunk<ELT, VEC>::EPL; ++i) m = fmaxf(m, ch.val(i));
            m = warp_max(m);
            if (m != kNegInf) {
#pragma unroll
                for (int i = 0; i < LaneChunk<ELT, VEC>::EPL; ++i)
                    z += ex2_approx((ch.val(i) - m) * a.s);
                z = warp_sum(z);
            }
        }
        if (lane == 0) a.parts[(size_t)rr * P + seg * kWarps + warp] = make_float2(m, z);
    }
}

// ---------------------------------------------------------------- pass 2
constexpr int kCT = kFinalChunkThreads;        // threads per chunk CTA (kFinalPerThread elements each)
constexpr int kCW = kCT / 32;

// exp((z - m) / T) for the final pass.  The default (SV_FINAL_EXACT_EXP=1)
// carries (z - m)/T as two floats into expf, leaving only expf's own rounding
// and one product: measured over 1e5 rows of the B=8, T=1 workload it halves
// the mismatches against the fp64 reference compared with the cheaper
// SV_FINAL_EXACT_EXP=0 form, 2^(z*s - m*s) from one fused multiply-add and the
// special-function unit (m*s is rounded once per row, a common factor that the
// normalisation cancels).
template <int ELT>
__device__ __forceinline__ float final_exp(float z, float m, float ms, bool wide, const FinalArgs& a) {
#if SV_FINAL_EXACT_EXP
    (void)ms;
    (void)wide;
    float d_hi, d_lo;
    if constexpr (ELT == 2) {
        d_hi = z - m;
        d_lo = 0.f;
    } else {
        d_hi = z - m;
        const float bb = d_hi - z;
        d_lo = (z - (d_hi - bb)) + (-m - bb);
    }
    if (d_hi == kNegInf) return 0.f;
    const float y = d_hi * a.invT;
    const float rem = fmaf(-y, a.T, d_hi) + d_lo;
    const float e = expf(y);
    return fmaf(e, rem * a.invT, e);
#else
    // wide (|m * s| beyond 1e30, only for extreme temperatures): subtract
    // first so no intermediate overflows
    return ex2_approx(wide ? (z - m) * a.s : fmaf(z, a.s, -ms));
#endif
}

constexpr int kPT = kFinalPerThread;

// The kPT logits of row `row` at [j0, j0 + kPT); entries at or beyond V are
// -inf.  All loads are issued before any is used.
template <int ELT, bool VEC>
__device__ __forceinline__ void load_seg(const char* row, int V, int j0, float (&z)[kPT]) {
    if constexpr (VEC) {
        constexpr int PV = 16 / ELT;                      // V is a multiple of PV
        uint4 q[kPT / PV];
#pragma unroll
        for (int h = 0; h < kPT / PV; ++h) {
            const int jj = j0 + PV * h;
            q[h] = jj < V ? ld_stream16(row + (size_t)jj * ELT)
                          : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
        }
#pragma unroll
        for (int h = 0; h < kPT / PV; ++h)
#pragma unroll
            for (int e = 0; e < PV; ++e) {
                if constexpr (ELT == 2) {
                    const uint32_t w = u4_get(q[h], e >> 1);
                    z[PV * h + e] = __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
                } else {
                    const uint32_t w = u4_get(q[h], e);
                    // -inf padding for fp32 vectors past V
                    z[PV * h + e] = (j0 + PV * h < V) ? __uint_as_float(w) : kNegInf;
                }
            }
    } else {
#pragma unroll
        for (int e = 0; e < kPT; ++e) z[e] = (j0 + e < V) ? load_logit<ELT>(row, j0 + e) : kNegInf;
    }
}

// Inclusive scan of one float-float value per thread over a kCT-thread block
// in thread order; *total receives the block total.  Deterministic: the same
// inputs give the same bits in every CTA.
__device__ __forceinline__ FF block_incl_scan_ff(FF v, FF* wtot, FF* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    FF x = warp_incl_scan_ff(v);
    if (lane == 31) wtot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        FF y = lane < kCW ? wtot[lane] : FF{0.f, 0.f};
        y = warp_incl_scan_ff(y);
        if (lane < kCW) wtot[lane] = y;
    }
    __syncthreads();
    const FF r = warp > 0 ? ff_combine(wtot[warp - 1], x) : x;
    *total = wtot[kCW - 1];
    __syncthreads();
    return r;
}

// Exclusive counterpart of an inclusive block scan result r (thread order).
__device__ __forceinline__ FF block_excl_from_incl(FF r, const FF* wtot_scanned) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const FF up = ff_shfl_up(r, 1);
    if (lane > 0) return up;
    return warp > 0 ? wtot_scanned[warp - 1] : FF{0.f, 0.f};
}

struct DecideSmem {
    float M[2 * kMaxGamma + 1];       // row max
    float lnZ[2 * kMaxGamma + 1];     // ln sum exp((z - M)/T)
    float lp[kMaxGamma], lq[kMaxGamma];
    int bad, k;
};

// Row statistics of sequence b from the pass-1 partials and the accept
// decisions.  Single precision throughout (GB300's double-precision rate is a
// small fraction of its float rate): ln p_i(x_i) and ln q_i(x_i) carry errors
// of ~1e-6, far inside the 1e-4 decision margin and the 1e-5 bar on returned
// probabilities.
template <int ELT>
__device__ void sample_decide(const FinalArgs& a, int b, DecideSmem& sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int P = a.nseg * kWarps;
    const size_t rowbytes = (size_t)a.V * ELT;
    if (threadIdx.x == 0) sm.bad = 0;
    __syncthreads();

    // M = max m_p, Z = sum Z_p 2^((m_p - M) s) over the row's warp partials
    // (float-float per lane, then across the warp).
    for (int r = warp; r < a.rows_per_seq; r += nwarps) {
        const float2* pr = a.parts + ((size_t)b * a.rows_per_seq + r) * P;
        float m = kNegInf;
        for (int p = lane; p < P; p += 32) m = fmaxf(m, pr[p].x);
        m = warp_max(m);
        FF z{0.f, 0.f};
        if (m != kNegInf) {
            for (int p = lane; p < P; p += 32) {
                const float2 q = pr[p];
                if (q.x != kNegInf) ff_add(z, q.y * ex2_approx((q.x - m) * a.s));
            }
        }
        z = ff_norm(warp_sum_ff(z));
        if (lane == 0) {
            sm.M[r] = m;
            sm.lnZ[r] = m == kNegInf ? 0.f : logf(z.hi) + z.lo / z.hi;
        }
    }
    __syncthreads();

    // Validate the drafts, gather z[x_i] and form ln p_i(x_i), ln q_i(x_i).
    for (int i = threadIdx.x; i < a.gamma; i += blockDim.x) {
        const int xi = a.x[(size_t)b * a.gamma + i];
        if (xi < 0 || xi >= a.V) {
            atomicOr(&sm.bad, SPEC_DEVERR_TOKEN_RANGE);
            sm.lp[i] = sm.lq[i] = 0.f;
        } else {
            const float ztx = load_logit<ELT>(seq_row(a.zt, a.zd, a.gamma, b, i, rowbytes), xi);
            const float zdx = load_logit<ELT>(seq_row(a.zt, a.zd, a.gamma, b, a.gamma + 1 + i, rowbytes), xi);
            sm.lp[i] = (ztx - sm.M[i]) * a.invT - sm.lnZ[i];
            sm.lq[i] = (zdx - sm.M[a.gamma + 1 + i]) * a.invT - sm.lnZ[a.gamma + 1 + i];
        }
    }
    for (int r = threadIdx.x; r < a.rows_per_seq; r += blockDim.x)
        if (sm.M[r] == kNegInf) atomicOr(&sm.bad, SPEC_DEVERR_EMPTY_ROW);
    __syncthreads();

    if (threadIdx.x == 0) {
        int k = -1;
        if (!sm.bad) {
            // Left to right; the first rejection voids the remaining drafts.
            k = a.gamma;
            for (int i = 0; i < a.gamma; ++i) {
                const float lp = sm.lp[i], lq = sm.lq[i];
                float r;
                if (lp == kNegInf) r = 0.f;
                else if (lq == kNegInf) r = CUDART_INF_F;
                else r = expf(lp - lq);
                if (!(a.u[(size_t)b * (a.gamma + 1) + i] < r)) { k = i; break; }
            }
        }
        sm.k = k;
    }
    __syncthreads();
}

template <int ELT>
__global__ void __launch_bounds__(kDecideThreadsS) sample_decide_kernel(const FinalArgs a) {
    __shared__ DecideSmem dsm;
    const int b = blockIdx.x, tid = threadIdx.x;
    pdl_trigger();
    pdl_wait();                                           // pass-1 partials are visible from here
    sample_decide<ELT>(a, b, dsm);
    const int k = dsm.k;
    if (tid == 0) {
        a.out_acc[b] = k;
        if (dsm.bad) atomicOr(a.err, dsm.bad);
        SampleDesc d;
        d.k = k;
        d.mt = k >= 0 ? dsm.M[k] : 0.f;
        d.md = (k >= 0 && k < a.gamma) ? dsm.M[a.gamma + 1 + k] : 0.f;
        d.pad = 0;
        a.desc[b] = d;
    }
    // Accepted drafts, padding and log-probabilities; slot k is written by
    // the search kernel.
    for (int i = tid; i <= a.gamma; i += blockDim.x)
        if (k < 0 || i != k)
            a.out_tok[(size_t)b * (a.gamma + 1) + i] = (k >= 0 && i < k) ? a.x[(size_t)b * a.gamma + i] : -1;
    if (a.out_lp)
        for (int i = tid; i < a.gamma; i += blockDim.x) {
            float* o = a.out_lp + ((size_t)b * a.gamma + i) * 2;
            o[0] = k >= 0 ? dsm.lp[i] : CUDART_NAN_F;
            o[1] = k >= 0 ? dsm.lq[i] : CUDART_NAN_F;
        }
}

// The exponentials of this thread's kPT elements of chunk c of the
// sequence's target row k (ea) and draft row k (eb, rejections only).
template <int ELT, bool VEC>
__device__ __forceinline__ void chunk_exps(const FinalArgs& a, int b, const SampleDesc& d, int c,
                                           float (&ea)[kPT], float (&eb)[kPT]) {
    const bool rej = d.k < a.gamma;
    const size_t rowbytes = (size_t)a.V * ELT;
    const int j0 = c * kFinalChunk + threadIdx.x * kPT;
    const float mts = d.mt * a.s, mds = d.md * a.s;
    const bool wt = !(fabsf(mts) < 1e30f), wd = !(fabsf(mds) < 1e30f);
    float zt[kPT], zd[kPT];
    load_seg<ELT, VEC>(a.zt + ((size_t)b * (a.gamma + 1) + d.k) * rowbytes, a.V, j0, zt);
    if (rej) load_seg<ELT, VEC>(a.zd + ((size_t)b * a.gamma + d.k) * rowbytes, a.V, j0, zd);
#pragma unroll
    for (int e = 0; e < kPT; ++e) {
        ea[e] = zt[e] == kNegInf ? 0.f : final_exp<ELT>(zt[e], d.mt, mts, wt, a);
        eb[e] = (rej && zd[e] != kNegInf) ? final_exp<ELT>(zd[e], d.md, mds, wd, a) : 0.f;
    }
}

// Residual weight max(0, p_k - q_k) scaled by Za: ea - (Za/Zb) eb, with the
// ratio as a float-float pair (Rhi, Rlo).
__device__ __forceinline__ float resid(float ea, float eb, float Rhi, float Rlo) {
    return fmaxf(fmaf(-Rlo, eb, fmaf(-Rhi, eb, ea)), 0.f);
}

__device__ __forceinline__ FF sum_seg(const float (&w)[kPT]) {
    FF acc{0.f, 0.f};
#pragma unroll
    for (int e = 0; e < kPT; ++e) ff_add(acc, w[e]);
    return ff_norm(acc);
}

// The ratio Za / Zb of the two row normalisers of sequence b, from the chunk
// sums (block-wide, identical in every CTA that calls it).
__device__ __forceinline__ FF normaliser_ratio(const FinalArgs& a, int b, FF* wtot) {
    FF za{0.f, 0.f}, zb{0.f, 0.f};
    if ((int)threadIdx.x < a.C) {
        const float4 q = a.zsum[(size_t)b * a.C + threadIdx.x];
        za = FF{q.x, q.y};
        zb = FF{q.z, q.w};
    }
    FF Za, Zb;
    block_incl_scan_ff(za, wtot, &Za);
    block_incl_scan_ff(zb, wtot, &Zb);
    return ff_div(Za, Zb);
}

template <int ELT, bool VEC>
__global__ void __launch_bounds__(kCT) sample_zsum_kernel(const FinalArgs a) {
    __shared__ FF wtot[kCW];
    const int c = blockIdx.x, b = blockIdx.y;
    pdl_trigger();
    pdl_wait();
    const SampleDesc d = a.desc[b];
    if (d.k < 0) return;
    float ea[kPT], eb[kPT];
    chunk_exps<ELT, VEC>(a, b, d, c, ea, eb);
    FF Za, Zb;
    block_incl_scan_ff(sum_seg(ea), wtot, &Za);
    block_incl_scan_ff(sum_seg(eb), wtot, &Zb);
    if (threadIdx.x == 0) a.zsum[(size_t)b * a.C + c] = make_float4(Za.hi, Za.lo, Zb.hi, Zb.lo);
}

template <int ELT, bool VEC>
__global__ void __launch_bounds__(kCT) sample_wsum_kernel(const FinalArgs a) {
    __shared__ FF wtot[kCW];
    const int c = blockIdx.x, b = blockIdx.y;
    pdl_trigger();
    pdl_wait();
    const SampleDesc d = a.desc[b];
    if (d.k < 0 || d.k >= a.gamma) return;               // bonus rows use the exponential sums
    const FF R = normaliser_ratio(a, b, wtot);
    float ea[kPT], eb[kPT], w[kPT];
    chunk_exps<ELT, VEC>(a, b, d, c, ea, eb);
#pragma unroll
    for (int e = 0; e < kPT; ++e) w[e] = resid(ea[e], eb[e], R.hi, R.lo);
    FF W;
    block_incl_scan_ff(sum_seg(w), wtot, &W);
    if (threadIdx.x == 0) a.wsum[(size_t)b * a.C + c] = make_float2(W.hi, W.lo);
}

template <int ELT, bool VEC>
__global__ void __launch_bounds__(kCT) sample_search_kernel(const FinalArgs a) {
    __shared__ FF wtot[kCW];
    __shared__ int s_sel, s_last;
    __shared__ FF s_lo;
    const int b = blockIdx.x, tid = threadIdx.x;
    pdl_wait();
    const SampleDesc d = a.desc[b];
    if (d.k < 0) return;
    bool rej = d.k < a.gamma;
    const FF R = rej ? normaliser_ratio(a, b, wtot) : FF{0.f, 0.f};

    // Chunk totals and their prefix; fall back to p_k if the residual is empty.
    FF T{0.f, 0.f}, S{0.f, 0.f}, incl{0.f, 0.f};
    for (int attempt = 0; attempt < 2; ++attempt) {
        T = FF{0.f, 0.f};
        if (tid < a.C) {
            if (rej) {
                const float2 q = a.wsum[(size_t)b * a.C + tid];
                T = FF{q.x, q.y};
            } else {
                const float4 q = a.zsum[(size_t)b * a.C + tid];
                T = FF{q.x, q.y};
            }
        }
        incl = block_incl_scan_ff(T, wtot, &S);
        if (S.hi > 0.f || !rej) break;
        rej = false;                                      // p_k equals q_k to rounding
    }
    if (!(S.hi > 0.f)) return;                            // unreachable for rows with a finite logit
    const FF excl = block_excl_from_incl(incl, wtot);
    FF target = ff_scale(a.u[(size_t)b * (a.gamma + 1) + a.gamma], S);
    if (!ff_lt(target, S))                                // u >= 1 clamps to the last token with mass
        target = ff_norm(FF{S.hi, S.lo - fabsf(S.hi) * 1.4210855e-14f});

    // The owning chunk: the one whose interval [excl, incl) holds the target.
    // The intervals tile [0, S) exactly, so there is one; the last chunk with
    // mass stands in should rounding ever leave a gap.
    if (tid == 0) { s_sel = -1; s_last = -1; }
    __syncthreads();
    bool has = tid < a.C && T.hi > 0.f;
    if (has && !ff_lt(target, excl) && ff_lt(target, incl)) { s_sel = tid; s_lo = excl; }
    if (has) atomicMax(&s_last, tid);
    __syncthreads();
    if (s_sel < 0 && tid == s_last) { s_sel = tid; s_lo = excl; }
    __syncthreads();
    const int cs = s_sel;
    const FF P = s_lo;
    __syncthreads();

    // Inside the chunk: the same weights and the same scan that produced its
    // total, so the thread intervals tile [P, P + T_cs) exactly.
    float ea[kPT], eb[kPT], w[kPT];
    chunk_exps<ELT, VEC>(a, b, d, cs, ea, eb);
#pragma unroll
    for (int e = 0; e < kPT; ++e) w[e] = rej ? resid(ea[e], eb[e], R.hi, R.lo) : ea[e];
    const FF ts = sum_seg(w);
    FF tot;
    const FF ti = block_incl_scan_ff(ts, wtot, &tot);
    const FF te = block_excl_from_incl(ti, wtot);
    const FF lo = ff_combine(P, te), hi = ff_combine(P, ti);
    if (tid == 0) { s_sel = -1; s_last = -1; }
    __syncthreads();
    has = ts.hi > 0.f;
    if (has && !ff_lt(target, lo) && ff_lt(target, hi)) s_sel = tid;
    if (has) atomicMax(&s_last, tid);
    __syncthreads();
    const int owner = s_sel >= 0 ? s_sel : s_last;
    if (tid == owner) {
        // first element whose inclusive prefix exceeds the target; the last
        // element with mass if rounding leaves none
        FF run{0.f, 0.f};
        int pick = -1, last = -1;
#pragma unroll
        for (int e = 0; e < kPT; ++e) {
            ff_add(run, w[e]);
            if (w[e] > 0.f) {
                last = e;
                if (pick < 0 && ff_lt(target, ff_combine(lo, ff_norm(run)))) pick = e;
            }
        }
        if (pick < 0) pick = last;
        if (pick >= 0)
            a.out_tok[(size_t)b * (a.gamma + 1) + d.k] = cs * kFinalChunk + tid * kPT + pick;
    }
}

// ---------------------------------------------------------------- launch
template <int ELT, bool VEC>
static cudaError_t launch_stats_t(const StatsArgs& sa, const DeviceInfo& di, cudaStream_t st) {
    static int occ = 0;                                   // blocks per SM, per template instance
    if (occ == 0) {
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, sample_rowstats_kernel<ELT, VEC>,
                                                          kThreads, 0) != cudaSuccess || o < 1)
            o = 1;
        occ = o;
    }
    long long g = (long long)di.sm_count * occ;
    if (sa.total_chunks < g) g = sa.total_chunks;
    sample_rowstats_kernel<ELT, VEC><<<(int)g, kThreads, 0, st>>>(sa);
    return cudaGetLastError();
}

// Launch with programmatic stream serialisation: the kernel may start while
// its predecessor drains and waits (griddepcontrol.wait) for its results.
template <typename K>
static cudaError_t launch_pdl(K kfn, dim3 grid, int threads, const FinalArgs& fa, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kfn, fa);
}

template <int ELT, bool VEC>
static cudaError_t launch_final_t(const FinalArgs& fa, cudaStream_t st) {
    cudaError_t e = launch_pdl(sample_decide_kernel<ELT>, dim3(fa.B), kDecideThreadsS, fa, st);
    if (e != cudaSuccess) return e;
    e = launch_pdl(sample_zsum_kernel<ELT, VEC>, dim3(fa.C, fa.B), kCT, fa, st);
    if (e != cudaSuccess) return e;
    e = launch_pdl(sample_wsum_kernel<ELT, VEC>, dim3(fa.C, fa.B), kCT, fa, st);
    if (e != cudaSuccess) return e;
    return launch_pdl(sample_search_kernel<ELT, VEC>, dim3(fa.B), kCT, fa, st);
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
    float2* parts_buf = reinterpret_cast<float2*>(w + L.part_off);
    const float s = (float)(1.4426950408889634 / (double)T);

    if (parts & kSampleStats) {
        StatsArgs sa;
        sa.zt = static_cast<const char*>(zt);
        sa.zd = static_cast<const char*>(zd);
        sa.s = s;
        sa.gamma = gamma;
        sa.V = V;
        sa.nseg = nseg(V, elt);
        sa.rows_per_seq = 2 * gamma + 1;
        sa.total_chunks = (long long)B * sa.rows_per_seq * sa.nseg;
        sa.parts = parts_buf;
        RingArgs ra;
        ra.zt = sa.zt;
        ra.zd = sa.zd;
        ra.gamma = gamma;
        ra.rows_per_seq = sa.rows_per_seq;
        ra.V = V;
        ra.nseg = sa.nseg;
        ra.total_chunks = sa.total_chunks;
        ra.s = s;
        ra.parts = parts_buf;
        ra.err = reinterpret_cast<int*>(w + L.err_off);
        bool used = false;
        e = elt == 2 ? launch_ring<2, false>(ra, di, st, &used) : launch_ring<4, false>(ra, di, st, &used);
        if (e != cudaSuccess) return e;
        if (!used) {
            if (elt == 2) e = vec ? launch_stats_t<2, true>(sa, di, st) : launch_stats_t<2, false>(sa, di, st);
            else e = vec ? launch_stats_t<4, true>(sa, di, st) : launch_stats_t<4, false>(sa, di, st);
            if (e != cudaSuccess) return e;
        }
    }
    if (parts & kSampleFinish) {
        FinalArgs fa;
        fa.zt = static_cast<const char*>(zt);
        fa.zd = static_cast<const char*>(zd);
        fa.x = x;
        fa.u = u;
        fa.T = T;
        fa.invT = 1.0f / T;
        fa.s = s;
        fa.B = B;
        fa.gamma = gamma;
        fa.V = V;
        fa.nseg = nseg(V, elt);
        fa.rows_per_seq = 2 * gamma + 1;
        fa.C = final_chunks(V);
        fa.parts = parts_buf;
        fa.desc = reinterpret_cast<SampleDesc*>(w + L.desc_off);
        fa.zsum = reinterpret_cast<float4*>(w + L.zsum_off);
        fa.wsum = reinterpret_cast<float2*>(w + L.wsum_off);
        fa.out_tok = out_tok;
        fa.out_acc = out_acc;
        fa.out_lp = out_lp;
        fa.err = reinterpret_cast<int*>(w + L.err_off);
        if (elt == 2) e = vec ? launch_final_t<2, true>(fa, st) : launch_final_t<2, false>(fa, st);
        else e = vec ? launch_final_t<4, true>(fa, st) : launch_final_t<4, false>(fa, st);
    }
    return e;
}

bool sample_supported_vocab(int V) {
    // the search kernel scans all chunk totals of a row in one CTA
    return final_chunks(V) <= kFinalChunkThreads;
}

}  // namespace sv
