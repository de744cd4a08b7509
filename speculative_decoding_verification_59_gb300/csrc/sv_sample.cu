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
// index order.  Four kernels, chained with programmatic dependent launch,
// keep every sequence in flight at once:
//   sample_decide_kernel  one CTA per sequence: row statistics from the
//                         partials, the accept decisions, every output but
//                         the final token;
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
#include "sv_stream.cuh"

namespace sv {

#ifndef SV_FINAL_EXACT_EXP
#define SV_FINAL_EXACT_EXP 0
#endif


// ---------------------------------------------------------------- pass 2
constexpr int kCT = kFinalChunkThreads;        // threads per chunk CTA (kFinalPerThread elements each)
constexpr int kCW = kCT / 32;

// exp((z - m) / T) for the final pass, as 2^x with x = (z - m) log2(e)/T
// carried in two floats: x_hi into the special-function unit, x_lo through
// the first-order factor (1 + x_lo ln 2).  Measured against exact values on
// GB300 the result has a relative error of mean -4.9e-8 and RMS 6.4e-8 over
// bf16 logits in [-25, 0] -- the mean is a common factor of every weight,
// which the normalisation cancels, and the rest matches expf's 3.8e-8 RMS at
// less than half its instruction count.  SV_FINAL_EXACT_EXP=1 selects expf
// with a two-float argument instead (for accuracy studies).
constexpr float kLn2 = 0.6931471805599453f;

template <int ELT>
__device__ __forceinline__ float final_exp(float z, float m, const VerifyArgs& a) {
    float d_hi = z - m, d_lo = 0.f;                       // exact for two bf16 values
    if constexpr (ELT == 4) {
        const float bb = d_hi - z;
        d_lo = (z - (d_hi - bb)) + (-m - bb);
    }
#if SV_FINAL_EXACT_EXP
    if (d_hi == kNegInf) return 0.f;
    const float y = d_hi * a.invT;
    const float rem = fmaf(-y, a.T, d_hi) + d_lo;
    const float e = expf(y);
    return fmaf(e, rem * a.invT, e);
#else
    const float xh = d_hi * a.s;
    if (xh == kNegInf) return 0.f;                        // masked logit, or far below the max
    const float xl = fmaf(d_hi, a.s, -xh) + fmaf(d_hi, a.s_lo, d_lo * a.s);
    const float c = ex2_approx(xh);
    return fmaf(c, xl * kLn2, c);
#endif
}

// Kahan-compensated running sum (four float operations per term).
struct KSum {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float x) {
        const float y = x - c;
        const float t = s + y;
        c = (t - s) - y;
        s = t;
    }
    __device__ __forceinline__ FF value() const { return ff_norm(FF{s, -c}); }
};

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

// The kPT logits of row `row` this thread holds in chunk c, lane-interleaved
// 16-byte vectors (coalesced): vector h is number tid + kCT h of the chunk.
// Entries at or beyond V are -inf.
template <int ELT, bool VEC>
__device__ __forceinline__ void load_interleaved(const char* row, int V, int c, float (&z)[kPT]) {
    constexpr int PV = 16 / ELT;
    const int j00 = c * kFinalChunk;
    if constexpr (VEC) {
        uint4 q[kPT / PV];
#pragma unroll
        for (int h = 0; h < kPT / PV; ++h) {
            const int jj = j00 + ((int)threadIdx.x + kCT * h) * PV;
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
                    const int jj = j00 + ((int)threadIdx.x + kCT * h) * PV;
                    z[PV * h + e] = jj < V ? __uint_as_float(u4_get(q[h], e)) : kNegInf;
                }
            }
    } else {
#pragma unroll
        for (int h = 0; h < kPT / PV; ++h)
#pragma unroll
            for (int e = 0; e < PV; ++e) {
                const int j = j00 + ((int)threadIdx.x + kCT * h) * PV + e;
                z[PV * h + e] = j < V ? load_logit<ELT>(row, j) : kNegInf;
            }
    }
}

// The exponentials of this thread's kPT elements of chunk c of the
// sequence's target row k (ea) and draft row k (eb, rejections only), in the
// interleaved layout (CONTIG = false) or as one contiguous run (CONTIG = true,
// index order, for the search).
template <int ELT, bool VEC, bool CONTIG>
__device__ __forceinline__ void chunk_exps(const VerifyArgs& a, int b, const SampleDesc& d, int c,
                                           float (&ea)[kPT], float (&eb)[kPT]) {
    const bool rej = d.k < a.gamma;
    const size_t rowbytes = (size_t)a.V * ELT;
    const char* rt = a.zt + ((size_t)b * (a.gamma + 1) + d.k) * rowbytes;
    const char* rd = a.zd + ((size_t)b * a.gamma + d.k) * rowbytes;
    float zt[kPT], zd[kPT];
    if constexpr (CONTIG) {
        const int j0 = c * kFinalChunk + threadIdx.x * kPT;
        load_seg<ELT, VEC>(rt, a.V, j0, zt);
        if (rej) load_seg<ELT, VEC>(rd, a.V, j0, zd);
    } else {
        load_interleaved<ELT, VEC>(rt, a.V, c, zt);
        if (rej) load_interleaved<ELT, VEC>(rd, a.V, c, zd);
    }
#pragma unroll
    for (int e = 0; e < kPT; ++e) {
        ea[e] = final_exp<ELT>(zt[e], d.mt, a);
        eb[e] = rej ? final_exp<ELT>(zd[e], d.md, a) : 0.f;
    }
}

// Residual weight max(0, p_k - q_k) scaled by Za: ea - (Za/Zb) eb, with the
// ratio as a float-float pair (Rhi, Rlo).
__device__ __forceinline__ float resid(float ea, float eb, float Rhi, float Rlo) {
    return fmaxf(fmaf(-Rlo, eb, fmaf(-Rhi, eb, ea)), 0.f);
}

__device__ __forceinline__ FF sum_seg(const float (&w)[kPT]) {
    KSum acc;
#pragma unroll
    for (int e = 0; e < kPT; ++e) acc.add(w[e]);
    return acc.value();
}

// The ratio Za / Zb of the two row normalisers of sequence b, from the chunk
// sums (block-wide, identical in every CTA that calls it).
__device__ __forceinline__ FF normaliser_ratio(const VerifyArgs& a, int b, FF* wtot) {
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

// One CTA per sequence: the accept decisions and every output but the final
// token, and the SampleDesc the chunk kernels read.
template <int ELT>
__global__ void __launch_bounds__(kGroup) sample_decide_kernel(const VerifyArgs a) {
    __shared__ SampleDecideSmem dsm;
    pdl_trigger();
    pdl_wait();                                           // the stream's partials are visible
    decide_sample<ELT>(a, blockIdx.x, threadIdx.x, dsm);
    write_sample_decision(a, blockIdx.x, threadIdx.x, dsm);
}

template <int ELT, bool VEC>
__global__ void __launch_bounds__(kCT) sample_zsum_kernel(const VerifyArgs a) {
    __shared__ FF wtot[kCW];
    const int b = blockIdx.x, c = blockIdx.y;
    pdl_trigger();
    pdl_wait();
    const SampleDesc d = a.desc[b];
    if (d.k < 0) return;
    float ea[kPT], eb[kPT];
    chunk_exps<ELT, VEC, false>(a, b, d, c, ea, eb);
    FF Za, Zb;
    block_incl_scan_ff(sum_seg(ea), wtot, &Za);
    block_incl_scan_ff(sum_seg(eb), wtot, &Zb);
    if (threadIdx.x == 0) a.zsum[(size_t)b * a.C + c] = make_float4(Za.hi, Za.lo, Zb.hi, Zb.lo);
}

template <int ELT, bool VEC>
__global__ void __launch_bounds__(kCT) sample_wsum_kernel(const VerifyArgs a) {
    __shared__ FF wtot[kCW];
    const int b = blockIdx.x, c = blockIdx.y;
    pdl_trigger();
    pdl_wait();
    const SampleDesc d = a.desc[b];
    if (d.k < 0 || d.k >= a.gamma) return;               // bonus rows use the exponential sums
    const FF R = normaliser_ratio(a, b, wtot);
    float ea[kPT], eb[kPT], w[kPT];
    chunk_exps<ELT, VEC, false>(a, b, d, c, ea, eb);
#pragma unroll
    for (int e = 0; e < kPT; ++e) w[e] = resid(ea[e], eb[e], R.hi, R.lo);
    FF W;
    block_incl_scan_ff(sum_seg(w), wtot, &W);
    if (threadIdx.x == 0) a.wsum[(size_t)b * a.C + c] = make_float2(W.hi, W.lo);
}

template <int ELT, bool VEC>
__global__ void __launch_bounds__(kCT) sample_search_kernel(const VerifyArgs a) {
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
    chunk_exps<ELT, VEC, true>(a, b, d, cs, ea, eb);
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
// Launch with programmatic stream serialisation: the kernel may start while
// its predecessor drains and waits (griddepcontrol.wait) for its results.
template <typename K>
static cudaError_t launch_pdl(K kfn, dim3 grid, int threads, const VerifyArgs& a, cudaStream_t st) {
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
    return cudaLaunchKernelEx(&cfg, kfn, a);
}

template <int ELT, bool VEC>
static cudaError_t launch_final_t(const VerifyArgs& a, cudaStream_t st) {
    cudaError_t e = launch_pdl(sample_decide_kernel<ELT>, dim3(a.B), kGroup, a, st);
    if (e != cudaSuccess) return e;
    e = launch_pdl(sample_zsum_kernel<ELT, VEC>, dim3(a.B, a.C), kCT, a, st);
    if (e != cudaSuccess) return e;
    e = launch_pdl(sample_wsum_kernel<ELT, VEC>, dim3(a.B, a.C), kCT, a, st);
    if (e != cudaSuccess) return e;
    return launch_pdl(sample_search_kernel<ELT, VEC>, dim3(a.B), kCT, a, st);
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
    a.desc = reinterpret_cast<SampleDesc*>(w + L.desc_off);
    a.zsum = reinterpret_cast<float4*>(w + L.zsum_off);
    a.wsum = reinterpret_cast<float2*>(w + L.wsum_off);
    a.err = reinterpret_cast<int*>(w + L.err_off);
    a.out_tok = out_tok;
    a.out_acc = out_acc;
    a.out_lp = out_lp;

    if (parts & kSampleStats) {
        e = elt == 2 ? launch_stream<2, kModeSample>(a, di, st) : launch_stream<4, kModeSample>(a, di, st);
        if (e != cudaSuccess) return e;
    }
    if (parts & kSampleFinish) {
        if (elt == 2) e = vec ? launch_final_t<2, true>(a, st) : launch_final_t<2, false>(a, st);
        else e = vec ? launch_final_t<4, true>(a, st) : launch_final_t<4, false>(a, st);
    }
    return e;
}

bool sample_supported_vocab(int V) {
    // the search kernel scans all chunk totals of a row in one CTA
    return final_chunks(V) <= kFinalChunkThreads;
}

}  // namespace sv
