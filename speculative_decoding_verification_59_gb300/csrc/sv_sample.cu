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
// index order.  Two kernels, chained with programmatic dependent launch,
// keep every sequence in flight at once:
//   sample_decide_kernel  one CTA per sequence: row statistics from the
//                         partials, the accept decisions, every output but
//                         the final token, and the approximate normaliser
//                         ratio rt = Z_t/Z_d of row k from those statistics;
//   sample_final_kernel   one CTA per 8192-element chunk of row k, one warp
//                         per 1024-element segment: sums of the exponentials
//                         of the target and draft segment and, after a
//                         rejection, the residual sum at ratio rt with its
//                         slope.  The sequence's last chunk CTA to finish (a
//                         ticket count) then runs the search: the exact ratio
//                         R from the exponential sums, the segment residual
//                         sums moved from rt to R to first order, prefix over
//                         them, the owning segment, its 1024 weights
//                         recomputed at R and scanned, the owning element.
// The weights are formed from the very exponentials whose sums normalise them
// (the same arithmetic in every kernel), and all sums are float-float (about
// 48 bits): the CDF each sequence samples from stays within ~1e-9 of the
// exact one, which matters because the long tail of a 150K-token vocabulary
// puts CDF boundaries ~1e-7 apart.
#include <stdlib.h>

#include "sv_stream.cuh"

namespace sv {


// ---------------------------------------------------------------- pass 2
constexpr int kCT = kFinalChunkThreads;        // threads per chunk CTA
constexpr int kCW = kCT / 32;                  // warps per chunk CTA = segments per chunk
constexpr int kSeg = kFinalChunk / kCW;        // elements per segment (1024)
constexpr int kSearchPT = kSeg / kCT;          // elements per thread in the search (4)
constexpr float kLn2 = 0.6931471805599453f;

// exp((z - m)/T) for the final pass, as 2^x with x = (z - m) log2(e)/T
// carried in two floats: x_hi into the special-function unit, x_lo through
// the first-order factor (1 + x_lo ln 2).  Measured against exact values on
// GB300 the result has a relative error of mean -4.9e-8 and RMS 6.4e-8 over
// bf16 logits in [-25, 0]; the mean is a common factor of every weight, which
// the normalisation cancels.  A single rounding of x, which reaches ~100 in
// magnitude, would cost up to 4e-6 per term.
//
// Two versions compute the same quantity.  The fast one works on pairs of
// logits with packed f32x2 arithmetic; it first raises every logit to a row
// floor m - 200/T' (T' = 1/s), below which the exponential flushes to zero
// anyway, so that no argument overflows and masked (-inf) logits need no
// test.  The guarded scalar one serves rows whose maximum or temperature is
// too extreme for that floor.

// Row constants of the fast version.
struct RowExp {
    f32x2 nm2;         // (-m, -m)
    f32x2 nmsh2;       // (-ms_hi, -ms_hi): m s as float-float (fp32 logits)
    f32x2 mslo2;       // (ms_lo, ms_lo)
    float floor;       // logits below this are raised to it
    uint32_t floor2;   // the floor as a packed bfloat16 pair (rounded down)
    float m;
};

// Packed temperature constants.
struct ExpK {
    f32x2 s2, ns2, slo2, nslo2, ln2_2, nln2_2;
};

__device__ __forceinline__ ExpK exp_consts(const VerifyArgs& a) {
    return ExpK{f2_pack(a.s, a.s), f2_pack(-a.s, -a.s), f2_pack(a.s_lo, a.s_lo),
                f2_pack(-a.s_lo, -a.s_lo), f2_pack(kLn2, kLn2), f2_pack(-kLn2, -kLn2)};
}

// Whether a row with maximum m can take the fast version: the floor
// m - 200/s must be finite and well below m.
__device__ __forceinline__ bool fast_row(float m, float s) {
    return fabsf(m) < 1e30f && s > 1e-30f && s < 1e30f && 200.f / s >= fabsf(m) * (1.f / 65536.f);
}

__device__ __forceinline__ RowExp row_exp(float m, const VerifyArgs& a) {
    RowExp r;
    r.m = m;
    r.nm2 = f2_pack(-m, -m);
    const float hi = m * a.s;
    const float lo = fmaf(m, a.s, -hi) + m * a.s_lo;
    r.nmsh2 = f2_pack(-hi, -hi);
    r.mslo2 = f2_pack(lo, lo);
    r.floor = m - 200.f / a.s;
    // bfloat16 rounding toward -inf: truncate positives, round negatives away from zero
    uint32_t fb = __float_as_uint(r.floor);
    fb = (fb & 0x80000000u) ? ((fb + 0xffffu) & 0xffff0000u) : (fb & 0xffff0000u);
    r.floor2 = (fb >> 16) | (fb & 0xffff0000u);
    return r;
}

// Fast version for the two bfloat16 logits packed in w.  z - m is exact for
// bfloat16 values of comparable magnitude, and its product with s splits
// exactly into x_hi + x_lo through one FMA: x_hi = d s rounded, then
// -x_lo = (x_hi - d s) - d s_lo, scaled by -ln 2 into the factor (1 + x_lo ln 2)
// -- an arrangement without negated operands.
__device__ __forceinline__ f32x2 exp_pair_bf16(uint32_t w, const RowExp& r, const ExpK& k) {
    asm("max.bf16x2 %0, %0, %1;" : "+r"(w) : "r"(r.floor2));
    const f32x2 d = f2_add(f2_pack(bf16_lo(w), bf16_hi(w)), r.nm2);
    const f32x2 xh = f2_mul(d, k.s2);
    const f32x2 nxl = f2_fma(d, k.nslo2, f2_fma(d, k.ns2, xh));   // -x_lo
    float h0, h1;
    f2_unpack(xh, h0, h1);
    const f32x2 c = f2_pack(ex2_approx(h0), ex2_approx(h1));
    return f2_fma(c, f2_mul(nxl, k.nln2_2), c);
}

// Fast version for two fp32 logits: z s - m s with z s split exactly
// (TwoProd through an FMA) and m s precomputed as float-float.
__device__ __forceinline__ f32x2 exp_pair_f32(float z0, float z1, const RowExp& r, const ExpK& k) {
    const f32x2 z = f2_pack(fmaxf(z0, r.floor), fmaxf(z1, r.floor));
    const f32x2 p = f2_mul(z, k.s2);                      // z s, rounded
    const f32x2 npe = f2_fma(z, k.ns2, p);                // p - z s, exact
    const f32x2 xh = f2_add(p, r.nmsh2);                  // x_hi = p - (m s)_hi
    const f32x2 nxl = f2_fma(z, k.nslo2, f2_add(npe, r.mslo2));   // -x_lo
    float h0, h1;
    f2_unpack(xh, h0, h1);
    const f32x2 c = f2_pack(ex2_approx(h0), ex2_approx(h1));
    return f2_fma(c, f2_mul(nxl, k.nln2_2), c);
}

// Guarded scalar version: any finite m and temperature, -inf logits give 0.
template <int ELT>
__device__ __forceinline__ float exp_guarded(float z, float m, const VerifyArgs& a) {
    float d_hi = z - m, d_lo = 0.f;                       // exact for two bf16 values
    if constexpr (ELT == 4) {
        const float bb = d_hi - z;
        d_lo = (z - (d_hi - bb)) + (-m - bb);
    }
    const float xh = d_hi * a.s;
    if (!(xh > kNegInf)) return 0.f;                      // masked logit, or far below the max
    const float xl = fmaf(d_hi, a.s, -xh) + fmaf(d_hi, a.s_lo, d_lo * a.s);
    const float c = ex2_approx(xh);
    return fmaf(c, xl * kLn2, c);
}

// The exponentials of the first NP pairs of logits in one 16-byte vector,
// as packed pairs in index order (a vector holds 4 pairs of bfloat16 logits,
// 2 pairs of fp32 ones).
template <int ELT, bool FAST, int NP = 8 / ELT>
__device__ __forceinline__ void vec_exps(const uint4& q, const RowExp& r, const ExpK& k,
                                         const VerifyArgs& a, f32x2 (&e)[NP]) {
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        if constexpr (FAST) {
            if constexpr (ELT == 2) e[i] = exp_pair_bf16(u4_get(q, i), r, k);
            else e[i] = exp_pair_f32(__uint_as_float(u4_get(q, 2 * i)),
                                     __uint_as_float(u4_get(q, 2 * i + 1)), r, k);
        } else {
            float z0, z1;
            if constexpr (ELT == 2) {
                z0 = bf16_lo(u4_get(q, i));
                z1 = bf16_hi(u4_get(q, i));
            } else {
                z0 = __uint_as_float(u4_get(q, 2 * i));
                z1 = __uint_as_float(u4_get(q, 2 * i + 1));
            }
            e[i] = f2_pack(exp_guarded<ELT>(z0, r.m, a), exp_guarded<ELT>(z1, r.m, a));
        }
    }
}

// 16 bytes of logits starting at element j (a multiple of 16/ELT); elements
// at or past V read as -inf.  VEC: 16-byte aligned rows and V a multiple of
// 16/ELT, so a vector is either wholly inside the row or wholly outside.
template <int ELT, bool VEC>
__device__ __forceinline__ uint4 load_vec(const char* row, int V, int j) {
    const uint32_t ninf = ELT == 4 ? 0xff800000u : 0xff80ff80u;
    if constexpr (VEC) {
        return j < V ? ld_stream16(row + (size_t)j * ELT) : make_uint4(ninf, ninf, ninf, ninf);
    } else {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (ELT == 4) {
                w[i] = j + i < V ? __ldg(reinterpret_cast<const uint32_t*>(row) + j + i) : ninf;
            } else {
                const unsigned short* r16 = reinterpret_cast<const unsigned short*>(row);
                const uint32_t lo = j + 2 * i < V ? __ldg(r16 + j + 2 * i) : 0xff80u;
                const uint32_t hi = j + 2 * i + 1 < V ? __ldg(r16 + j + 2 * i + 1) : 0xff80u;
                w[i] = lo | (hi << 16);
            }
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Kahan-compensated running sums of a pair of floats (packed).
struct KSum2 {
    f32x2 s = 0ull, c = 0ull;
    __device__ __forceinline__ void add(f32x2 x) {
        const f32x2 y = f2_sub(x, c);
        const f32x2 t = f2_add(s, y);
        c = f2_sub(f2_sub(t, s), y);
        s = t;
    }
    __device__ __forceinline__ FF value() const {
        float s0, s1, c0, c1;
        f2_unpack(s, s0, s1);
        f2_unpack(c, c0, c1);
        return ff_combine(ff_norm(FF{s0, -c0}), ff_norm(FF{s1, -c1}));
    }
};

// Residual weights max(0, ea - R eb) of a pair (R = Za / Zb as (Rhi, Rlo)),
// i.e. max(0, p - q) scaled by Za.
__device__ __forceinline__ f32x2 resid_pair(f32x2 ea, f32x2 eb, f32x2 nRhi2, f32x2 nRlo2) {
    float w0, w1;
    f2_unpack(f2_fma(nRlo2, eb, f2_fma(nRhi2, eb, ea)), w0, w1);
    return f2_pack(fmaxf(w0, 0.f), fmaxf(w1, 0.f));
}

// The sequence's final-pass rows: target row k (a) and, after a rejection,
// draft row k (b).
struct FinalRows {
    const char* ra;
    const char* rb;
    RowExp xa, xb;
    bool rej, fast;
};

template <int ELT>
__device__ __forceinline__ FinalRows final_rows(const VerifyArgs& a, int b, const SampleDesc& d) {
    FinalRows f;
    const size_t rowbytes = (size_t)a.V * ELT;
    f.rej = d.k < a.gamma;
    f.ra = a.zt + ((size_t)b * (a.gamma + 1) + d.k) * rowbytes;
    f.rb = f.rej ? a.zd + ((size_t)b * a.gamma + d.k) * rowbytes : f.ra;
    f.xa = row_exp(d.mt, a);
    f.xb = row_exp(f.rej ? d.md : d.mt, a);
    f.fast = fast_row(d.mt, a.s) && (!f.rej || fast_row(d.md, a.s));
    return f;
}

// Segment layout of a chunk CTA: warp w covers the kSeg consecutive elements
// [c kFinalChunk + w kSeg, + kSeg) -- one "segment" -- with its lanes
// interleaved over 16-byte vectors (vector h of lane l starts at element
// (l + 32 h) 16/ELT of the segment), so every load instruction of a warp
// reads 512 contiguous bytes.  Per segment: za = sum ea, and after a
// rejection zb = sum eb, w = sum max(0, ea - rt eb) at the approximate
// normaliser ratio rt, and dd = sum of eb over the elements with
// ea > rt eb -- minus the slope of w in the ratio.  The search turns w into
// the residual sum at the exact ratio R to first order, w - (R - rt) dd: the
// only elements the correction misses are those whose ea/eb lies between rt
// and R (~1e-6 apart), each off by at most |R - rt| eb.
template <int ELT, bool VEC, bool FAST>
__device__ __forceinline__ void segment_sums(const VerifyArgs& a, const FinalRows& f, int c,
                                             float rt, FF* za, FF* zb, FF* w, float* dd) {
    constexpr int PV = 16 / ELT;
    constexpr int NV = kSeg / (32 * PV);                  // vectors per lane: 4 (bf16), 8 (fp32)
    constexpr int NB = FAST ? 4 : 1;                      // vectors per load batch
    constexpr int NP = 8 / ELT;                           // pairs per vector
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int j0 = c * kFinalChunk + warp * kSeg;
    const ExpK k = exp_consts(a);
    const f32x2 nrt2 = f2_pack(-rt, -rt);
    KSum2 ka, kb, kw;
    f32x2 d2 = f2_pack(0.f, 0.f);
#pragma unroll
    for (int h0 = 0; h0 < NV; h0 += NB) {
        uint4 qa[NB], qb[NB];
#pragma unroll
        for (int h = 0; h < NB; ++h) {
            const int j = j0 + (lane + 32 * (h0 + h)) * PV;
            qa[h] = load_vec<ELT, VEC>(f.ra, a.V, j);
            if (f.rej) qb[h] = load_vec<ELT, VEC>(f.rb, a.V, j);
        }
#pragma unroll
        for (int h = 0; h < NB; ++h) {
            f32x2 ea[NP], eb[NP];
            vec_exps<ELT, FAST>(qa[h], f.xa, k, a, ea);
            if (f.rej) vec_exps<ELT, FAST>(qb[h], f.xb, k, a, eb);
#pragma unroll
            for (int i = 0; i < NP; ++i) {
                ka.add(ea[i]);
                if (f.rej) {
                    kb.add(eb[i]);
                    float t0, t1, b0, b1;
                    f2_unpack(f2_fma(nrt2, eb[i], ea[i]), t0, t1);
                    f2_unpack(eb[i], b0, b1);
                    kw.add(f2_pack(fmaxf(t0, 0.f), fmaxf(t1, 0.f)));
                    d2 = f2_add(d2, f2_pack(t0 > 0.f ? b0 : 0.f, t1 > 0.f ? b1 : 0.f));
                }
            }
        }
    }
    *za = warp_sum_ff(ka.value());
    if (f.rej) {
        *zb = warp_sum_ff(kb.value());
        *w = warp_sum_ff(kw.value());
        float d0, d1;
        f2_unpack(d2, d0, d1);
        *dd = warp_sum(d0 + d1);
    } else {
        *zb = *w = FF{0.f, 0.f};
        *dd = 0.f;
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

// The ratio Za / Zb of the two row normalisers of sequence b from each
// thread's share of the segment sums (one block reduction of both).
__device__ __forceinline__ FF normaliser_ratio_of(FF za, FF zb, FF* wtot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    za = warp_sum_ff(za);
    zb = warp_sum_ff(zb);
    __syncthreads();                                      // wtot may still be read by a caller's scan
    if (lane == 0) {
        wtot[warp] = za;
        wtot[kCW + warp] = zb;
    }
    __syncthreads();
    FF Za{0.f, 0.f}, Zb{0.f, 0.f};
    for (int w = 0; w < kCW; ++w) {
        Za = ff_combine(Za, wtot[w]);
        Zb = ff_combine(Zb, wtot[kCW + w]);
    }
    __syncthreads();
    return ff_div(Za, Zb);
}

// The same from the segment sums in the workspace (thread t takes segments
// t, t + kCT, ...).
__device__ __forceinline__ FF normaliser_ratio(const VerifyArgs& a, int b, FF* wtot) {
    const int ns = a.C * kCW;
    const float4* zs = a.zsum + (size_t)b * ns;
    FF za{0.f, 0.f}, zb{0.f, 0.f};
    for (int s = threadIdx.x; s < ns; s += kCT) {
        const float4 q = __ldcg(&zs[s]);
        za = ff_combine(za, FF{q.x, q.y});
        zb = ff_combine(zb, FF{q.z, q.w});
    }
    return normaliser_ratio_of(za, zb, wtot);
}

// One CTA per sequence: the accept decisions and every output but the final
// token, and the SampleDesc the chunk kernels read.
// 16 warps: one row's partials per warp for gamma <= 7 (15 rows), so the
// merge is a single round of loads.
constexpr int kSampleDecideThreads = 512;

template <int ELT>
__global__ void __launch_bounds__(kSampleDecideThreads) sample_decide_kernel(const VerifyArgs a) {
    __shared__ SampleDecideSmem dsm;
    pdl_trigger();
    const int k = decide_sample<ELT, kSampleDecideThreads>(a, blockIdx.x, threadIdx.x, dsm);  // waits for the stream's partials
    write_sample_decision<kSampleDecideThreads>(a, blockIdx.x, threadIdx.x, k, dsm);
}

// The weights of the kSearchPT consecutive elements this thread holds in
// segment sg: j = sg kSeg + kSearchPT tid + e.
template <int ELT, bool VEC, bool FAST>
__device__ __forceinline__ void search_weights(const VerifyArgs& a, const FinalRows& f, int sg,
                                               FF R, bool rej, float (&w)[kSearchPT]) {
    static_assert(kSearchPT == 4, "one 8- or 16-byte load per row and thread");
    const int j = sg * kSeg + kSearchPT * (int)threadIdx.x;
    uint4 qa, qb;
    if constexpr (ELT == 4) {
        qa = load_vec<4, VEC>(f.ra, a.V, j);
        if (rej) qb = load_vec<4, VEC>(f.rb, a.V, j);
    } else {
        // four bfloat16 values: the low half of a 16-byte vector
        auto ld8 = [&](const char* row) -> uint4 {
            if constexpr (VEC) {
                if (j >= a.V) return make_uint4(0xff80ff80u, 0xff80ff80u, 0u, 0u);
                uint2 v;
                asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                    : "=r"(v.x), "=r"(v.y) : "l"(row + (size_t)j * 2));
                return make_uint4(v.x, v.y, 0u, 0u);
            } else {
                return load_vec<2, false>(row, a.V, j);   // elements past j + 3 are unused
            }
        };
        qa = ld8(f.ra);
        if (rej) qb = ld8(f.rb);
    }
    const ExpK k = exp_consts(a);
    const f32x2 nRhi2 = f2_pack(-R.hi, -R.hi), nRlo2 = f2_pack(-R.lo, -R.lo);
    f32x2 ea[2], eb[2];
    vec_exps<ELT, FAST, 2>(qa, f.xa, k, a, ea);
    if (rej) vec_exps<ELT, FAST, 2>(qb, f.xb, k, a, eb);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const f32x2 p = rej ? resid_pair(ea[i], eb[i], nRhi2, nRlo2) : ea[i];
        f2_unpack(p, w[2 * i], w[2 * i + 1]);
    }
}

// Shared memory of the final-pass CTAs.
struct FinalSmem {
    FF wtot[2 * kCW];
    FF lo;
    int sel, last, seg;
    int mine;                 // this CTA finished its sequence's last chunk
};

// The search of sequence b, by one whole CTA once every chunk's segment sums
// are in the workspace: the owning segment from the segment totals, then the
// owning element from that segment's weights, recomputed with the same
// arithmetic that produced its total.
template <int ELT, bool VEC>
__device__ __forceinline__ void search_sequence(const VerifyArgs& a, int b, const SampleDesc& d,
                                                FinalSmem& sm) {
    FF* wtot = sm.wtot;
    int& s_sel = sm.sel;
    int& s_last = sm.last;
    int& s_seg = sm.seg;
    FF& s_lo = sm.lo;
    const int tid = threadIdx.x;
    bool rej = d.k < a.gamma;
    const int ns = a.C * kCW;                             // segments in the row
    const int G = (ns + kCT - 1) / kCT;                   // consecutive segments per thread
    // With one segment per thread (V <= kCT kSeg) each thread loads its
    // segment's sums once, normaliser and residual sums together; otherwise
    // they are read where needed.
    const bool one = G == 1;
    float4 qz = make_float4(0.f, 0.f, 0.f, 0.f), qw = qz;
    if (one && tid < ns) {
        qz = __ldcg(&a.zsum[(size_t)b * ns + tid]);
        if (rej) qw = __ldcg(&a.wsum[(size_t)b * ns + tid]);
    }
    FF R{0.f, 0.f};
    if (rej) R = one ? normaliser_ratio_of(FF{qz.x, qz.y}, FF{qz.z, qz.w}, wtot) : normaliser_ratio(a, b, wtot);
    // residual sums at the exact ratio: w(rt) - (R - rt) dd, to first order
    const float dR = (R.hi - d.rt) + R.lo;
    auto seg_total = [&](int s) -> FF {
        const float4 q = one ? (rej ? qw : qz) : __ldcg(rej ? &a.wsum[(size_t)b * ns + s] : &a.zsum[(size_t)b * ns + s]);
        return rej ? ff_combine(FF{q.x, q.y}, FF{-dR * q.z, 0.f}) : FF{q.x, q.y};
    };

    // Thread totals over its segments and their prefix; fall back to p_k if
    // the residual is empty.
    FF T{0.f, 0.f}, S{0.f, 0.f}, incl{0.f, 0.f};
    for (int attempt = 0; attempt < 2; ++attempt) {
        T = FF{0.f, 0.f};
        for (int g = 0; g < G; ++g) {
            const int s = tid * G + g;
            if (s < ns) T = ff_combine(T, seg_total(s));
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

    // The owning thread: the one whose interval [excl, incl) holds the target
    // (the intervals tile [0, S) exactly; the last thread with mass stands in
    // should rounding ever leave a gap), then its owning segment.
    if (tid == 0) { s_sel = -1; s_last = -1; }
    __syncthreads();
    bool has = T.hi > 0.f;
    if (has && !ff_lt(target, excl) && ff_lt(target, incl)) s_sel = tid;
    if (has) atomicMax(&s_last, tid);
    __syncthreads();
    if (tid == (s_sel >= 0 ? s_sel : s_last)) {
        FF run = excl;
        int pick = -1, last = -1;
        FF plo = excl, llo = excl;
        for (int g = 0; g < G; ++g) {
            const int s = tid * G + g;
            if (s >= ns) break;
            const FF t = seg_total(s);
            const FF nxt = ff_combine(run, t);
            if (t.hi > 0.f) {
                last = s;
                llo = run;
                if (pick < 0 && ff_lt(target, nxt)) { pick = s; plo = run; }
            }
            run = nxt;
        }
        if (pick < 0) { pick = last; plo = llo; }
        s_seg = pick;
        s_lo = plo;
    }
    __syncthreads();
    const int sg = s_seg;
    const FF P = s_lo;
    __syncthreads();

    // Inside the segment: kSearchPT consecutive elements per thread.
    const FinalRows f = final_rows<ELT>(a, b, d);
    float w[kSearchPT];
    if (f.fast) search_weights<ELT, VEC, true>(a, f, sg, R, rej, w);
    else search_weights<ELT, VEC, false>(a, f, sg, R, rej, w);
    FF ts{0.f, 0.f};
#pragma unroll
    for (int e = 0; e < kSearchPT; ++e) ff_add(ts, w[e]);
    ts = ff_norm(ts);
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
        for (int e = 0; e < kSearchPT; ++e) {
            ff_add(run, w[e]);
            if (w[e] > 0.f) {
                last = e;
                if (pick < 0 && ff_lt(target, ff_combine(lo, ff_norm(run)))) pick = e;
            }
        }
        if (pick < 0) pick = last;
        if (pick >= 0)
            a.out_tok[(size_t)b * (a.gamma + 1) + d.k] = sg * kSeg + tid * kSearchPT + pick;
    }
}

// Ticket of a finished chunk: a gpu-scope acquire-release increment, so the
// CTA that draws the last ticket sees every other chunk's segment sums.
__device__ __forceinline__ unsigned take_ticket(unsigned* t) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(t) : "memory");
    return old;
}

// Per (chunk, sequence): the sums of the exponentials of target row k and
// (after a rejection) draft row k over each of the chunk's segments, and the
// residual sums at the approximate ratio with their slopes; then, in the
// last of the sequence's C chunk CTAs to finish, the search.  The decide
// kernel (or the lazy pass) zeroes the sequence's ticket count before this
// kernel's wait returns.
template <int ELT, bool VEC>
__global__ void __launch_bounds__(kCT, 4) sample_final_kernel(const VerifyArgs a) {
    __shared__ FinalSmem sm;
    const int b = blockIdx.x / a.C, c = blockIdx.x - b * a.C;   // chunks of a sequence adjacent
    pdl_trigger();
    pdl_wait();
    const SampleDesc d = a.desc[b];
    if (d.k < 0) return;
    {
        const FinalRows f = final_rows<ELT>(a, b, d);
        FF za, zb, w;
        float dd;
        if (f.fast) segment_sums<ELT, VEC, true>(a, f, c, d.rt, &za, &zb, &w, &dd);
        else segment_sums<ELT, VEC, false>(a, f, c, d.rt, &za, &zb, &w, &dd);
        if ((threadIdx.x & 31) == 0) {
            const size_t sg = ((size_t)b * a.C + c) * kCW + (threadIdx.x >> 5);
            a.zsum[sg] = make_float4(za.hi, za.lo, zb.hi, zb.lo);
            if (f.rej) a.wsum[sg] = make_float4(w.hi, w.lo, dd, 0.f);
        }
    }
    // The CTA's sums, ordered before the ticket by the barrier, are published
    // at gpu scope by the ticket thread's fence (the pattern of a grid-wide
    // barrier: bar.sync, then one thread fences and increments).
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        sm.mine = take_ticket(&a.tick[b]) == (unsigned)(a.C - 1);
    }
    __syncthreads();
    if (!sm.mine) return;
    search_sequence<ELT, VEC>(a, b, d, sm);
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
        a.desc[b] = d;
        a.tick[b] = 0u;
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
// variable SPEC_VERIFY_LAZY_SPLIT_BYTES overrides the figure (0: always
// split); outputs do not depend on it.
constexpr double kLazySplitBytes = 96.0 * (1 << 20);

static double lazy_split_bytes() {
    const char* e = getenv("SPEC_VERIFY_LAZY_SPLIT_BYTES");
    if (!e || !*e) return kLazySplitBytes;
    char* end = nullptr;
    const double v = strtod(e, &end);
    return (end && *end == '\0' && v >= 0.0) ? v : kLazySplitBytes;
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
template <int ELT, bool VEC>
static cudaError_t launch_final_t(const VerifyArgs& a, cudaStream_t st, bool decide = true) {
    cudaError_t e = cudaSuccess;
    if (decide) {
        e = launch_pdl(sample_decide_kernel<ELT>, dim3(a.B), kSampleDecideThreads, 0, st, a);
        if (e != cudaSuccess) return e;
    }
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
    a.tick = reinterpret_cast<unsigned*>(w + L.tick_off);
    a.zsum = reinterpret_cast<float4*>(w + L.zsum_off);
    a.wsum = reinterpret_cast<float4*>(w + L.wsum_off);
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
