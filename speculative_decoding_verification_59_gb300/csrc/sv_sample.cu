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

// The ratio Za / Zb of the two row normalisers of sequence b, from the
// segment sums (block-wide, identical in every CTA that calls it).
__device__ __forceinline__ FF normaliser_ratio(const VerifyArgs& a, int b, FF* wtot) {
    const int ns = a.C * kCW;
    const float4* zs = a.zsum + (size_t)b * ns;
    FF za{0.f, 0.f}, zb{0.f, 0.f};
    for (int s = threadIdx.x; s < ns; s += kCT) {
        const float4 q = __ldcg(&zs[s]);
        za = ff_combine(za, FF{q.x, q.y});
        zb = ff_combine(zb, FF{q.z, q.w});
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
    decide_sample<ELT>(a, blockIdx.x, threadIdx.x, dsm);  // waits for the stream's partials
    write_sample_decision(a, blockIdx.x, threadIdx.x, dsm);
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
    FF wtot[kCW];
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
    const FF R = rej ? normaliser_ratio(a, b, wtot) : FF{0.f, 0.f};
    const int ns = a.C * kCW;                             // segments in the row
    const int G = (ns + kCT - 1) / kCT;                   // consecutive segments per thread
    // residual sums at the exact ratio: w(rt) - (R - rt) dd, to first order
    const float dR = (R.hi - d.rt) + R.lo;
    auto seg_total = [&](int s) -> FF {
        if (rej) {
            const float4 q = __ldcg(&a.wsum[(size_t)b * ns + s]);
            return ff_combine(FF{q.x, q.y}, FF{-dR * q.z, 0.f});
        }
        const float4 q = __ldcg(&a.zsum[(size_t)b * ns + s]);
        return FF{q.x, q.y};
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
            __threadfence();
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) sm.mine = take_ticket(&a.tick[b]) == (unsigned)(a.C - 1);
    __syncthreads();
    if (!sm.mine) return;
    search_sequence<ELT, VEC>(a, b, d, sm);
}

// ------------------------------------------------ lazy (early-exit) pass 1
// Source: "Speculative decoding: guess a few tokens first - why the answer
// stays the same", section "What happens in one round", step 3: drafts are
// checked left to right and the first rejection discards every later draft.
// The lazy pass therefore reads a position's two rows only while the drafts
// before it are accepted, give or take one position of look-ahead.
//
// One thread-block cluster of kLazyCluster CTAs per sequence; each CTA takes
// a fixed share of the block chunks of every row.  Per CTA:
//   producer warp   lane 0 copies the CTA's chunks of position p (target row
//                   p and draft row p; target row gamma last) into the same
//                   kind of bulk-copy ring as the full pass, but only for
//                   p <= (last position decided "accept") + 2;
//   8 consumer warps turn the copied chunks into the full pass's per-warp
//                   partials (warp_rowstats), position by position, exactly
//                   the positions the producer issued;
//   2 decision warps wait until every CTA of the cluster has the partials of
//                   position j, merge its two rows (merge_row_stats) and take
//                   the accept decision (accept_draft) -- the same arithmetic
//                   as the full pass, in every CTA alike, so every decision
//                   is bit-identical to it and all CTAs agree.
// The cluster barrier is used split: each role arrives at phase p when its
// part of position p is done and waits for phase p-1 only before arriving at
// p, so the streaming of position j+1 overlaps the decision on position j.
// Rows read per sequence: those of positions 0..min(k+1, gamma) after a
// rejection at k (2 gamma + 1 when all drafts are accepted).  The final
// sample runs the usual final-pass kernel.
constexpr int kLazyCluster = 4;
constexpr int kLazyDecWarps = 2;
constexpr int kLazyThreads = kRingThreads + 32 * kLazyDecWarps;
constexpr int kSmemSpinLimit = 1 << 22;

__device__ __forceinline__ unsigned cluster_ctarank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The two decision warps only.
__device__ __forceinline__ void decision_sync() {
    asm volatile("bar.sync 2, %0;" ::"n"(32 * kLazyDecWarps) : "memory");
}

// Bounded wait on a condition over shared memory.
template <typename Pred>
__device__ __forceinline__ bool smem_wait(Pred pred) {
    for (int i = 0; i < kSmemSpinLimit; ++i) {
        if (pred()) return true;
        __nanosleep(32);
    }
    return false;
}

template <int ELT>
__global__ void __launch_bounds__(kLazyThreads, 2) lazy_sample_kernel(const VerifyArgs a) {
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
    __shared__ float sM[2], slnZ[2], s_Mt, s_Md, s_Rt;
    __shared__ float s_lp[kMaxGamma], s_lq[kMaxGamma];
    __shared__ float s_zt[kMaxGamma], s_zd[kMaxGamma];   // z^t_i[x_i], z^d_i[x_i], gathered up front
    __shared__ int s_bad, s_ok, s_k;
    __shared__ volatile int s_limit, s_stop, s_issued, s_pdone;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned rank = cluster_ctarank();
    const int b = blockIdx.x / kLazyCluster;
    const size_t rowbytes = (size_t)a.V * ELT;
    const int P = a.nseg * kWarps;
    unsigned sg0, sg1;
    cta_range((unsigned)a.nseg, rank, kLazyCluster, &sg0, &sg1);
    const unsigned nmine = sg1 - sg0;                     // this CTA's block chunks of a row
    pdl_wait();

    if (threadIdx.x == 0) {
        for (int st = 0; st < kStages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], kWarps);
        }
        mbar_init_fence();
        int bad = 0;
        for (int i = 0; i < a.gamma; ++i) {
            const int xi = a.x[(size_t)b * a.gamma + i];
            if (xi < 0 || xi >= a.V) bad = SPEC_DEVERR_TOKEN_RANGE;
        }
        s_bad = bad;
        s_ok = 1;
        s_k = -1;
        s_Mt = s_Md = s_Rt = 0.f;
        s_limit = 1;
        s_stop = 0;
        s_issued = -1;
        s_pdone = 0;
    }
    for (int i = threadIdx.x; i < a.gamma; i += blockDim.x) {
        const int xi = a.x[(size_t)b * a.gamma + i];
        const bool in = xi >= 0 && xi < a.V;
        s_zt[i] = in ? load_logit<ELT>(sample_row(a, b, i, rowbytes), xi) : 0.f;
        s_zd[i] = in ? load_logit<ELT>(sample_row(a, b, a.gamma + 1 + i, rowbytes), xi) : 0.f;
    }
    __syncthreads();
    pdl_trigger();
    // rows of position p: chunk cc < nmine of target row p, else of draft row p
    auto row_of = [&](unsigned cc, int p) { return cc < nmine ? p : a.gamma + 1 + p; };

    if (!s_bad) {
        if (warp == 0) {
            // ---- producer
            unsigned issued = 0;
            bool ok = true;
            for (int p = 0; p <= a.gamma; ++p) {
                int go = 0;
                if (lane == 0) {
                    if (!smem_wait([&] { return s_stop != 0 || p <= s_limit; })) ok = false;
                    go = ok && !s_stop;
                    if (go) s_issued = p;
                    else s_pdone = 1;
                    __threadfence_block();
                    const unsigned nchunks = (p < a.gamma ? 2u : 1u) * nmine;
                    for (unsigned cc = 0; go && cc < nchunks; ++cc, ++issued) {
                        const int st = (int)(issued % kStages);
                        const unsigned use = issued / kStages;
                        if (use > 0 && !wait_bounded(&empty[st], (use - 1) & 1u)) {
                            ok = false;
                            break;
                        }
                        const int seg = (int)(sg0 + cc % nmine);
                        const size_t off = (size_t)seg * kStageBytes;
                        const uint32_t bytes = (uint32_t)min((size_t)kStageBytes, rowbytes - off);
                        mbar_arrive_expect_tx(&full[st], bytes);
                        bulk_g2s(ring + (size_t)st * kStageBytes,
                                 sample_row(a, b, row_of(cc, p), rowbytes) + off, bytes, &full[st]);
                    }
                    if (!ok) s_ok = 0;
                }
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) break;
                if (p > 0) cluster_wait();
                cluster_arrive();
            }
            if (lane == 0) {
                s_pdone = 1;
                // copies still in flight must land before the CTA may exit
                const unsigned first = issued > kStages ? issued - kStages : 0;
                for (unsigned i = first; i < issued; ++i)
                    if (!wait_bounded(&full[i % kStages], (i / kStages) & 1u)) {
                        atomicOr(a.err, SPEC_DEVERR_TIMEOUT);
                        break;
                    }
            }
        } else if (warp <= kWarps) {
            // ---- consumers: the positions the producer issued, in order
            const int cw = warp - 1;
            unsigned it = 0;
            bool ok = true;
            for (int p = 0;; ++p) {
                int have = 0;
                if (lane == 0) {
                    const bool w = smem_wait([&] { return s_issued >= p || s_pdone != 0; });
                    have = w && s_issued >= p;
                    if (!w) s_ok = 0;
                }
                have = __shfl_sync(0xffffffffu, have, 0);
                if (!have) break;
                const unsigned nchunks = (p < a.gamma ? 2u : 1u) * nmine;
                for (unsigned cc = 0; cc < nchunks; ++cc, ++it) {
                    const int st = (int)(it % kStages);
                    if (ok && !wait_bounded(&full[st], (it / kStages) & 1u)) ok = false;
                    const int seg = (int)(sg0 + cc % nmine);
                    const size_t off = (size_t)seg * kStageBytes;
                    const int bytes = (int)min((size_t)kStageBytes, rowbytes - off);
                    const int wb = bytes - cw * (32 * kLaneBytes);
                    const bool use = __all_sync(0xffffffffu, ok) && wb > 0;
                    float2 part = make_float2(kNegInf, 0.f);
                    if (use) {
                        uint4 v[kVecPerLane];
                        const unsigned char* chunk = ring + (size_t)st * kStageBytes + cw * (32 * kLaneBytes);
                        if (wb >= 32 * kLaneBytes) {
#pragma unroll
                            for (int t = 0; t < kVecPerLane; ++t)
                                v[t] = *reinterpret_cast<const uint4*>(chunk + (lane + 32 * t) * 16);
                        } else {
                            lane_words<ELT>(chunk, wb, v);
                        }
                        part = warp_rowstats<ELT>(v, a.s);
                    }
                    __syncwarp();
                    if (lane == 0) {
                        if (ok) mbar_arrive(&empty[st]);
                        a.parts[((size_t)b * a.rows_per_seq + row_of(cc, p)) * P + seg * kWarps + cw] = part;
                    }
                }
                if (!ok && lane == 0) s_ok = 0;
                if (p > 0) cluster_wait();
                cluster_arrive();                         // this CTA's partials of position p are written
            }
        } else {
            // ---- decision warps
            const int dw = warp - (kWarps + 1);
            for (int j = 0; j <= a.gamma; ++j) {
                cluster_arrive();
                cluster_wait();                           // every CTA's partials of position j are visible
                if (dw == 0 || j < a.gamma) {
                    float M, lnZ;
                    merge_row_stats(a, b, dw == 0 ? j : a.gamma + 1 + j, lane, &M, &lnZ);
                    if (lane == 0) { sM[dw] = M; slnZ[dw] = lnZ; }
                }
                decision_sync();
                if (dw == 0 && lane == 0) {
                    bool stop = true;
                    if (!s_ok) {
                        atomicOr(a.err, SPEC_DEVERR_TIMEOUT);
                        s_k = -1;
                    } else if (sM[0] == kNegInf || (j < a.gamma && sM[1] == kNegInf)) {
                        s_bad = SPEC_DEVERR_EMPTY_ROW;
                        s_k = -1;
                    } else if (j == a.gamma) {
                        s_k = a.gamma;                    // every draft accepted
                    } else {
                        const float lp = row_log_prob(s_zt[j], sM[0], slnZ[0], a);
                        const float lq = row_log_prob(s_zd[j], sM[1], slnZ[1], a);
                        s_lp[j] = lp;
                        s_lq[j] = lq;
                        if (accept_draft(lp, lq, a.u[(size_t)b * (a.gamma + 1) + j])) {
                            stop = false;
                            s_limit = j + 2;
                        } else {
                            s_k = j;
                        }
                    }
                    if (stop) {
                        s_Mt = sM[0];
                        s_Md = j < a.gamma ? sM[1] : 0.f;
                        s_Rt = j < a.gamma ? expf(slnZ[0] - slnZ[1]) : 0.f;   // as the decide step
                        s_stop = 1;
                    }
                    __threadfence_block();
                }
                decision_sync();
                if (s_stop) break;                        // the same in both warps and every CTA
            }
        }
    }
    // ---- outputs of the sequence: the decision warps of CTA 0
    if (rank != 0 || warp <= kWarps) return;
    const int t = threadIdx.x - (kWarps + 1) * 32;
    const int T = 32 * kLazyDecWarps;
    int k = s_k;
    if (s_bad) {
        k = -1;
        if (t == 0) atomicOr(a.err, s_bad);
    }
    if (t == 0) {
        a.out_acc[b] = k;
        SampleDesc d;
        d.k = k;
        d.mt = k >= 0 ? s_Mt : 0.f;
        d.md = (k >= 0 && k < a.gamma) ? s_Md : 0.f;
        d.rt = (k >= 0 && k < a.gamma) ? s_Rt : 0.f;
        a.desc[b] = d;
        a.tick[b] = 0u;
    }
    for (int i = t; i <= a.gamma; i += T)
        if (k < 0 || i != k)
            a.out_tok[(size_t)b * (a.gamma + 1) + i] = (k >= 0 && i < k) ? a.x[(size_t)b * a.gamma + i] : -1;
    if (a.out_lp)
        for (int i = t; i < a.gamma; i += T) {
            float* o = a.out_lp + ((size_t)b * a.gamma + i) * 2;
            const bool have = k >= 0 && i <= k;           // positions decided
            o[0] = have ? s_lp[i] : CUDART_NAN_F;
            o[1] = have ? s_lq[i] : CUDART_NAN_F;
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

template <int ELT>
static cudaError_t launch_lazy(const VerifyArgs& a, cudaStream_t st) {
    auto kfn = lazy_sample_kernel<ELT>;
    const int smem = kStages * kStageBytes;
    static DeviceSlots slots = {};                       // once per device: the opt-in
    int done = 0;
    cudaError_t e = device_once(slots, &done, [&](int, int* v) {
        *v = 1;
        return cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.B * kLazyCluster, 1, 1);
    cfg.blockDim = dim3(kLazyThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kLazyCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kfn, a);
}

// ---------------------------------------------------------------- launch
template <int ELT, bool VEC>
static cudaError_t launch_final_t(const VerifyArgs& a, cudaStream_t st, bool decide = true) {
    cudaError_t e = cudaSuccess;
    if (decide) {
        e = launch_pdl(sample_decide_kernel<ELT>, dim3(a.B), kGroup, 0, st, a);
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
            e = elt == 2 ? launch_lazy<2>(a, st) : launch_lazy<4>(a, st);
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
