// The final sample of stochastic verification: the sums of the exponentials
// of one target row (and, after a rejection, one draft row) over 1024-element
// segments, and the inverse-CDF search over those segment sums.  Shared by
// the standalone final-pass kernel (sv_sample.cu) and the consumer warps of
// the fused sampling kernel (sv_fused.cu).
//
// Source: "Speculative decoding: guess a few tokens first - why the answer
// stays the same", section "What happens in one round", step 4 (after a
// rejection at k draw from the residual, after a full acceptance draw the
// bonus token from p_gamma), and section "Why fixing wrong guesses does not
// leave the target distribution" (residual p'(x) = norm(max(0, p(x) - q(x)))).
//
// Every function here runs in a group of kCT = 256 threads (tid 0..255) that
// synchronises on named barrier 1 (fin_sync): a whole final-pass CTA, or the
// eight consumer warps of a fused-kernel CTA, whose producer warp never joins
// that barrier.
#pragma once

#include "sv_stream.cuh"

namespace sv {

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


// Named barrier 1 over the kCT threads of a final-pass group.
__device__ __forceinline__ void fin_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kCT) : "memory"); }

// Segment layout: warp w of a final-pass group sums one "segment" of kSeg
// consecutive elements, [j0, j0 + kSeg), with its lanes interleaved over
// 16-byte vectors (vector h of lane l starts at element j0 + (l + 32 h) 16/ELT),
// so every load instruction of a warp reads 512 contiguous bytes.  ldA(j) and
// ldB(j) return the 16-byte vector of the target and draft row starting at
// element j (-inf at or past V): plain global loads in the final-pass kernel,
// shared-memory stages in the fused kernel -- the same values either way, and
// the same arithmetic in the same order, so both give the same bits.
// Per segment: za = sum ea, and after a rejection zb = sum eb, w = sum max(0,
// ea - rt eb) at the approximate normaliser ratio rt, and dd = sum of eb over
// the elements with ea > rt eb -- minus the slope of w in the ratio.  The
// search turns w into the residual sum at the exact ratio R to first order,
// w - (R - rt) dd: the only elements the correction misses are those whose
// ea/eb lies between rt and R (~1e-6 apart), each off by at most |R - rt| eb.
template <int ELT, bool FAST, int NB, typename LdA, typename LdB>
__device__ __forceinline__ void segment_sums(const VerifyArgs& a, const FinalRows& f, int j0, int lane,
                                             float rt, LdA ldA, LdB ldB, FF* za, FF* zb, FF* w,
                                             float* dd) {
    constexpr int PV = 16 / ELT;
    constexpr int NV = kSeg / (32 * PV);                  // vectors per lane: 4 (bf16), 8 (fp32)
    constexpr int NP = 8 / ELT;                           // pairs per vector
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
            qa[h] = ldA(j);
            if (f.rej) qb[h] = ldB(j);
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

// Segment sums of segment `sg` of row pair f, loading from global memory, and
// their store in the workspace (lane 0).
template <int ELT, bool VEC>
__device__ __forceinline__ void segment_sums_global(const VerifyArgs& a, const FinalRows& f, int b, int sg,
                                                    float rt, int lane) {
    FF za, zb, w;
    float dd;
    auto ldA = [&](int j) { return load_vec<ELT, VEC>(f.ra, a.V, j); };
    auto ldB = [&](int j) { return load_vec<ELT, VEC>(f.rb, a.V, j); };
    if (f.fast) segment_sums<ELT, true, 4>(a, f, sg * kSeg, lane, rt, ldA, ldB, &za, &zb, &w, &dd);
    else segment_sums<ELT, false, 1>(a, f, sg * kSeg, lane, rt, ldA, ldB, &za, &zb, &w, &dd);
    if (lane == 0) {
        const size_t i = (size_t)b * a.C * kCW + sg;
        a.zsum[i] = make_float4(za.hi, za.lo, zb.hi, zb.lo);
        if (f.rej) a.wsum[i] = make_float4(w.hi, w.lo, dd, 0.f);
    }
}

// Inclusive scan of one float-float value per thread over the kCT-thread
// group in thread order; *total receives the group total.  Deterministic: the
// same inputs give the same bits in every group.
__device__ __forceinline__ FF block_incl_scan_ff(FF v, FF* wtot, FF* total, int tid) {
    const int lane = tid & 31, warp = tid >> 5;
    FF x = warp_incl_scan_ff(v);
    if (lane == 31) wtot[warp] = x;
    fin_sync();
    if (warp == 0) {
        FF y = lane < kCW ? wtot[lane] : FF{0.f, 0.f};
        y = warp_incl_scan_ff(y);
        if (lane < kCW) wtot[lane] = y;
    }
    fin_sync();
    const FF r = warp > 0 ? ff_combine(wtot[warp - 1], x) : x;
    *total = wtot[kCW - 1];
    fin_sync();
    return r;
}

// Exclusive counterpart of an inclusive group scan result r (thread order).
__device__ __forceinline__ FF block_excl_from_incl(FF r, const FF* wtot_scanned, int tid) {
    const int lane = tid & 31, warp = tid >> 5;
    const FF up = ff_shfl_up(r, 1);
    if (lane > 0) return up;
    return warp > 0 ? wtot_scanned[warp - 1] : FF{0.f, 0.f};
}

// The ratio Za / Zb of the two row normalisers of sequence b from each
// thread's share of the segment sums (one group reduction of both).
__device__ __forceinline__ FF normaliser_ratio_of(FF za, FF zb, FF* wtot, int tid) {
    const int lane = tid & 31, warp = tid >> 5;
    za = warp_sum_ff(za);
    zb = warp_sum_ff(zb);
    fin_sync();                                           // wtot may still be read by a caller's scan
    if (lane == 0) {
        wtot[warp] = za;
        wtot[kCW + warp] = zb;
    }
    fin_sync();
    FF Za{0.f, 0.f}, Zb{0.f, 0.f};
    for (int w = 0; w < kCW; ++w) {
        Za = ff_combine(Za, wtot[w]);
        Zb = ff_combine(Zb, wtot[kCW + w]);
    }
    fin_sync();
    return ff_div(Za, Zb);
}

// The same from the segment sums in the workspace (thread t takes segments
// t, t + kCT, ...).
__device__ __forceinline__ FF normaliser_ratio(const VerifyArgs& a, int b, FF* wtot, int tid) {
    const int ns = a.C * kCW;
    const float4* zs = a.zsum + (size_t)b * ns;
    FF za{0.f, 0.f}, zb{0.f, 0.f};
    for (int s = tid; s < ns; s += kCT) {
        const float4 q = __ldcg(&zs[s]);
        za = ff_combine(za, FF{q.x, q.y});
        zb = ff_combine(zb, FF{q.z, q.w});
    }
    return normaliser_ratio_of(za, zb, wtot, tid);
}

// The weights of the kSearchPT consecutive elements thread tid holds in
// segment sg: j = sg kSeg + kSearchPT tid + e.
template <int ELT, bool VEC, bool FAST>
__device__ __forceinline__ void search_weights(const VerifyArgs& a, const FinalRows& f, int sg,
                                               FF R, bool rej, float (&w)[kSearchPT], int tid) {
    static_assert(kSearchPT == 4, "one 8- or 16-byte load per row and thread");
    const int j = sg * kSeg + kSearchPT * tid;
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

// Shared memory of a final-pass group.
struct FinalSmem {
    FF wtot[2 * kCW];
    FF lo;
    int sel, last, seg;
    int mine;                 // final-pass kernel: this CTA finished its sequence's last chunk
};

// The search of sequence b, by one final-pass group once every segment sum
// of the row pair is in the workspace: the owning segment from the segment totals, then the
// owning element from that segment's weights, recomputed with the same
// arithmetic that produced its total.
template <int ELT, bool VEC>
__device__ __forceinline__ void search_sequence(const VerifyArgs& a, int b, const SampleDesc& d,
                                                FinalSmem& sm, int tid) {
    FF* wtot = sm.wtot;
    int& s_sel = sm.sel;
    int& s_last = sm.last;
    int& s_seg = sm.seg;
    FF& s_lo = sm.lo;
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
    if (rej) R = one ? normaliser_ratio_of(FF{qz.x, qz.y}, FF{qz.z, qz.w}, wtot, tid) : normaliser_ratio(a, b, wtot, tid);
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
        incl = block_incl_scan_ff(T, wtot, &S, tid);
        if (S.hi > 0.f || !rej) break;
        rej = false;                                      // p_k equals q_k to rounding
    }
    if (!(S.hi > 0.f)) return;                            // unreachable for rows with a finite logit
    const FF excl = block_excl_from_incl(incl, wtot, tid);
    FF target = ff_scale(a.u[(size_t)b * (a.gamma + 1) + a.gamma], S);
    if (!ff_lt(target, S))                                // u >= 1 clamps to the last token with mass
        target = ff_norm(FF{S.hi, S.lo - fabsf(S.hi) * 1.4210855e-14f});

    // The owning thread: the one whose interval [excl, incl) holds the target
    // (the intervals tile [0, S) exactly; the last thread with mass stands in
    // should rounding ever leave a gap), then its owning segment.
    if (tid == 0) { s_sel = -1; s_last = -1; }
    fin_sync();
    bool has = T.hi > 0.f;
    if (has && !ff_lt(target, excl) && ff_lt(target, incl)) s_sel = tid;
    if (has) atomicMax(&s_last, tid);
    fin_sync();
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
    fin_sync();
    const int sg = s_seg;
    const FF P = s_lo;
    fin_sync();

    // Inside the segment: kSearchPT consecutive elements per thread.
    const FinalRows f = final_rows<ELT>(a, b, d);
    float w[kSearchPT];
    if (f.fast) search_weights<ELT, VEC, true>(a, f, sg, R, rej, w, tid);
    else search_weights<ELT, VEC, false>(a, f, sg, R, rej, w, tid);
    FF ts{0.f, 0.f};
#pragma unroll
    for (int e = 0; e < kSearchPT; ++e) ff_add(ts, w[e]);
    ts = ff_norm(ts);
    FF tot;
    const FF ti = block_incl_scan_ff(ts, wtot, &tot, tid);
    const FF te = block_excl_from_incl(ti, wtot, tid);
    const FF lo = ff_combine(P, te), hi = ff_combine(P, ti);
    if (tid == 0) { s_sel = -1; s_last = -1; }
    fin_sync();
    has = ts.hi > 0.f;
    if (has && !ff_lt(target, lo) && ff_lt(target, hi)) s_sel = tid;
    if (has) atomicMax(&s_last, tid);
    fin_sync();
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

}  // namespace sv
