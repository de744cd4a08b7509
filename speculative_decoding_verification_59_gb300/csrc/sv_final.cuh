// The final sample of stochastic verification: the sums of the exponentials
// of one target row (and, after a rejection, one draft row) over 1024-element
// segments, and the inverse-CDF search over those segment sums, for the
// final-pass kernel (sv_sample.cu).
//
// Source: "Speculative decoding: guess a few tokens first - why the answer
// stays the same", section "What happens in one round", step 4 (after a
// rejection at k draw from the residual, after a full acceptance draw the
// bonus token from p_gamma), and section "Why fixing wrong guesses does not
// leave the target distribution" (residual p'(x) = norm(max(0, p(x) - q(x)))).
//
// Every group function here runs in a final-pass CTA of kCT = 256 threads
// (tid 0..255), which synchronises on named barrier 1 (fin_sync).
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
// element j (-inf at or past V).
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
            // A vector's NP terms per packed lane are summed plainly, then the
            // sum enters the compensated running sum: each plain sum is off by
            // at most (NP - 1) ulp of itself, independently from vector to
            // vector, which leaves a segment total within ~u/8 of its value
            // (u = 2^-24) -- far inside what the search needs -- for a
            // quarter of the compensation work.
            f32x2 sa = ea[0];
#pragma unroll
            for (int i = 1; i < NP; ++i) sa = f2_add(sa, ea[i]);
            ka.add(sa);
            if (f.rej) {
                f32x2 sb = eb[0], sw = 0ull;
#pragma unroll
                for (int i = 1; i < NP; ++i) sb = f2_add(sb, eb[i]);
                kb.add(sb);
#pragma unroll
                for (int i = 0; i < NP; ++i) {
                    float t0, t1, b0, b1;
                    f2_unpack(f2_fma(nrt2, eb[i], ea[i]), t0, t1);
                    f2_unpack(eb[i], b0, b1);
                    sw = f2_add(sw, f2_pack(fmaxf(t0, 0.f), fmaxf(t1, 0.f)));
                    d2 = f2_add(d2, f2_pack(t0 > 0.f ? b0 : 0.f, t1 > 0.f ? b1 : 0.f));
                }
                kw.add(sw);
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
    const int j0 = sg * kSeg;
    auto ldA = [&](int j) { return load_vec<ELT, VEC>(f.ra, a.V, j); };
    auto ldB = [&](int j) { return load_vec<ELT, VEC>(f.rb, a.V, j); };
    if (f.fast) segment_sums<ELT, true, 4>(a, f, j0, lane, rt, ldA, ldB, &za, &zb, &w, &dd);
    else segment_sums<ELT, false, 1>(a, f, j0, lane, rt, ldA, ldB, &za, &zb, &w, &dd);
    if (lane == 0) {
        unsigned long long* p = a.sums + ((size_t)b * a.C * kCW + sg) * kSumWords;
        st_tagged2(p, __float_as_uint(za.hi), __float_as_uint(za.lo), a.ptag);
        st_tagged2(p + 2, __float_as_uint(zb.hi), __float_as_uint(zb.lo), a.ptag);
        st_tagged2(p + 4, __float_as_uint(w.hi), __float_as_uint(w.lo), a.ptag);
        st_tagged2(p + 6, __float_as_uint(dd), 0u, a.ptag);
    }
}

// The sums of segment s of sequence b, once they carry this call's tag
// (waiting, bounded, for a writer that may still run): za, zb, the residual
// sum w and its slope dd.
struct SegSums {
    FF za, zb, w;
    float dd;
};

__device__ __forceinline__ SegSums seg_sums(const VerifyArgs& a, size_t i) {
    const unsigned long long* p = a.sums + i * kSumWords;
    uint32_t v[8];
    for (uint32_t n = 0;; ++n) {
        bool ok = ld_tagged2(p, a.ptag, &v[0], &v[1]);
        ok &= ld_tagged2(p + 2, a.ptag, &v[2], &v[3]);
        ok &= ld_tagged2(p + 4, a.ptag, &v[4], &v[5]);
        ok &= ld_tagged2(p + 6, a.ptag, &v[6], &v[7]);
        if (ok) break;
        if (n >= a.wait_limit) {
            atomicOr(a.err, SPEC_DEVERR_TIMEOUT);
            break;
        }
        __nanosleep(100);
    }
    SegSums r;
    r.za = FF{__uint_as_float(v[0]), __uint_as_float(v[1])};
    r.zb = FF{__uint_as_float(v[2]), __uint_as_float(v[3])};
    r.w = FF{__uint_as_float(v[4]), __uint_as_float(v[5])};
    r.dd = __uint_as_float(v[6]);
    return r;
}

// Shared memory of a final-pass group.
struct FinalSmem {
    FF wv[kCW], wa[kCW], wb[kCW];   // per-warp totals: scanned sums, target and draft normalisers
    float wd[kCW];                  // per-warp totals of the residual slopes
    FF xs[kCT];                     // each thread's exclusive prefix (base of its segments)
    FF P;                           // base of the owning segment (several segments per thread)
    int sel, last, sel2, last2, seg;
    int mine;                       // final-pass kernel: this CTA finished its sequence's last chunk
    SampleDesc desc;                // final-pass kernel: the sequence's SampleDesc
};

// Inclusive float-float and float prefixes of one value per thread over the
// group, in thread order, from the per-warp totals in sm (written by each
// warp's lane 31 before the group barrier): *excl and *incl tile the range
// exactly -- thread t's incl and thread t+1's excl are the same bits -- and
// the last thread's incl equals *tot.
struct GroupPrefix {
    FF excl, incl, tot;
    float dexcl, dincl, dtot;
};

__device__ __forceinline__ GroupPrefix group_prefix(FF vin, float din, const FF* wv, const float* wd, int tid) {
    const int lane = tid & 31, warp = tid >> 5;
    FF acc{0.f, 0.f}, pre{0.f, 0.f};
    float dacc = 0.f, dpre = 0.f;
#pragma unroll
    for (int i = 0; i < kCW; ++i) {
        if (i == warp) { pre = acc; dpre = dacc; }
        acc = ff_combine(acc, wv[i]);
        dacc += wd[i];
    }
    const FF vex = ff_shfl_up(vin, 1);
    const float dex = __shfl_up_sync(0xffffffffu, din, 1);
    GroupPrefix g;
    g.excl = lane > 0 ? ff_combine(pre, vex) : pre;
    g.incl = ff_combine(pre, vin);
    g.dexcl = lane > 0 ? dpre + dex : dpre;
    g.dincl = dpre + din;
    g.tot = acc;
    g.dtot = dacc;
    return g;
}

// Inclusive warp scan of floats in lane order.
__device__ __forceinline__ float warp_incl_scan(float x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
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

// Segment totals of sequence b that thread tid sums: segments tid G ... tid G
// + G - 1 of the ns in the row.  za and zb are the target and draft
// normalisers' shares; v the quantity the search scans (the residual sums at
// rt after a rejection, else the target sums) and dv its slope in the ratio.
struct ThreadSums {
    FF za, zb, v;
    float dv;
};

__device__ __forceinline__ ThreadSums thread_sums(const VerifyArgs& a, int b, int ns, int G, bool rej, int tid) {
    ThreadSums t{{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, 0.f};
    for (int g = 0; g < G; ++g) {
        const int s = tid * G + g;
        if (s >= ns) break;
        const SegSums q = seg_sums(a, (size_t)b * ns + s);
        t.za = ff_combine(t.za, q.za);
        t.zb = ff_combine(t.zb, q.zb);
        if (rej) {
            t.v = ff_combine(t.v, q.w);
            t.dv += q.dd;
        }
    }
    if (!rej) t.v = t.za;
    return t;
}

// Group barrier phase of the search: the scanned quantity's prefixes and,
// after a rejection, the normalisers' totals.  One barrier.
__device__ __forceinline__ GroupPrefix scan_phase(const ThreadSums& t, bool rej, FinalSmem& sm, FF* Za,
                                                  FF* Zb, int tid) {
    const int lane = tid & 31, warp = tid >> 5;
    const FF vin = warp_incl_scan_ff(t.v);
    const float din = warp_incl_scan(rej ? t.dv : 0.f);
    FF za{0.f, 0.f}, zb{0.f, 0.f};
    if (rej) {
        za = warp_sum_ff(t.za);
        zb = warp_sum_ff(t.zb);
    }
    if (lane == 31) {
        sm.wv[warp] = vin;
        sm.wd[warp] = din;
        sm.wa[warp] = za;
        sm.wb[warp] = zb;
    }
    fin_sync();
    *Za = *Zb = FF{0.f, 0.f};
    if (rej)
#pragma unroll
        for (int i = 0; i < kCW; ++i) {
            *Za = ff_combine(*Za, sm.wa[i]);
            *Zb = ff_combine(*Zb, sm.wb[i]);
        }
    return group_prefix(vin, din, sm.wv, sm.wd, tid);
}

// x - d dR as float-float: a scanned residual sum moved from ratio rt to R
// to first order (dR = R - rt).  The same bits for the same inputs in every
// thread, so corrected prefixes still tile their range exactly.
__device__ __forceinline__ FF at_ratio(FF x, float d, float dR) { return ff_combine(x, FF{-dR * d, 0.f}); }

// The search of sequence b, by one final-pass group once every segment sum
// of the row pair is in the workspace: the owning segment from the segment
// totals, then the owning element from that segment's weights, recomputed
// with the same arithmetic that produced its total.  u is the sequence's
// uniform for the final token.  Four group barriers: segment prefixes and
// normalisers together, the owning segment, the segment's weight prefixes,
// the owning element.
template <int ELT, bool VEC>
__device__ __forceinline__ void search_sequence(const VerifyArgs& a, int b, const SampleDesc& d, float u,
                                                FinalSmem& sm, int tid) {
    bool rej = d.k < a.gamma;
    const int ns = a.C * kCW;                             // segments in the row
    const int G = (ns + kCT - 1) / kCT;                   // consecutive segments per thread
    if (tid == 0) {
        sm.sel = sm.sel2 = 0x7fffffff;
        sm.last = sm.last2 = -1;
    }
    ThreadSums t = thread_sums(a, b, ns, G, rej, tid);
    FF Za, Zb, R{0.f, 0.f};
    GroupPrefix g = scan_phase(t, rej, sm, &Za, &Zb, tid);
    float dR = 0.f;
    if (rej) {
        R = ff_div(Za, Zb);
        dR = (R.hi - d.rt) + R.lo;                        // residual sums at R: w(rt) - (R - rt) dd
    }
    FF S = rej ? at_ratio(g.tot, g.dtot, dR) : g.tot;
    if (rej && !(S.hi > 0.f)) {
        // p_k equals q_k to rounding: the residual has no mass, draw from p_k
        rej = false;
        dR = 0.f;
        t.v = t.za;
        t.dv = 0.f;
        fin_sync();                                       // every thread has read the warp totals
        g = scan_phase(t, false, sm, &Za, &Zb, tid);
        S = g.tot;
    }
    if (!(S.hi > 0.f)) return;                            // unreachable for rows with a finite logit
    const FF excl = rej ? at_ratio(g.excl, g.dexcl, dR) : g.excl;
    const FF incl = rej ? at_ratio(g.incl, g.dincl, dR) : g.incl;
    FF target = ff_scale(u, S);
    if (!ff_lt(target, S))                                // u >= 1 clamps to the last token with mass
        target = ff_norm(FF{S.hi, S.lo - fabsf(S.hi) * 1.4210855e-14f});

    // The owning thread: the first whose interval [excl, incl) holds the
    // target (the intervals tile [0, S), so one does; the last thread with
    // mass stands in should that ever fail), then its owning segment.
    sm.xs[tid] = excl;
    const bool has = ff_lt(excl, incl);
    if (has && !ff_lt(target, excl) && ff_lt(target, incl)) atomicMin(&sm.sel, tid);
    if (has) atomicMax(&sm.last, tid);
    fin_sync();
    const int owner = sm.sel != 0x7fffffff ? sm.sel : sm.last;
    if (owner < 0) return;
    int sg;
    FF P;
    if (G == 1) {
        sg = owner;
        P = sm.xs[owner];
    } else {
        if (tid == owner) {
            FF run = excl;
            int pick = -1, last = -1;
            FF plo = excl, llo = excl;
            for (int gg = 0; gg < G; ++gg) {
                const int s = tid * G + gg;
                if (s >= ns) break;
                const SegSums q = seg_sums(a, (size_t)b * ns + s);
                const FF ts = rej ? at_ratio(q.w, q.dd, dR) : q.za;
                const FF nxt = ff_combine(run, ts);
                if (ts.hi > 0.f) {
                    last = s;
                    llo = run;
                    if (pick < 0 && ff_lt(target, nxt)) { pick = s; plo = run; }
                }
                run = nxt;
            }
            if (pick < 0) { pick = last; plo = llo; }
            sm.seg = pick;
            sm.P = plo;
        }
        fin_sync();
        sg = sm.seg;
        P = sm.P;
        if (sg < 0) return;
    }

    // Inside the segment: kSearchPT consecutive elements per thread.
    const FinalRows f = final_rows<ELT>(a, b, d);
    float w[kSearchPT];
    if (f.fast) search_weights<ELT, VEC, true>(a, f, sg, R, rej, w, tid);
    else search_weights<ELT, VEC, false>(a, f, sg, R, rej, w, tid);
    FF ts{0.f, 0.f};
#pragma unroll
    for (int e = 0; e < kSearchPT; ++e) ff_add(ts, w[e]);
    ts = ff_norm(ts);
    const int lane = tid & 31, warp = tid >> 5;
    const FF tin = warp_incl_scan_ff(ts);
    if (lane == 31) {
        sm.wv[warp] = tin;                                // the scan phase's reads ended at the barrier above
        sm.wd[warp] = 0.f;
    }
    fin_sync();
    const GroupPrefix h = group_prefix(tin, 0.f, sm.wv, sm.wd, tid);
    const FF lo = ff_combine(P, h.excl), hi = ff_combine(P, h.incl);
    const bool has2 = ts.hi > 0.f;
    if (has2 && !ff_lt(target, lo) && ff_lt(target, hi)) atomicMin(&sm.sel2, tid);
    if (has2) atomicMax(&sm.last2, tid);
    fin_sync();
    const int owner2 = sm.sel2 != 0x7fffffff ? sm.sel2 : sm.last2;
    if (tid == owner2) {
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

// Ticket of a finished chunk of sequence b: this call's count of the
// sequence's finished chunks before this one.  The counter holds
// (launch tag << kClaimIdxBits) | count; each CTA raises it to
// (tag << kClaimIdxBits) before its increment, which therefore sees this
// call's tag (launch tags increase from call to call) except after the
// process's tag count wrapped, when the first increment that finds an older
// tag installs this one by compare-and-swap.  No fence: the segment sums are
// tagged words that the search waits for.
__device__ unsigned take_ticket(const VerifyArgs& a, int b) {
    unsigned long long* t = a.tick + b;
    const unsigned long long tag = a.epoch << kClaimIdxBits;
    const unsigned long long tmask = ~((1ull << kClaimIdxBits) - 1ull);
    asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(t), "l"(tag) : "memory");
    unsigned long long v;
    asm volatile("atom.relaxed.gpu.global.add.u64 %0, [%1], 1;" : "=l"(v) : "l"(t) : "memory");
    for (uint32_t i = 0; (v & tmask) != tag; ++i) {
        if (i >= a.wait_limit) {
            atomicOr(a.err, SPEC_DEVERR_TIMEOUT);
            return 0u;
        }
        unsigned long long old;
        asm volatile("atom.relaxed.gpu.global.cas.b64 %0, [%1], %2, %3;"
                     : "=l"(old)
                     : "l"(t), "l"(v), "l"(tag | 1ull)
                     : "memory");
        if (old == v) return 0u;
        v = old;
        if ((v & tmask) == tag)
            asm volatile("atom.relaxed.gpu.global.add.u64 %0, [%1], 1;" : "=l"(v) : "l"(t) : "memory");
    }
    return (unsigned)(v & ~tmask);
}

}  // namespace sv
