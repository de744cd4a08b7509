// Device helpers shared by the verification kernels: streaming loads, the
// per-lane view of a warp chunk of logits, warp reductions and compensated
// summation.
#pragma once

#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "sv_internal.h"

namespace sv {

constexpr float kNegInf = -__builtin_huge_valf();

// 16-byte read-only streaming load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// 2^x on the special-function unit (flushes subnormal results to zero).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t u4_get(const uint4& v, int c) {
    return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

// Pairs of floats in one 64-bit register, for the packed f32x2 arithmetic of
// sm_100 and later (one instruction does two fp32 FMAs or adds).
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2_pack(float lo, float hi) {
    f32x2 p;
    asm("mov.b64 %0, {%1, %2};" : "=l"(p) : "f"(lo), "f"(hi));
    return p;
}
__device__ __forceinline__ void f2_unpack(f32x2 p, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p));
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 f2_sub(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// One logit as float.  ELT = 2: bfloat16 bits, ELT = 4: fp32.
template <int ELT>
__device__ __forceinline__ float load_logit(const char* row, int j) {
    if constexpr (ELT == 4) {
        return __ldg(reinterpret_cast<const float*>(row) + j);
    } else {
        unsigned short b = __ldg(reinterpret_cast<const unsigned short*>(row) + j);
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
}

// The part of a warp chunk one lane holds.  Vectorised layout: 8 vectors of
// 16 bytes at element offsets base + (lane + 32 t) * PV (PV = 16 / ELT),
// requiring 16-byte aligned rows.  Scalar layout (any alignment): elements
// base + lane + 32 i.  Either way val(i) walks the lane's elements in
// increasing index order and out-of-row elements read as -inf.
template <int ELT, bool VEC>
struct LaneChunk;

template <int ELT>
struct LaneChunk<ELT, true> {
    static constexpr int PV = 16 / ELT;
    static constexpr int EPL = kVecPerLane * PV;
    uint4 r[kVecPerLane];

    __device__ __forceinline__ void load(const char* row, int V, int base, int lane) {
        const uint32_t ninf = ELT == 4 ? 0xff800000u : 0xff80ff80u;
#pragma unroll
        for (int t = 0; t < kVecPerLane; ++t) {
            const int e = base + (lane + 32 * t) * PV;
            if (e < V) r[t] = ld_stream16(row + (size_t)e * ELT);
            else r[t] = make_uint4(ninf, ninf, ninf, ninf);
        }
    }
    __device__ __forceinline__ float val(int i) const {
        const int t = i / PV, e = i % PV;
        if constexpr (ELT == 4) {
            return __uint_as_float(u4_get(r[t], e));
        } else {
            const uint32_t w = u4_get(r[t], e >> 1);
            return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
        }
    }
    __device__ __forceinline__ int idx(int base, int lane, int i) const {
        return base + (lane + 32 * (i / PV)) * PV + (i % PV);
    }
};

template <int ELT>
struct LaneChunk<ELT, false> {
    static constexpr int EPL = kVecPerLane * (16 / ELT);
    float v[EPL];

    __device__ __forceinline__ void load(const char* row, int V, int base, int lane) {
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = base + lane + 32 * i;
            v[i] = e < V ? load_logit<ELT>(row, e) : kNegInf;
        }
    }
    __device__ __forceinline__ float val(int i) const { return v[i]; }
    __device__ __forceinline__ int idx(int base, int lane, int i) const {
        return base + lane + 32 * i;
    }
};

// ---- warp reductions -------------------------------------------------------
// Order-preserving integer key of a float: a larger float has a larger key
// (-0.0 falls just below +0.0), so that a warp maximum is one redux.sync.
__device__ __forceinline__ int ord_key(float v) {
    const int b = __float_as_int(v);
    return b >= 0 ? b : b ^ 0x7fffffff;
}
__device__ __forceinline__ float key_value(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff); }
constexpr int kNoKey = (int)0x80000000;                 // below every float's key

// The largest v of the warp (of -0.0 and +0.0, +0.0; NaN logits are undefined).
__device__ __forceinline__ float warp_max(float v) {
    return key_value(__reduce_max_sync(0xffffffffu, ord_key(v)));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// (value, index) order for argmax: larger value first, lower index on ties.
__device__ __forceinline__ bool am_better(float v1, int i1, float v2, int i2) {
    return v1 > v2 || (v1 == v2 && i1 < i2);
}

// The warp's best (v, i) in am_better's order, in every lane: the largest
// value (-0.0 and +0.0 equal), then the lowest index among the lanes holding
// it -- two redux.sync.  Indices are non-negative (INT_MAX for none).
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
    const int k = ord_key(v + 0.0f);
    const int t = __reduce_max_sync(0xffffffffu, k);
    i = (int)__reduce_min_sync(0xffffffffu, k == t ? (unsigned)i : 0xffffffffu);
    v = key_value(t);
}

// ---- float-float accumulation (Knuth's TwoSum) -----------------------------
struct FF {
    float hi, lo;
};

__device__ __forceinline__ void ff_add(FF& a, float x) {
    const float s = a.hi + x;
    const float bb = s - a.hi;
    const float err = (a.hi - (s - bb)) + (x - bb);
    a.hi = s;
    a.lo += err;
}

__device__ __forceinline__ double ff_value(const FF& a) { return (double)a.hi + (double)a.lo; }

// Sum of two float-float values (exact TwoSum of the leading parts, then the
// trailing parts), renormalised.  Symmetric in its operands.
__device__ __forceinline__ FF ff_combine(FF a, FF b) {
    const float s = a.hi + b.hi;
    const float bb = s - a.hi;
    float e = (a.hi - (s - bb)) + (b.hi - bb);
    e += a.lo + b.lo;
    const float hi = s + e;
    return FF{hi, e - (hi - s)};
}

__device__ __forceinline__ FF ff_shfl_xor(FF a, int o) {
    return FF{__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
}

__device__ __forceinline__ FF ff_shfl_up(FF a, int o) {
    return FF{__shfl_up_sync(0xffffffffu, a.hi, o), __shfl_up_sync(0xffffffffu, a.lo, o)};
}

// Canonical (non-overlapping) form of an accumulated float-float value.
__device__ __forceinline__ FF ff_norm(FF a) {
    const float s = a.hi + a.lo;
    return FF{s, a.lo - (s - a.hi)};
}

// a < b for canonical float-float values.
__device__ __forceinline__ bool ff_lt(FF a, FF b) {
    return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
}

// u * a for a float u and a canonical float-float a.
__device__ __forceinline__ FF ff_scale(float u, FF a) {
    const float p = u * a.hi;
    const float e = fmaf(u, a.hi, -p) + u * a.lo;
    return ff_norm(FF{p, e});
}

// a / b for canonical float-float values (one correction step).
__device__ __forceinline__ FF ff_div(FF a, FF b) {
    const float q = a.hi / b.hi;
    const float r = (fmaf(-q, b.hi, a.hi) + a.lo) - q * b.lo;
    return ff_norm(FF{q, r / b.hi});
}

// Warp sum of float-float values; every lane receives lane 0's result.
__device__ __forceinline__ FF warp_sum_ff(FF a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = ff_combine(a, ff_shfl_xor(a, o));
    return FF{__shfl_sync(0xffffffffu, a.hi, 0), __shfl_sync(0xffffffffu, a.lo, 0)};
}

// Inclusive warp scan of float-float values in lane order.
__device__ __forceinline__ FF warp_incl_scan_ff(FF a) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const FF y = ff_shfl_up(a, o);
        if (lane >= o) a = ff_combine(y, a);
    }
    return a;
}

// ---- tagged words --------------------------------------------------------------
// A value that a kernel may read while its writer (another kernel of the same
// call, running beside it) may not have written it yet travels as 64-bit
// words, each holding 32 bits of data in its low half and the call's tag in
// its high half.  Aligned 64-bit words are written and read whole, so a
// reader that sees its call's tag in a word has that word's data from its
// call -- no fence on either side; an older call's data carries another tag.
// Stored and loaded in pairs (16 bytes, each word whole).
__device__ __forceinline__ void st_tagged2(unsigned long long* p, uint32_t v0, uint32_t v1, uint32_t tag) {
    const unsigned long long t = (unsigned long long)tag << 32;
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(t | v0), "l"(t | v1) : "memory");
}

// Loads a pair; true when both words carry tag.
__device__ __forceinline__ bool ld_tagged2(const unsigned long long* p, uint32_t tag, uint32_t* v0,
                                           uint32_t* v1) {
    unsigned long long x, y;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(x), "=l"(y) : "l"(p) : "memory");
    *v0 = (uint32_t)x;
    *v1 = (uint32_t)y;
    return (uint32_t)(x >> 32) == tag && (uint32_t)(y >> 32) == tag;
}

// ---- programmatic dependent launch -------------------------------------------
// The kernels of the library are launched with programmatic stream
// serialisation (launch_pdl): a kernel may begin launching once every CTA of
// the kernel before it in the stream has triggered (or exited), and it waits (in hardware,
// griddepcontrol.wait) until that kernel has completed and its writes are
// visible before it touches global memory that the earlier kernel may write,
// or may still read.  A kernel may load the call's own inputs before waiting
// only when the kernel before it is the call's own first kernel, which waited
// for its predecessor before it triggered.  The streaming kernels trigger
// when each CTA is on its last chunk, the small kernels on entry.  Both
// instructions are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
static inline cudaError_t launch_pdl(void (*kfn)(KArgs...), dim3 grid, int threads, size_t smem,
                                     cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kfn, args...);
}

}  // namespace sv
