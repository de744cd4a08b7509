// The streaming pass over the logit rows of every verification mode: per-warp
// partials that the decision step (sv_decide.cuh) merges per sequence.
//
// ring_stream_kernel (rows whose byte length is a multiple of 16): a
// persistent CTA has one producer warp and kWarps consumer warps.  Lane 0 of
// the producer walks the CTA's block chunks (row, segment) and issues one
// cp.async.bulk per chunk into a ring of kStages shared-memory stages, each
// guarded by a "full" mbarrier (copy landed) and an "empty" mbarrier (all
// consumer warps done).  Consumer warp w reduces the w-th 4 KB warp chunk of
// the stage -- (max m, sum 2^((z - m) s)) for sampling, (value, lowest index)
// for greedy and tree verification -- and writes one partial per warp chunk.
//
// reg_stream_kernel (any row alignment): the same partials from register
// loads, one CTA of kThreads per block chunk in a persistent loop.
//
// Which chunks a ring CTA streams is ChunkSource's: three quarters dealt
// statically, the rest claimed one at a time from a tagged counter.  The
// bulk copies carry an evict-first L2 policy, and a CTA prefetches its first
// chunks into L2 before it waits on the kernel before.  No CTA waits on
// another; the decisions run in the kernels launched beside or after the
// stream.
#pragma once

#include "sv_common.cuh"
#include "sv_decide.cuh"
#include "sv_tma.cuh"

namespace sv {

constexpr int kStages = 3;
constexpr int kRingThreads = (kWarps + 1) * 32;
constexpr int kStageBytes = kWarps * 32 * kLaneBytes;     // 32 KB block chunk

// Row rr of a stream as the index of its partials' row (for sampling and
// lazy groups: sequence-major, 2 gamma + 1 rows per sequence), and that row's
// logits.  Only a lazy group maps: its row space is survivor i's target rows
// of the group's positions, then its draft rows.  The survivor lookup is
// cached, consecutive rows mostly belonging to one sequence.
struct StreamRows {
    unsigned seq_i = 0xffffffffu;
    int seq_b = 0;

    template <int MODE>
    __device__ __forceinline__ unsigned part_row(const VerifyArgs& a, unsigned rr) {
        if constexpr (MODE == kModeLazy) {
            const unsigned nr = (unsigned)(a.lz_nt + a.lz_nd);
            const unsigned i = rr / nr;
            const int q = (int)(rr - i * nr);
            if (i != seq_i) {
                seq_i = i;
                seq_b = a.lz_list ? __ldcg(a.lz_list + i) : (int)i;
            }
            const int r = q < a.lz_nt ? a.lz_lo + q : a.gamma + 1 + a.lz_lo + (q - a.lz_nt);
            return (unsigned)seq_b * (unsigned)a.rows_per_seq + (unsigned)r;
        } else {
            return rr;
        }
    }
};

template <int MODE>
__device__ __forceinline__ const char* stream_row(const VerifyArgs& a, unsigned rr, size_t rowbytes) {
    if constexpr (MODE == kModeSample || MODE == kModeLazy) {
        const unsigned b = rr / (unsigned)a.rows_per_seq;
        return sample_row(a, (int)b, (int)(rr - b * (unsigned)a.rows_per_seq), rowbytes);
    } else {
        return a.zt + (size_t)rr * rowbytes;
    }
}

// The lane's 128 bytes of a warp chunk in shared memory; bytes past
// valid_bytes read as -inf.
template <int ELT>
__device__ __forceinline__ void lane_words(const unsigned char* chunk, int valid_bytes, uint4 (&v)[kVecPerLane]) {
    const int lane = threadIdx.x & 31;
    const uint32_t ninf = ELT == 4 ? 0xff800000u : 0xff80ff80u;
#pragma unroll
    for (int t = 0; t < kVecPerLane; ++t) {
        const int off = (lane + 32 * t) * 16;
        v[t] = off < valid_bytes ? *reinterpret_cast<const uint4*>(chunk + off)
                                 : make_uint4(ninf, ninf, ninf, ninf);
    }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Largest logit the lane holds (packed bf16x2 maxima for bfloat16).
template <int ELT>
__device__ __forceinline__ float lane_max(const uint4 (&v)[kVecPerLane]) {
    if constexpr (ELT == 2) {
        uint32_t m2 = v[0].x;
#pragma unroll
        for (int t = 0; t < kVecPerLane; ++t)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t w = u4_get(v[t], c);
                asm("max.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(w));
            }
        return fmaxf(bf16_lo(m2), bf16_hi(m2));
    } else {
        float m = kNegInf;
#pragma unroll
        for (int t = 0; t < kVecPerLane; ++t)
#pragma unroll
            for (int c = 0; c < 4; ++c) m = fmaxf(m, __uint_as_float(u4_get(v[t], c)));
        return m;
    }
}

// Row statistics of one warp chunk: its max m and sum_j 2^((z_j - m) s).
// While |m s| < kFmaArgLimit each argument is one FMA, z_j s - fl(m s): the
// whole chunk then carries the common factor 2^(m s - fl(m s)), which the
// merge of partials (sv_decide.cuh) divides out exactly.  Beyond that limit
// (tiny temperatures) the arguments are (z_j - m) s.  The arguments and the
// running sums go through packed f32x2 FMAs and adds, two logits per
// instruction.
template <int ELT>
__device__ __forceinline__ float2 warp_rowstats(const uint4 (&v)[kVecPerLane], float s) {
    const float m = warp_max(lane_max<ELT>(v));
    if (m == kNegInf) return make_float2(m, 0.f);          // warp-uniform
    const float ms = m * s;
    float z;
    if (fabsf(ms) < kFmaArgLimit) {
        const f32x2 s2 = f2_pack(s, s), nms2 = f2_pack(-ms, -ms);
        f32x2 acc = f2_pack(0.f, 0.f);
#pragma unroll
        for (int t = 0; t < kVecPerLane; ++t)
#pragma unroll
            for (int c = 0; c < 4; c += (ELT == 2 ? 1 : 2)) {
                f32x2 x;
                if constexpr (ELT == 2) {
                    const uint32_t w = u4_get(v[t], c);
                    x = f2_pack(bf16_lo(w), bf16_hi(w));
                } else {
                    x = f2_pack(__uint_as_float(u4_get(v[t], c)), __uint_as_float(u4_get(v[t], c + 1)));
                }
                float a, b;
                f2_unpack(f2_fma(x, s2, nms2), a, b);
                acc = f2_add(acc, f2_pack(ex2_approx(a), ex2_approx(b)));
            }
        float a, b;
        f2_unpack(acc, a, b);
        z = a + b;
    } else {                                               // tiny temperature
        z = 0.f;
#pragma unroll
        for (int t = 0; t < kVecPerLane; ++t)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t w = u4_get(v[t], c);
                if constexpr (ELT == 2) {
                    z += ex2_approx((bf16_lo(w) - m) * s);
                    z += ex2_approx((bf16_hi(w) - m) * s);
                } else {
                    z += ex2_approx((__uint_as_float(w) - m) * s);
                }
            }
    }
    return make_float2(m, warp_sum(z));
}

// Largest logit of one 16-byte vector, as a packed bf16x2 pair (bfloat16) or
// a float (fp32).
template <int ELT>
__device__ __forceinline__ uint32_t vec_max_bits(const uint4& q) {
    if constexpr (ELT == 2) {
        uint32_t a = q.x, b = q.z;
        asm("max.bf16x2 %0, %0, %1;" : "+r"(a) : "r"(q.y));
        asm("max.bf16x2 %0, %0, %1;" : "+r"(b) : "r"(q.w));
        asm("max.bf16x2 %0, %0, %1;" : "+r"(a) : "r"(b));
        return a;
    } else {
        return __float_as_uint(fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)),
                                     fmaxf(__uint_as_float(q.z), __uint_as_float(q.w))));
    }
}

template <int ELT>
__device__ __forceinline__ float vec_max_value(uint32_t bits) {
    if constexpr (ELT == 2) return fmaxf(bf16_lo(bits), bf16_hi(bits));
    else return __uint_as_float(bits);
}

// Position (0..16/ELT-1) of the first element of a vector equal to m, or
// 16/ELT when there is none.  Float compares: -0.0 == +0.0.
template <int ELT>
__device__ __forceinline__ int vec_first_eq(const uint4& q, float m) {
    constexpr int PV = 16 / ELT;
    int e = PV;
#pragma unroll
    for (int i = PV - 1; i >= 0; --i) {
        float x;
        if constexpr (ELT == 4) {
            x = __uint_as_float(u4_get(q, i));
        } else {
            const uint32_t w = u4_get(q, i >> 1);
            x = (i & 1) ? bf16_hi(w) : bf16_lo(w);
        }
        if (x == m) e = i;
    }
    return e;
}

// (value, lowest index) of one warp chunk whose first element is row index
// base; padding past the row reads as -inf and follows every valid element
// in index order.  The lane's elements are in vectors t = 0..7 at positions
// base + (lane + 32 t) * PV, so index order is vector t first, then lane,
// then position in the vector: after the warp agrees on the maximum m, the
// first vector t holding m (one ballot per vector) and the lowest lane with it
// locate the first occurrence, and that lane's vector is searched alone.
template <int ELT>
__device__ __forceinline__ float2 warp_argmax_chunk(const uint4 (&v)[kVecPerLane], int base) {
    constexpr int PV = 16 / ELT;
    float vm[kVecPerLane];
    float lm = kNegInf;
#pragma unroll
    for (int t = 0; t < kVecPerLane; ++t) {
        vm[t] = vec_max_value<ELT>(vec_max_bits<ELT>(v[t]));
        lm = fmaxf(lm, vm[t]);
    }
    const float m = warp_max(lm);
    int bi = 0x7fffffff;
#pragma unroll
    for (int t = 0; t < kVecPerLane; ++t) {
        const unsigned hit = __ballot_sync(0xffffffffu, vm[t] == m);
        if (hit && bi == 0x7fffffff) {                       // warp-uniform
            const int src = __ffs(hit) - 1;
            const int e = __shfl_sync(0xffffffffu, vec_first_eq<ELT>(v[t], m), src);
            bi = base + (src + 32 * t) * PV + e;
        }
    }
    return make_float2(m + 0.0f, __int_as_float(bi));
}

// Bit e set for every element e of a bfloat16 vector that is >= the bf16 value
// in both halves of t2.  A packed compare gives 0xffff per element that
// reaches it; byte-permutes keep one byte per element (elements 0-3, then
// 4-7), each masked to its own bit, and a multiply by 0x01010101 adds the
// four bytes into the top byte (every bit distinct, so no carries).
__device__ __forceinline__ unsigned vec_ge_bits_bf16(const uint4& q, uint32_t t2) {
    uint32_t m0, m1, m2, m3;
    asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(m0) : "r"(q.x), "r"(t2));
    asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(m1) : "r"(q.y), "r"(t2));
    asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(q.z), "r"(t2));
    asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(m3) : "r"(q.w), "r"(t2));
    const uint32_t x = __byte_perm(m0, m1, 0x6420);
    const uint32_t y = __byte_perm(m2, m3, 0x6420);
    return ((x & 0x08040201u) | (y & 0x80402010u)) * 0x01010101u >> 24;
}

// ---- top-K lists (branch tokens of a draft tree) -----------------------------
// The K best (value, index) pairs seen by a lane, best first: larger value
// first, lower index first among equal values (am_better).  Empty slots hold
// (-inf, INT_MAX), which every real element beats.
template <int K>
struct TopList {
    float v[K];
    int i[K];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int k = 0; k < K; ++k) { v[k] = kNegInf; i[k] = 0x7fffffff; }
    }
    __device__ __forceinline__ void insert(float x, int j) {
        if (!am_better(x, j, v[K - 1], i[K - 1])) return;
        v[K - 1] = x;
        i[K - 1] = j;
#pragma unroll
        for (int k = K - 1; k > 0; --k)
            if (am_better(v[k], i[k], v[k - 1], i[k - 1])) {
                const float tv = v[k]; v[k] = v[k - 1]; v[k - 1] = tv;
                const int ti = i[k]; i[k] = i[k - 1]; i[k - 1] = ti;
            }
    }
};

// The warp's K best entries over all lanes' lists, best first, in every
// lane: K rounds of a warp argmax over the list heads, the winning lane
// popping its head (indices are distinct across lanes).
template <int K>
__device__ __forceinline__ void warp_merge_topk(TopList<K>& L, float (&ov)[K], int (&oi)[K]) {
#pragma unroll
    for (int r = 0; r < K; ++r) {
        float hv = L.v[0];
        int hi = L.i[0];
        warp_argmax(hv, hi);
        ov[r] = hv;
        oi[r] = hi;
        if (L.i[0] == hi && hi != 0x7fffffff) {
#pragma unroll
            for (int k = 0; k < K - 1; ++k) { L.v[k] = L.v[k + 1]; L.i[k] = L.i[k + 1]; }
            L.v[K - 1] = kNegInf;
            L.i[K - 1] = 0x7fffffff;
        }
    }
}

// Entries a warp chunk leaves for a top-K merge: up to 2K candidates in any
// order, the rest (-inf, INT_MAX).
__host__ __device__ constexpr int topk_slots(int K) { return 2 * K; }

// Top-K candidates of one warp chunk whose first element is row index base,
// of which valid_bytes lie inside the row; v holds the lane's vectors, chunk
// the same bytes in shared memory.  The chunk must yield every element of
// the row's top K that it holds; those are all at least any lower bound of
// the row's K-th largest element.  thr is such a bound: on the warp's first
// chunk of a row (have_thr false) the K-th largest of the 32 lane maxima
// (K distinct elements of the row), afterwards the bound carried from the
// warp's earlier chunks of the same row, which skips the K warp-max rounds.
// Each lane marks its elements >= thr in a 64-bit mask (bit 8 t + e for
// element e of vector t): for bfloat16 with packed compares of every element,
// no branch.  When the warp marks at most 2K elements (nearly always: a few
// more than K) they are written as they are, unsorted, into the chunk's 2K
// slots -- the merge orders them.  Otherwise the lanes insert their marked
// elements into sorted lists and the warp merges the lists into the chunk's
// exact top K, whose K-th value then raises thr.  Marked elements are read
// back from shared memory in one loop, which keeps the kernel's instruction
// footprint small.
template <int ELT, int K>
__device__ __forceinline__ void warp_topk_chunk(const uint4 (&v)[kVecPerLane],
                                                const unsigned char* chunk, int valid_bytes,
                                                int base, float2* out, float& thr, bool have_thr) {
    const int lane = threadIdx.x & 31;
    constexpr int PV = 16 / ELT;
    constexpr int KS = topk_slots(K);
    if (!have_thr) {                                       // warp-uniform
        float x = lane_max<ELT>(v);
        thr = kNegInf;
#pragma unroll
        for (int r = 0; r < K; ++r) {
            thr = warp_max(x);
            const unsigned own = __ballot_sync(0xffffffffu, x == thr);
            if (lane == __ffs(own) - 1) x = kNegInf;
        }
    }
    unsigned long long mask = 0ull;
    if constexpr (ELT == 2) {
        // thr is a logit of the row (or -inf), so exact in bfloat16
        const uint32_t tb = __float_as_uint(thr) >> 16;
        const uint32_t t2 = tb | (tb << 16);
        uint32_t lo = 0u, hi = 0u;
#pragma unroll
        for (int t = 0; t < kVecPerLane; ++t) {
            const uint32_t b = vec_ge_bits_bf16(v[t], t2);
            if (t < 4) lo |= b << (8 * t);
            else hi |= b << (8 * (t - 4));
        }
        mask = (unsigned long long)hi << 32 | lo;
    } else {
#pragma unroll
        for (int t = 0; t < kVecPerLane; ++t) {
            if (vec_max_value<ELT>(vec_max_bits<ELT>(v[t])) >= thr) {
                unsigned bits = 0u;
#pragma unroll
                for (int e = 0; e < PV; ++e)
                    bits |= (__uint_as_float(u4_get(v[t], e)) >= thr ? 1u : 0u) << e;
                mask |= (unsigned long long)bits << (8 * t);
            }
        }
    }
    if (valid_bytes < 32 * kLaneBytes) {                   // warp-uniform
        // vectors past the row's end read as -inf in v but hold stale bytes
        // in shared memory; they reach thr = -inf, so unmark them
#pragma unroll
        for (int t = 0; t < kVecPerLane; ++t)
            if ((lane + 32 * t) * 16 >= valid_bytes) mask &= ~(0xffull << (8 * t));
    }
    auto element = [&](int bit, float* y, int* j) {
        const int t = bit >> 3, e = bit & 7;
        const int off = (lane + 32 * t) * 16 + e * ELT;
        if constexpr (ELT == 4) *y = *reinterpret_cast<const float*>(chunk + off);
        else *y = __uint_as_float((uint32_t)*reinterpret_cast<const unsigned short*>(chunk + off) << 16);
        *y += 0.0f;                                        // -0.0 counts as +0.0
        *j = base + (lane + 32 * t) * PV + e;
    };
    // inclusive prefix of the lanes' counts: a popcount of a ballot when no
    // lane marks more than one element (the common case), else a warp scan
    const int n = __popcll(mask);
    const unsigned has = __ballot_sync(0xffffffffu, n > 0);
    int incl, total;
    if (__ballot_sync(0xffffffffu, n > 1) == 0u) {        // warp-uniform
        incl = __popc(has & ((2u << lane) - 1u));
        total = __popc(has);
    } else {
        incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        total = __shfl_sync(0xffffffffu, incl, 31);
    }
    if (total <= KS) {                                     // warp-uniform
        int slot = incl - n;
#pragma unroll 1
        while (mask) {
            const int bit = __ffsll((long long)mask) - 1;
            mask &= mask - 1ull;
            float y;
            int j;
            element(bit, &y, &j);
            out[slot++] = make_float2(y, __int_as_float(j));
        }
        if (lane >= total && lane < KS) out[lane] = make_float2(kNegInf, __int_as_float(0x7fffffff));
        return;
    }
    TopList<K> L;
    L.init();
#pragma unroll 1
    while (mask) {
        const int bit = __ffsll((long long)mask) - 1;
        mask &= mask - 1ull;
        float y;
        int j;
        element(bit, &y, &j);
        L.insert(y, j);
    }
    float ov[K];
    int oi[K];
    warp_merge_topk<K>(L, ov, oi);
    if (lane == 0)
#pragma unroll
        for (int r = 0; r < K; ++r) out[r] = make_float2(ov[r], __int_as_float(oi[r]));
    if (lane >= K && lane < KS) out[lane] = make_float2(kNegInf, __int_as_float(0x7fffffff));
    thr = fmaxf(thr, ov[K - 1]);                          // more than 2K marked: K of them reach it
}

// A partial of a sampling, greedy or tree stream -- (m, s), or (value,
// index) -- stored as a pair of tagged words (sv_common.cuh), so that the
// decide kernel, running beside the stream, can tell a partial of this call
// from an older one without any fence.
__device__ __forceinline__ void store_tagged_part(const VerifyArgs& a, size_t i, float2 v) {
    st_tagged2(reinterpret_cast<unsigned long long*>(a.parts) + 2 * i, __float_as_uint(v.x),
               __float_as_uint(v.y), a.ptag);
}

// Stage marker of the end of a CTA's chunks.
constexpr unsigned kNoChunk = 0xffffffffu;

// The block chunks that one CTA of a ring stream takes, in order.  Three
// quarters of a stream's chunks are dealt out statically, a contiguous range
// per CTA; the rest are claimed one at a time from the workspace's counter,
// so CTAs that stream faster (the rate differs by SM and by die) take more
// of them and the stream ends together instead of with its slowest CTA.
// Each claim is issued one chunk ahead of its use, so its round trip
// overlaps the copies in flight.
//
// The counter holds (launch tag << kClaimIdxBits) | next index.  Every CTA
// first raises it to (tag << kClaimIdxBits) | (first dynamic index) with an
// atomic max: tags increase from launch to launch, so the first such max of
// a launch restarts the count and the others change nothing, and a CTA's own
// max precedes its claims, which therefore always see this launch's tag --
// except after the process's tag count wrapped (once in 2^40 launches), when
// the first claim that finds an older tag installs this one by compare-and-swap.
struct ChunkSource {
    unsigned s, s_end, step, total, first_dyn;
    bool dyn, have;
    unsigned long long* ctr;
    unsigned long long tag, pending;
    uint32_t limit;
    int* err;

    // round_robin: the static share is dealt chunk by chunk (CTA i takes
    // chunks i, i + G, i + 2G, ... of G CTAs), so the stream advances through
    // the chunks -- and the sequences -- in index order; otherwise each CTA
    // takes a contiguous range.
    // This CTA's static share: chunks s, s + step, ... below s_end; dyn when
    // the rest, from first_dyn on, is claimed from the counter.
    __device__ __forceinline__ static void static_share(unsigned total, bool round_robin, unsigned* s,
                                                        unsigned* s_end, unsigned* step, bool* dyn,
                                                        unsigned* first_dyn) {
        const unsigned q = (3u * (total >> 2) + ((3u * (total & 3u)) >> 2)) / gridDim.x;   // floor(3 total / 4) / G
        *step = 1;
        *dyn = q >= 2 && total < (1u << (kClaimIdxBits - 1));
        if (*dyn) {
            *first_dyn = q * gridDim.x;
            if (round_robin) {
                *s = blockIdx.x;
                *step = gridDim.x;
                *s_end = blockIdx.x + q * gridDim.x;
            } else {
                *s = blockIdx.x * q;
                *s_end = *s + q;
            }
        } else {
            *first_dyn = total;
            cta_range(total, blockIdx.x, gridDim.x, s, s_end);
        }
    }

    __device__ __forceinline__ ChunkSource(const VerifyArgs& a, unsigned total_, bool round_robin) {
        total = total_;
        ctr = a.claim;
        tag = a.claim_tag;
        limit = a.wait_limit;
        err = a.err;
        have = false;
        pending = 0ull;
        static_share(total, round_robin, &s, &s_end, &step, &dyn, &first_dyn);
        if (dyn)
            asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(ctr), "l"(tag | first_dyn)
                         : "memory");
    }

    __device__ __forceinline__ void claim() {
        asm volatile("atom.relaxed.gpu.global.add.u64 %0, [%1], 1;" : "=l"(pending) : "l"(ctr) : "memory");
        have = true;
    }

    // A claim that found another launch's tag: install this launch's with
    // compare-and-swap (taking the first dynamic index), or, if another CTA
    // already did, claim again.
    __device__ unsigned long long reclaim(unsigned long long v) {
        const unsigned long long tmask = ~((1ull << kClaimIdxBits) - 1ull);
        for (uint32_t i = 0; i < limit; ++i) {
            if ((v & tmask) == tag) {
                asm volatile("atom.relaxed.gpu.global.add.u64 %0, [%1], 1;" : "=l"(v) : "l"(ctr) : "memory");
                if ((v & tmask) == tag) return v;
                continue;
            }
            unsigned long long old;
            asm volatile("atom.relaxed.gpu.global.cas.b64 %0, [%1], %2, %3;"
                         : "=l"(old)
                         : "l"(ctr), "l"(v), "l"(tag | (first_dyn + 1ull))
                         : "memory");
            if (old == v) return tag | first_dyn;
            v = old;
        }
        atomicOr(err, SPEC_DEVERR_TIMEOUT);
        return tag | total;                               // gives up: no further chunks
    }

    // The next chunk index, kNoChunk at the end.
    __device__ __forceinline__ unsigned next() {
        if (s < s_end) {
            const unsigned c = s;
            s += step;
            if (s >= s_end && dyn) claim();
            return c;
        }
        if (!have) return kNoChunk;
        have = false;
        unsigned long long v = pending;
        if ((v & ~((1ull << kClaimIdxBits) - 1ull)) != tag) v = reclaim(v);
        const unsigned c = (unsigned)(v & ((1ull << kClaimIdxBits) - 1ull));
        if (c >= total) return kNoChunk;
        claim();
        return c;
    }
};

// Chunks of its static share that a ring CTA prefetches into L2 before it
// waits for the kernel before it, on streams of at least kPrefetchMinChunks
// chunks (32 MB).  Measured on GB300: shorter streams (chain-b8's 640-chunk
// argmax streams, chain-small's 9 chunks) lost 0.3-0.5 us a call to the
// prefetch, longer ones gained 1.3-3.3 us.
constexpr int kPrefetchChunks = 3;
constexpr long long kPrefetchMinChunks = 1024;

// The L2 prefetch of this CTA's first static chunks, issued before the wait
// on the kernel before (one thread): the HBM latency of the stream's first
// copies then overlaps that kernel's tail.  Only the logits are touched, never
// the workspace the kernel before may still use; a kernel before that writes
// the logits writes them through L2, where the copies issued after the wait
// find them current.  Lazy groups after the first take their rows and chunk
// count from the workspace and prefetch nothing.
template <int MODE>
__device__ __forceinline__ void prefetch_first_chunks(const VerifyArgs& a, size_t rowbytes, bool round_robin) {
    if (a.total_chunks < kPrefetchMinChunks) return;
    if constexpr (MODE == kModeLazy)
        if (a.lz_list != nullptr || a.lz_count != nullptr) return;
    unsigned s, s_end, step, first_dyn;
    bool dyn;
    ChunkSource::static_share((unsigned)a.total_chunks, round_robin, &s, &s_end, &step, &dyn, &first_dyn);
    StreamRows rows;
    for (int i = 0; i < kPrefetchChunks && s < s_end; ++i, s += step) {
        const unsigned rr = s / (unsigned)a.nseg;
        const int seg = (int)(s - rr * (unsigned)a.nseg);
        const size_t off = (size_t)seg * kStageBytes;
        bulk_prefetch_l2(stream_row<MODE>(a, rows.part_row<MODE>(a, rr), rowbytes) + off,
                         (uint32_t)min((size_t)kStageBytes, rowbytes - off));
    }
}

template <int ELT, int MODE>
__device__ __forceinline__ void ring_stream_body(const VerifyArgs& a) {
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
    __shared__ uint4 stage_info[kStages];              // (row, partial row, segment, length) a stage holds
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int KT = topk_of(MODE);
    const size_t rowbytes = (size_t)a.V * ELT;
    const int P = a.nseg * kWarps;

    constexpr bool kBeside = MODE == kModeSample || MODE == kModeGreedy || MODE == kModeTree;
    if (threadIdx.x == 0) {
        prefetch_first_chunks<MODE>(a, rowbytes, kBeside);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        mbar_init_fence();
    }
    __syncthreads();
    pdl_wait();                 // the kernel before may still read this workspace or write the rows
    // Sampling, greedy and tree verification: the decide kernel may start
    // now.  It runs beside the stream and takes each sequence's decision once
    // that sequence's partials all carry this call's tag.
    if (kBeside && threadIdx.x == 0) pdl_trigger();
    unsigned total = (unsigned)a.total_chunks;
    if constexpr (MODE == kModeLazy) {
        if (a.lz_count) total = (unsigned)__ldcg(a.lz_count) * (unsigned)(a.lz_nt + a.lz_nd) * (unsigned)a.nseg;
        if (blockIdx.x == 0 && (int)threadIdx.x < a.lz_nzero) a.lz_zero[threadIdx.x] = 0;
    }
    StreamRows rows;

    if (warp == 0) {
        // ---- producer: one lane issues the bulk copies and hands each
        // stage's row, partial row, segment and length to the consumers (row
        // kNoChunk ends the stream), so that they divide no chunk index
        if (lane == 0) {
            // The stream reads each logit once: its lines go first when L2
            // needs room, which keeps the partials, decisions and candidates
            // that the kernels beside and after it poll and read (same-box,
            // chain-b64: sampling 61.5 -> 60.4 us, greedy 26.6 -> 26.3, top-K
            // 30.9 -> 30.0 per call).
            const uint64_t evict_first = l2_evict_first_policy();
            ChunkSource src(a, total, kBeside);
            unsigned issued = 0;
            bool ok = true, ended = false, triggered = kBeside;
            for (;; ++issued) {
                const int st = (int)(issued % kStages);
                const unsigned use = issued / kStages;
                if (use > 0 && !wait_bounded(&empty[st], (use - 1) & 1u, a.wait_limit)) { ok = false; break; }
                const unsigned c = src.next();
                if (c == kNoChunk) {
                    if (!triggered) pdl_trigger();
                    stage_info[st] = make_uint4(kNoChunk, 0u, 0u, 0u);
                    mbar_arrive(&full[st]);                   // releases the consumers' last wait
                    ended = true;
                    break;
                }
                const unsigned rr = c / (unsigned)a.nseg;
                const int seg = (int)(c - rr * (unsigned)a.nseg);
                const size_t off = (size_t)seg * kStageBytes;
                const uint32_t bytes = (uint32_t)min((size_t)kStageBytes, rowbytes - off);
                const unsigned pr = rows.part_row<MODE>(a, rr);
                if (!triggered && src.s >= src.s_end) {
                    // static share issued: the next kernel may start launching
                    pdl_trigger();
                    triggered = true;
                }
                stage_info[st] = make_uint4(rr, pr, (unsigned)seg, bytes);
                mbar_arrive_expect_tx(&full[st], bytes);
                bulk_g2s(ring + (size_t)st * kStageBytes, stream_row<MODE>(a, pr, rowbytes) + off, bytes,
                         &full[st], evict_first);
            }
            if (!ok) {
                if (!triggered) pdl_trigger();
                atomicOr(a.err, SPEC_DEVERR_TIMEOUT);
            }
            // Do not leave while a copy may still be writing this CTA's shared
            // memory.  The end marker reused the stage of copy issued - kStages
            // after its consumers had released it (that copy is complete, and
            // its barrier has moved two phases on), so the check starts after it.
            unsigned first = issued > kStages ? issued - kStages : 0;
            if (ended && issued >= kStages) first = issued - kStages + 1;
            for (unsigned i = first; i < issued; ++i)
                if (!wait_bounded(&full[i % kStages], (i / kStages) & 1u)) {
                    atomicOr(a.err, SPEC_DEVERR_TIMEOUT);
                    break;
                }
        }
        return;
    }

    // ---- consumers.  A timed-out wait flags the error and stops the warp
    // from touching the ring.
    const int cw = warp - 1;
    unsigned tk_row = 0xffffffffu;                        // top-K: row of the carried bound
    float tk_thr = kNegInf;
    bool ok = true;
    for (unsigned it = 0;; ++it) {
        const int st = (int)(it % kStages);
        if (!wait_bounded(&full[st], (it / kStages) & 1u, a.wait_limit)) ok = false;
        if (!__all_sync(0xffffffffu, ok)) break;
        // the producer's division of the chunk index and row mapping; the
        // length is recomputed here (reading it from the stage as well
        // measured 2% slower fp32 sampling calls, chain-b256)
        const uint4 si = stage_info[st];
        const unsigned rr = si.x;
        if (rr == kNoChunk) break;
        const unsigned pr = si.y;
        const int seg = (int)si.z;
        const size_t off = (size_t)seg * kStageBytes;
        const int bytes = (int)min((size_t)kStageBytes, rowbytes - off);
        const int wb = bytes - cw * (32 * kLaneBytes);            // valid bytes of this warp chunk
        const bool use = wb > 0;
        float2 part = make_float2(0.f, 0.f);
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
            const int base = (int)(off / ELT) + cw * (32 * kLaneBytes / ELT);
            if constexpr (MODE == kModeSample || MODE == kModeLazy) part = warp_rowstats<ELT>(v, a.s);
            else if constexpr (KT > 0) {
                warp_topk_chunk<ELT, KT>(v, chunk, wb, base,
                                         a.parts + ((size_t)rr * P + seg * kWarps + cw) * topk_slots(KT),
                                         tk_thr, tk_row == rr);
                tk_row = rr;
            }
            else part = warp_argmax_chunk<ELT>(v, base);
        } else {
            part = (MODE == kModeSample || MODE == kModeLazy) ? make_float2(kNegInf, 0.f)
                                                              : make_float2(kNegInf, __int_as_float(0x7fffffff));
            if constexpr (KT > 0)
                if (lane < topk_slots(KT))
                    a.parts[((size_t)rr * P + seg * kWarps + cw) * topk_slots(KT) + lane] = part;
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&empty[st]);
            if constexpr (kBeside) store_tagged_part(a, (size_t)pr * P + seg * kWarps + cw, part);
            else if constexpr (KT == 0) a.parts[(size_t)pr * P + seg * kWarps + cw] = part;
        }
    }
    if (!ok && lane == 0) atomicOr(a.err, SPEC_DEVERR_TIMEOUT);
}

template <int ELT, int MODE>
__global__ void __launch_bounds__(kRingThreads, 2) ring_stream_kernel(const VerifyArgs a) {
    ring_stream_body<ELT, MODE>(a);
}

// The sampling stream, held to 64 registers a thread: two of its CTAs, a
// decide CTA and a final-pass CTA then fit on one SM's registers together,
// as they run in a whole sampling call.
template <int ELT>
__global__ void __maxnreg__(64) ring_sample_kernel(const VerifyArgs a) {
    ring_stream_body<ELT, kModeSample>(a);
}

template <int ELT, bool VEC, int MODE>
__global__ void __launch_bounds__(kThreads) reg_stream_kernel(const VerifyArgs a) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int WE = 32 * kLaneBytes / ELT;                  // elements per warp chunk
    const int P = a.nseg * kWarps;
    const size_t rowbytes = (size_t)a.V * ELT;
    const unsigned total = (unsigned)a.total_chunks;

    unsigned c0, c1;
    cta_range(total, blockIdx.x, gridDim.x, &c0, &c1);
    pdl_wait();                 // the kernel before may still read this workspace or write the rows
    for (unsigned c = c0; c < c1; ++c) {
        if (c + 1 == c1) pdl_trigger();
        const unsigned rr = c / (unsigned)a.nseg;
        const int seg = (int)(c - rr * (unsigned)a.nseg);
        const char* row = stream_row<MODE>(a, rr, rowbytes);
        const int base = (seg * kWarps + warp) * WE;
        float2 part = make_float2(0.f, 0.f);
        if constexpr (topk_of(MODE) > 0) {
            // as warp_topk_chunk: threshold from the K-th largest lane
            // maximum, a mask of the lane's elements that reach it, one
            // insertion loop (the marked logits are re-read from the row)
            constexpr int KT = topk_of(MODE);
            static_assert(LaneChunk<ELT, VEC>::EPL <= 64, "one mask bit per lane element");
            unsigned long long mask = 0ull;
            if (base < a.V) {                                  // warp-uniform
                LaneChunk<ELT, VEC> ch;
                ch.load(row, a.V, base, lane);
                float x = kNegInf;
#pragma unroll
                for (int i = 0; i < LaneChunk<ELT, VEC>::EPL; ++i) x = fmaxf(x, ch.val(i));
                float thr = kNegInf;
#pragma unroll
                for (int r = 0; r < KT; ++r) {
                    thr = warp_max(x);
                    const unsigned own = __ballot_sync(0xffffffffu, x == thr);
                    if (lane == __ffs(own) - 1) x = kNegInf;
                }
#pragma unroll
                for (int i = 0; i < LaneChunk<ELT, VEC>::EPL; ++i)
                    if (ch.idx(base, lane, i) < a.V && ch.val(i) >= thr) mask |= 1ull << i;
            }
            TopList<KT> L;
            L.init();
#pragma unroll 1
            while (mask) {
                const int i = __ffsll((long long)mask) - 1;
                mask &= mask - 1ull;
                const int j = base + lane + 32 * i;
                L.insert(load_logit<ELT>(row, j) + 0.0f, j);
            }
            float ov[KT];
            int oi[KT];
            warp_merge_topk<KT>(L, ov, oi);
            float2* out = a.parts + ((size_t)rr * P + seg * kWarps + warp) * topk_slots(KT);
            if (lane == 0)
#pragma unroll
                for (int r = 0; r < KT; ++r) out[r] = make_float2(ov[r], __int_as_float(oi[r]));
            if (lane >= KT && lane < topk_slots(KT))
                out[lane] = make_float2(kNegInf, __int_as_float(0x7fffffff));
            continue;
        } else if constexpr (MODE == kModeSample) {
            float m = kNegInf, z = 0.f;
            if (base < a.V) {
                LaneChunk<ELT, VEC> ch;
                ch.load(row, a.V, base, lane);
#pragma unroll
                for (int i = 0; i < LaneChunk<ELT, VEC>::EPL; ++i) m = fmaxf(m, ch.val(i));
                m = warp_max(m);
                if (m != kNegInf) {
                    // the same arguments as warp_rowstats
                    const float ms = m * a.s;
                    const bool fmapath = fabsf(ms) < kFmaArgLimit;
#pragma unroll
                    for (int i = 0; i < LaneChunk<ELT, VEC>::EPL; ++i) {
                        const float x = ch.val(i);
                        z += ex2_approx(fmapath ? fmaf(x, a.s, -ms) : (x - m) * a.s);
                    }
                    z = warp_sum(z);
                }
            }
            part = make_float2(m, z);
        } else {
            float bv = kNegInf;
            int bi = 0x7fffffff;
            if (base < a.V) {
                LaneChunk<ELT, VEC> ch;
                ch.load(row, a.V, base, lane);
                // lane elements come in increasing index order: strict '>'
                // keeps the first maximum; +0.0f folds -0.0 into +0.0
                bv = ch.val(0) + 0.0f;
                bi = ch.idx(base, lane, 0);
#pragma unroll
                for (int i = 1; i < LaneChunk<ELT, VEC>::EPL; ++i) {
                    const float v = ch.val(i) + 0.0f;
                    if (v > bv) { bv = v; bi = ch.idx(base, lane, i); }
                }
                if (bi >= a.V) bi = 0x7fffffff;            // only padding seen
                warp_argmax(bv, bi);
            }
            part = make_float2(bv, __int_as_float(bi));
        }
        if (lane == 0) {
            if constexpr (MODE == kModeSample || MODE == kModeGreedy || MODE == kModeTree)
                store_tagged_part(a, (size_t)rr * P + seg * kWarps + warp, part);
            else a.parts[(size_t)rr * P + seg * kWarps + warp] = part;
        }
    }
}

// Launches the streaming pass of MODE over the rows of a (persistent grid):
// the bulk-copy ring for 16-byte rows, the register path otherwise.
template <int ELT, int MODE>
cudaError_t launch_stream(const VerifyArgs& args, const DeviceInfo& di, cudaStream_t st) {
    VerifyArgs a = args;
    a.claim = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(a.err) + kClaimOff);
    a.claim_tag = next_launch_tag() << kClaimIdxBits;
    if (((size_t)a.V * ELT) % 16 == 0) {
        auto kfn = MODE == kModeSample ? ring_sample_kernel<ELT> : ring_stream_kernel<ELT, MODE>;
        const int smem = kStages * kStageBytes;
        // once per device: the shared-memory opt-in, then the occupancy it allows
        static DeviceSlots slots = {};
        int occ = 0;
        cudaError_t e = device_once(slots, &occ, [&](int, int* o) {
            cudaError_t r = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (r != cudaSuccess) return r;
            // the whole carveout as shared memory, as the kernels that run
            // beside this one prefer it too, so an SM can hold both
            r = cudaFuncSetAttribute(kfn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
            if (r != cudaSuccess) return r;
            return cudaOccupancyMaxActiveBlocksPerMultiprocessor(o, kfn, kRingThreads, smem);
        });
        if (e != cudaSuccess) return e;
        long long g = (long long)di.sm_count * occ;
        if (a.total_chunks < g) g = a.total_chunks;
        return launch_pdl(kfn, dim3((unsigned)g), kRingThreads, smem, st, a);
    }
    if constexpr (MODE == kModeLazy) {
        return cudaErrorInvalidValue;      // lazy groups stream 16-byte rows only
    } else {
        auto kfn = reg_stream_kernel<ELT, false, MODE>;
        static DeviceSlots slots = {};
        int occ = 0;
        cudaError_t e = device_once(slots, &occ, [&](int, int* o) {
            return cudaOccupancyMaxActiveBlocksPerMultiprocessor(o, kfn, kThreads, 0);
        });
        if (e != cudaSuccess) return e;
        long long g = (long long)di.sm_count * occ;
        if (a.total_chunks < g) g = a.total_chunks;
        return launch_pdl(kfn, dim3((unsigned)g), kThreads, 0, st, a);
    }
}

}  // namespace sv
