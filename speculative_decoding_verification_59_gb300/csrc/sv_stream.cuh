// Persistent streaming kernel over logit rows with a bulk-copy (TMA) ring.
//
// Used by the row-statistics pass of stochastic verification and by the
// argmax pass of greedy / tree verification, for rows whose byte length is a
// multiple of 16 (so every 32 KB block chunk of a row is a legal bulk copy).
//
// Each CTA has one producer warp and kWarps consumer warps.  Lane 0 of the
// producer walks the CTA's block chunks (row, segment) and issues one
// cp.async.bulk per chunk into a ring of kStages shared-memory stages, each
// guarded by a "full" mbarrier (copy landed) and an "empty" mbarrier (all
// consumer warps done).  Consumer warp w reduces the w-th 4 KB warp chunk of
// the stage -- (max m, sum 2^((z - m) s)) for row statistics, (value, lowest
// index) for argmax -- and writes one partial per warp chunk, at the same
// workspace position the register-path kernels use.
#pragma once

#include "sv_common.cuh"
#include "sv_tma.cuh"

namespace sv {

constexpr int kStages = 3;
constexpr int kRingThreads = (kWarps + 1) * 32;
constexpr int kStageBytes = kWarps * 32 * kLaneBytes;     // 32 KB block chunk

struct RingArgs {
    const char* zt;
    const char* zd;       // draft rows (row statistics of a sampling batch), else null
    int gamma;            // >= 0: rows are the 2*gamma+1 rows of each sampling sequence
    int rows_per_seq;
    int V;
    int nseg;
    long long total_chunks;
    float s;              // log2(e) / T (row statistics)
    float2* parts;
    int* err;
};

__device__ __forceinline__ const char* ring_row(const RingArgs& a, unsigned rr, size_t rowbytes) {
    if (a.gamma < 0) return a.zt + (size_t)rr * rowbytes;
    const unsigned b = rr / (unsigned)a.rows_per_seq;
    const int r = (int)(rr - b * (unsigned)a.rows_per_seq);
    return r <= a.gamma ? a.zt + ((size_t)b * (a.gamma + 1) + r) * rowbytes
                        : a.zd + ((size_t)b * a.gamma + (r - a.gamma - 1)) * rowbytes;
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

// Row statistics of one warp chunk held in shared memory: the chunk max m and
// sum_j 2^(z_j s - m s).  m s is rounded once for the whole chunk, a common
// factor the merge of partials absorbs within ~1e-6.
template <int ELT>
__device__ __forceinline__ float2 warp_rowstats(const unsigned char* chunk, int valid_bytes, float s) {
    uint4 v[kVecPerLane];
    lane_words<ELT>(chunk, valid_bytes, v);
    const float m = warp_max(lane_max<ELT>(v));
    float z = 0.f;
    if (m != kNegInf) {
        const float ms = m * s;
        if (fabsf(ms) < 1e30f) {
#pragma unroll
            for (int t = 0; t < kVecPerLane; ++t)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t w = u4_get(v[t], c);
                    if constexpr (ELT == 2) {
                        z += ex2_approx(fmaf(bf16_lo(w), s, -ms));
                        z += ex2_approx(fmaf(bf16_hi(w), s, -ms));
                    } else {
                        z += ex2_approx(fmaf(__uint_as_float(w), s, -ms));
                    }
                }
        } else {                                           // extreme temperature: no overflow
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
        z = warp_sum(z);
    }
    return make_float2(m, z);
}

// (value, lowest index) of one warp chunk held in shared memory; base is the
// row index of the chunk's first element.  The warp first agrees on the
// chunk maximum; only lanes holding it search for its first position.
template <int ELT>
__device__ __forceinline__ float2 warp_argmax_chunk(const unsigned char* chunk, int valid_bytes,
                                                    int base) {
    const int lane = threadIdx.x & 31;
    constexpr int PV = 16 / ELT;
    uint4 v[kVecPerLane];
    lane_words<ELT>(chunk, valid_bytes, v);
    const float lm = lane_max<ELT>(v);
    const float m = warp_max(lm);
    int bi = 0x7fffffff;
    if (lm == m) {                                         // float compare: -0.0 == +0.0
        for (int t = 0; t < kVecPerLane && bi == 0x7fffffff; ++t) {
            if ((lane + 32 * t) * 16 >= valid_bytes) break;
#pragma unroll
            for (int e = 0; e < PV; ++e) {
                float x;
                if constexpr (ELT == 4) {
                    x = __uint_as_float(u4_get(v[t], e));
                } else {
                    const uint32_t w = u4_get(v[t], e >> 1);
                    x = (e & 1) ? bf16_hi(w) : bf16_lo(w);
                }
                if (x == m && bi == 0x7fffffff) bi = base + (lane + 32 * t) * PV + e;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bi = min(bi, __shfl_xor_sync(0xffffffffu, bi, o));
    return make_float2(m + 0.0f, __int_as_float(bi));
}

template <int ELT, bool ARGMAX>
__global__ void __launch_bounds__(kRingThreads) ring_stream_kernel(const RingArgs a) {
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t rowbytes = (size_t)a.V * ELT;
    const int P = a.nseg * kWarps;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == 0) {
        // ---- producer: one lane issues the bulk copies
        if (lane == 0) {
            const unsigned total = (unsigned)a.total_chunks;
            unsigned issued = 0;
            bool ok = true;
            for (unsigned c = blockIdx.x; c < total; c += gridDim.x, ++issued) {
                const int st = (int)(issued % kStages);
                const unsigned use = issued / kStages;
                if (use > 0 && !wait_bounded(&empty[st], (use - 1) & 1u)) { ok = false; break; }
                const unsigned rr = c / (unsigned)a.nseg;
                const int seg = (int)(c - rr * (unsigned)a.nseg);
                const size_t off = (size_t)seg * kStageBytes;
                const uint32_t bytes = (uint32_t)min((size_t)kStageBytes, rowbytes - off);
                if (c + gridDim.x >= total) pdl_trigger();
                mbar_arrive_expect_tx(&full[st], bytes);
                bulk_g2s(ring + (size_t)st * kStageBytes, ring_row(a, rr, rowbytes) + off, bytes, &full[st]);
            }
            if (!ok) atomicOr(a.err, SPEC_DEVERR_TIMEOUT);
            // Do not leave while a copy may still be writing this CTA's shared memory.
            const unsigned first = issued > kStages ? issued - kStages : 0;
            for (unsigned i = first; i < issued; ++i)
                if (!wait_bounded(&full[i % kStages], (i / kStages) & 1u)) {
                    atomicOr(a.err, SPEC_DEVERR_TIMEOUT);
                    break;
                }
        }
        return;
    }

    // ---- consumers
    const int cw = warp - 1;
    const unsigned total = (unsigned)a.total_chunks;
    unsigned it = 0;
    for (unsigned c = blockIdx.x; c < total; c += gridDim.x, ++it) {
        const int st = (int)(it % kStages);
        if (!wait_bounded(&full[st], (it / kStages) & 1u)) {
            if (lane == 0) atomicOr(a.err, SPEC_DEVERR_TIMEOUT);
            return;
        }
        const unsigned rr = c / (unsigned)a.nseg;
        const int seg = (int)(c - rr * (unsigned)a.nseg);
        const size_t off = (size_t)seg * kStageBytes;
        const int bytes = (int)min((size_t)kStageBytes, rowbytes - off);
        const int wb = bytes - cw * (32 * kLaneBytes);            // valid bytes of this warp chunk
        const unsigned char* chunk = ring + (size_t)st * kStageBytes + cw * (32 * kLaneBytes);
        float2 part;
        if constexpr (ARGMAX) {
            part = wb > 0 ? warp_argmax_chunk<ELT>(chunk, wb, (int)(off / ELT) + cw * (32 * kLaneBytes / ELT))
                          : make_float2(kNegInf, __int_as_float(0x7fffffff));
        } else {
            part = wb > 0 ? warp_rowstats<ELT>(chunk, wb, a.s) : make_float2(kNegInf, 0.f);
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&empty[st]);
            a.parts[(size_t)rr * P + seg * kWarps + cw] = part;
        }
    }
}

// Launches the ring kernel (persistent grid); true when it applies (rows a
// multiple of 16 bytes), false when the caller must use the register path.
template <int ELT, bool ARGMAX>
cudaError_t launch_ring(const RingArgs& a, const DeviceInfo& di, cudaStream_t st, bool* used) {
    *used = false;
    if (((size_t)a.V * ELT) % 16 != 0) return cudaSuccess;
    if (a.total_chunks >= (1ll << 31)) return cudaSuccess;   // 32-bit chunk indices in the ring
    auto kfn = ring_stream_kernel<ELT, ARGMAX>;
    const int smem = kStages * kStageBytes;
    static int occ = 0;
    if (occ == 0) {
        cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kfn, kRingThreads, smem) != cudaSuccess || o < 1)
            o = 1;
        occ = o;
    }
    long long g = (long long)di.sm_count * occ;
    if (a.total_chunks < g) g = a.total_chunks;
    kfn<<<(int)g, kRingThreads, smem, st>>>(a);
    *used = true;
    return cudaGetLastError();
}

}  // namespace sv
