// Semantic fallback of the reuse-position search: the window rows whose
// hidden states are most similar (cosine) to the current one.
//
// Source: "AdaPLD: adaptive retrieval and reuse for efficient model-free
// speculative decoding", section 3.2 (semantic fallback stage: when the
// lexical stage finds nothing, score(j) = h_current . h_j / (|h_current|
// |h_j|) over the hidden states of a sliding window of the most recent 30
// forward steps, and the most similar positions are retrieved) and
// Algorithm 1 (SemanticFallback: top-delta positions).
//
// Each window row is read once: one warp per row accumulates h.q, h.h and
// q.q in fp32 with packed f32x2 FMAs over 16-byte vectors, a batch of
// kCosBatch vectors per lane loaded at once (the query vectors come through
// L1, shared by the CTA's warps).  A row with a zero norm, or
// a zero query, scores 0.  One warp per sequence then keeps the delta best
// scores (larger first, lower window index first among equal scores) and
// maps them to context positions.  The pass is a batched matrix-vector
// product, bound by HBM; it has no dense contraction for tensor cores.
#include "sv_stream.cuh"

namespace sv {

constexpr int kCosThreads = 256;
constexpr int kCosRowsPerCta = kCosThreads / 32; // one row per warp
constexpr int kCosBatch = 4;                     // 16-byte vectors per lane per batch

struct CosArgs {
    const char* H;            // [B, W, d]
    const char* q;            // [B, d]
    const int32_t* positions; // [B, W] or null
    int B, W, d, delta;
    float* scores;            // [B, W] (workspace)
    int32_t* out_idx;         // [B, delta]
    int32_t* out_pos;         // [B, delta] or null
    float* out_score;         // [B, delta] or null
};

// Pair i of the values in a 16-byte vector (bfloat16: word i; fp32: words
// 2i and 2i + 1).
template <int ELT>
__device__ __forceinline__ f32x2 vec_pair(const uint4& v, int i) {
    if constexpr (ELT == 2) {
        const uint32_t w = u4_get(v, i);
        return f2_pack(bf16_lo(w), bf16_hi(w));
    } else {
        return f2_pack(__uint_as_float(u4_get(v, 2 * i)), __uint_as_float(u4_get(v, 2 * i + 1)));
    }
}

// One warp per window row.  A batch that lies wholly inside the row is
// loaded without per-vector bounds tests, so its loads issue together; the
// query vectors are read as they are used.  (One warp per row gives a grid of
// B x W/8 CTAs, 1920 for the cosine-b64 windows: measured 26.7 us against
// 31.6 us for four rows per warp.)
template <int ELT>
__global__ void __launch_bounds__(kCosThreads) cosine_scores_kernel(const CosArgs a) {
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int b = blockIdx.x;
    const int r = blockIdx.y * kCosRowsPerCta + warp;
    if (r >= a.W) return;
    const int nvec = a.d * ELT / 16;
    constexpr int NP = 8 / ELT;                           // pairs per vector
    const uint4* qrow = reinterpret_cast<const uint4*>(a.q + (size_t)b * a.d * ELT);
    const char* hrow = a.H + ((size_t)b * a.W + r) * a.d * ELT;
    f32x2 dot = f2_pack(0.f, 0.f), nh = dot, nq = dot;
    for (int v0 = lane; v0 < nvec; v0 += 32 * kCosBatch) {
        uint4 hv[kCosBatch];
        const bool whole = v0 + 32 * (kCosBatch - 1) < nvec;
        if (whole) {
#pragma unroll
            for (int u = 0; u < kCosBatch; ++u) hv[u] = ld_stream16(hrow + (size_t)(v0 + 32 * u) * 16);
        } else {
#pragma unroll
            for (int u = 0; u < kCosBatch; ++u) {
                const int v = v0 + 32 * u;
                hv[u] = v < nvec ? ld_stream16(hrow + (size_t)v * 16) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int u = 0; u < kCosBatch; ++u) {
            const int v = v0 + 32 * u;
            const uint4 qv = (whole || v < nvec) ? __ldg(qrow + v) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int i = 0; i < NP; ++i) {
                const f32x2 h2 = vec_pair<ELT>(hv[u], i), q2 = vec_pair<ELT>(qv, i);
                dot = f2_fma(h2, q2, dot);
                nh = f2_fma(h2, h2, nh);
                nq = f2_fma(q2, q2, nq);
            }
        }
    }
    float d0, d1, h0, h1, q0, q1;
    f2_unpack(dot, d0, d1);
    f2_unpack(nh, h0, h1);
    f2_unpack(nq, q0, q1);
    const float sd = warp_sum(d0 + d1), sh = warp_sum(h0 + h1), sq = warp_sum(q0 + q1);
    if (lane == 0)
        a.scores[(size_t)b * a.W + r] = (sh > 0.f && sq > 0.f) ? sd / sqrtf(sh) / sqrtf(sq) : 0.f;
}

constexpr int kCosTopWarps = 8;

template <int KC>
__global__ void __launch_bounds__(kCosTopWarps * 32) cosine_top_kernel(const CosArgs a) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kCosTopWarps + (threadIdx.x >> 5);
    if (b >= a.B) return;                                 // warp-uniform
    TopList<KC> L;
    L.init();
    for (int j = lane; j < a.W; j += 32) L.insert(__ldcg(a.scores + (size_t)b * a.W + j), j);
    float ov[KC];
    int oi[KC];
    warp_merge_topk<KC>(L, ov, oi);
    if (lane == 0)
        for (int k = 0; k < a.delta; ++k) {
            const bool have = k < KC && oi[k] >= 0 && oi[k] < a.W;
            const int j = have ? oi[k] : -1;
            a.out_idx[(size_t)b * a.delta + k] = j;
            if (a.out_pos)
                a.out_pos[(size_t)b * a.delta + k] =
                    have ? (a.positions ? a.positions[(size_t)b * a.W + j] : j) : -1;
            if (a.out_score) a.out_score[(size_t)b * a.delta + k] = have ? ov[k] : kNegInf;
        }
}

size_t cosine_workspace_size(int B, int W) {
    return 256 + align256(sizeof(float) * (size_t)B * (size_t)W);
}

cudaError_t launch_cosine(const void* hidden, const void* query, spec_dtype_t dt, int B, int W,
                          int d, int delta, const int32_t* positions, int32_t* out_idx,
                          int32_t* out_pos, float* out_score, void* ws, cudaStream_t st) {
    CosArgs a;
    a.H = static_cast<const char*>(hidden);
    a.q = static_cast<const char*>(query);
    a.positions = positions;
    a.B = B;
    a.W = W;
    a.d = d;
    a.delta = delta;
    a.scores = reinterpret_cast<float*>(static_cast<char*>(ws) + 256);
    a.out_idx = out_idx;
    a.out_pos = out_pos;
    a.out_score = out_score;
    const dim3 grid((unsigned)B, (unsigned)((W + kCosRowsPerCta - 1) / kCosRowsPerCta), 1);
    cudaError_t e = dt == SPEC_DTYPE_BF16 ? launch_pdl(cosine_scores_kernel<2>, grid, kCosThreads, 0, st, a)
                                          : launch_pdl(cosine_scores_kernel<4>, grid, kCosThreads, 0, st, a);
    if (e != cudaSuccess) return e;
    const dim3 tgrid((B + kCosTopWarps - 1) / kCosTopWarps);
    const int KC = topk_list_len(delta);
    if (KC == 2) return launch_pdl(cosine_top_kernel<2>, tgrid, kCosTopWarps * 32, 0, st, a);
    if (KC == 4) return launch_pdl(cosine_top_kernel<4>, tgrid, kCosTopWarps * 32, 0, st, a);
    return launch_pdl(cosine_top_kernel<8>, tgrid, kCosTopWarps * 32, 0, st, a);
}

}  // namespace sv
