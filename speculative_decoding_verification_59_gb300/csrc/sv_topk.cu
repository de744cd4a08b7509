// Branch tokens of a draft tree: the top K tokens of each logit row with one
// token excluded.
//
// Source: "AdaPLD: adaptive retrieval and reuse for efficient model-free
// speculative decoding", section 3.3 (strict hit path: the branches are the
// target model's top K next tokens, without the token the copied main path
// already starts with) and Algorithm 1 (TopKNextTokens(M, x_{<=p*}, K) minus
// {d_main[1]}; without the exclusion on the semantic hit path).
//
// The top K of a row is taken by (larger logit, lower index): temperature does
// not change it.  The excluded token is removed from that list afterwards,
// which leaves K-1 tokens when it was among them; the list is padded with -1.
//
// One streaming pass (sv_stream.cuh, top-K mode) turns every 4 KB warp chunk
// of every row into at most 2 KC candidates that include the chunk's top KC
// (KC = 2, 4 or 8, the smallest that is at least K); one warp per row then
// merges the row's candidates into its top KC and applies the exclusion,
// chained behind the stream with programmatic dependent launch.
#include "sv_stream.cuh"

namespace sv {

constexpr int kTopkRowsPerCta = kThreads / 32;
constexpr int kOnePass = 24;          // candidates a lane holds in registers (640 a row for V = 151936 bf16)

// The candidates carry no -0.0 (the stream adds 0.0 to every value it
// stores), so ordering them by ord_key (sv_common.cuh) is ordering them by value.

// The KC-th largest of the 32 lanes' x (KC rounds of a warp maximum of the
// keys, the lowest lane holding it dropping out): KC values of distinct lanes.
template <int KC>
__device__ __forceinline__ float kth_lane_max(float x, int lane) {
    int k = ord_key(x), t = kNoKey;
#pragma unroll
    for (int r = 0; r < KC; ++r) {
        t = __reduce_max_sync(0xffffffffu, k);
        const unsigned own = __ballot_sync(0xffffffffu, k == t);
        if (lane == __ffs(own) - 1) k = kNoKey;
    }
    return key_value(t);
}

// The KC best of at most 32 entries held one to a lane (c, present when
// has), best first: KC rounds of the largest key, then the lowest index among
// the lanes holding it (larger value first, lower index first among equal
// values); (-inf, INT_MAX) once none is left.
template <int KC>
__device__ __forceinline__ void lanes_topk(float2 c, bool has, float (&ov)[KC], int (&oi)[KC]) {
    int ck = has ? ord_key(c.x) : kNoKey;
    const unsigned ci = has ? (unsigned)__float_as_int(c.y) : 0xffffffffu;
#pragma unroll
    for (int r = 0; r < KC; ++r) {
        const int t = __reduce_max_sync(0xffffffffu, ck);
        const unsigned j = __reduce_min_sync(0xffffffffu, ck == t ? ci : 0xffffffffu);
        const bool none = t == kNoKey;
        ov[r] = none ? kNegInf : key_value(t);
        oi[r] = none ? 0x7fffffff : (int)j;
        if (ck == t && ci == j) ck = kNoKey;
    }
}

template <int KC>
__global__ void __launch_bounds__(kThreads) topk_merge_kernel(const VerifyArgs a, int K,
                                                              const int32_t* exclude,
                                                              float* out_val) {
    constexpr int KS = topk_slots(KC);
    __shared__ float2 tk_pool[kTopkRowsPerCta][32];      // a warp's entries that reach thr
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * kTopkRowsPerCta + (threadIdx.x >> 5);
    if (r >= a.B) return;                                 // warp-uniform
    // The row's candidates are one contiguous array of n entries.  The row's
    // top KC are all at least thr, the KC-th largest of the 32 lane maxima.
    // When the row's entries fit kOnePass a lane, they are loaded in one round
    // and kept in registers; the few that reach thr (at least KC, a handful
    // more as a rule) go one to a lane through shared memory and lanes_topk
    // orders them.  Otherwise (more than 32 reach thr, or longer rows) the
    // lanes insert them into sorted lists, merged by warp_merge_topk; longer
    // rows take a pass for thr and a second pass that reloads them.
    const int n = a.nseg * kWarps * KS;
    const float2* pr = a.parts + (size_t)r * n;
    float ov[KC];
    int oi[KC];
    if (n <= 32 * kOnePass) {                             // warp-uniform
        float2 e[kOnePass];
#pragma unroll
        for (int q = 0; q < kOnePass; ++q) {
            const int i = lane + 32 * q;
            e[q] = i < n ? __ldcg(pr + i) : make_float2(kNegInf, __int_as_float(0x7fffffff));
        }
        float x = kNegInf;
#pragma unroll
        for (int q = 0; q < kOnePass; ++q) x = fmaxf(x, e[q].x);
        const float thr = kth_lane_max<KC>(x, lane);
        unsigned sel = 0u;                                // bit q: e[q] reaches thr
#pragma unroll
        for (int q = 0; q < kOnePass; ++q) sel |= (e[q].x >= thr ? 1u : 0u) << q;
        const int cnt = __popc(sel);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        if (total <= 32) {                                // warp-uniform: nearly always
            float2* pool = tk_pool[threadIdx.x >> 5];
            int pos = incl - cnt;
#pragma unroll
            for (int q = 0; q < kOnePass; ++q)
                if ((sel >> q) & 1u) pool[pos++] = e[q];
            __syncwarp();
            lanes_topk<KC>(pool[lane], lane < total, ov, oi);
        } else {
            // rare (many equal values): the marked entries are reloaded, so
            // that e stays in registers
            TopList<KC> L;
            L.init();
#pragma unroll 1
            for (int q = 0; q < kOnePass; ++q)
                if ((sel >> q) & 1u) {
                    const int i = lane + 32 * q;
                    const float2 t = i < n ? __ldcg(pr + i) : make_float2(kNegInf, __int_as_float(0x7fffffff));
                    L.insert(t.x, __float_as_int(t.y));
                }
            warp_merge_topk<KC>(L, ov, oi);
        }
    } else {
        TopList<KC> L;
        L.init();
        constexpr int kBatch = 8;                         // loads in flight per lane
        float x = kNegInf;
        for (int q0 = lane; q0 < n; q0 += 32 * kBatch) {
            float2 e[kBatch];
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const int i = q0 + 32 * q;
                e[q] = i < n ? __ldcg(pr + i) : make_float2(kNegInf, 0.f);
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q) x = fmaxf(x, e[q].x);
        }
        const float thr = kth_lane_max<KC>(x, lane);
        for (int q0 = lane; q0 < n; q0 += 32 * kBatch) {
            float2 e[kBatch];
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const int i = q0 + 32 * q;
                e[q] = i < n ? __ldcg(pr + i) : make_float2(kNegInf, __int_as_float(0x7fffffff));
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q)
                if (e[q].x >= thr) L.insert(e[q].x, __float_as_int(e[q].y));
        }
        warp_merge_topk<KC>(L, ov, oi);
    }
    if (lane == 0) {
        const int ex = exclude ? exclude[r] : -1;
        int o = 0;
#pragma unroll
        for (int k = 0; k < KC; ++k) {
            const bool keep = k < K && oi[k] >= 0 && oi[k] < a.V && oi[k] != ex;
            if (keep) {
                a.out_tok[(size_t)r * K + o] = oi[k];
                if (out_val) out_val[(size_t)r * K + o] = ov[k];
                ++o;
            }
        }
        for (; o < K; ++o) {
            a.out_tok[(size_t)r * K + o] = -1;
            if (out_val) out_val[(size_t)r * K + o] = kNegInf;
        }
    }
}

int topk_list_len(int K) { return K <= 2 ? 2 : K <= 4 ? 4 : 8; }

template <int KC>
static cudaError_t launch_topk_t(const VerifyArgs& a, int elt, int K, const int32_t* exclude,
                                 float* out_val, const DeviceInfo& di, cudaStream_t st) {
    constexpr int MODE = KC == 2 ? kModeTopK2 : KC == 4 ? kModeTopK4 : kModeTopK8;
    cudaError_t e = elt == 2 ? launch_stream<2, MODE>(a, di, st) : launch_stream<4, MODE>(a, di, st);
    if (e != cudaSuccess) return e;
    // the merge prefers the whole carveout as shared memory, as the ring
    // stream does, so that its CTAs can wait on SMs that hold stream CTAs
    // (an SM runs CTAs of several kernels only under one carveout)
    static DeviceSlots slots = {};
    int unused = 0;
    e = device_once(slots, &unused, [&](int, int* o) {
        *o = 1;
        return cudaFuncSetAttribute(topk_merge_kernel<KC>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                    cudaSharedmemCarveoutMaxShared);
    });
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_merge_kernel<KC>, dim3((a.B + kTopkRowsPerCta - 1) / kTopkRowsPerCta),
                      kThreads, 0, st, a, K, exclude, out_val);
}

cudaError_t launch_topk(const void* logits, spec_dtype_t dt, int rows, int V, int K,
                        const int32_t* exclude, int32_t* out_idx, float* out_val, void* ws,
                        cudaStream_t st) {
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int elt = elt_size(dt);
    char* w = static_cast<char*>(ws);
    VerifyArgs a = {};
    a.wait_limit = ring_wait_limit();
    a.zt = static_cast<const char*>(logits);
    a.rows_per_seq = 1;
    a.V = V;
    a.nseg = nseg(V, elt);
    a.total_chunks = (long long)rows * a.nseg;
    a.B = rows;
    a.parts = reinterpret_cast<float2*>(w + 256);
    a.err = reinterpret_cast<int*>(w);
    a.out_tok = out_idx;
    const int KC = topk_list_len(K);
    if (KC == 2) return launch_topk_t<2>(a, elt, K, exclude, out_val, di, st);
    if (KC == 4) return launch_topk_t<4>(a, elt, K, exclude, out_val, di, st);
    return launch_topk_t<8>(a, elt, K, exclude, out_val, di, st);
}

size_t topk_workspace_size(int rows, int V, int K) {
    // error word, then 2 KC candidate entries per warp chunk (fp32 has the most chunks)
    return 256 + align256(sizeof(float2) * (size_t)rows * (size_t)nseg(V, 4) * kWarps *
                          (size_t)topk_slots(topk_list_len(K)));
}

}  // namespace sv
