// The C ABI of libspecverify.so: argument validation, workspace sizing and
// dispatch to the launchers.  Declarations and their contracts are in
// include/spec_verify.h.
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "sv_internal.h"

namespace sv {

constexpr int kMaxGammaApi = 256;
constexpr int kMaxNodesApi = 1024;
constexpr float kMinTemperature = 1e-20f;   // log2(e)/T stays a finite float

cudaError_t device_info(DeviceInfo* out) {
    // Immutable device properties, cached per device ordinal.
    static DeviceSlots sms = {}, smem = {};
    cudaError_t e = device_once(sms, &out->sm_count, [](int dev, int* v) {
        return cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev);
    });
    if (e != cudaSuccess) return e;
    return device_once(smem, &out->max_smem_optin, [](int dev, int* v) {
        return cudaDeviceGetAttribute(v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    });
}

static std::atomic<uint32_t> g_wait_limit{kWaitLimitDefault};

uint32_t ring_wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }

static std::atomic<uint64_t> g_launch_tag{0};
uint64_t next_launch_tag() {
    constexpr uint64_t mask = (1ull << kClaimTagBits) - 1;
    uint64_t t;
    do {
        t = (g_launch_tag.fetch_add(1, std::memory_order_relaxed) + 1) & mask;
    } while (t == 0);
    return t;
}

bool is_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
static bool aligned(const void* p, size_t a) { return is_aligned(p, a); }

spec_status_t check_sample_args(const void* target_logits, const void* draft_logits,
                                spec_dtype_t dtype, const int32_t* draft_tokens,
                                const float* uniforms, float temperature, int B, int gamma, int V,
                                const int32_t* out_tokens, const int32_t* out_num_accepted,
                                bool finish) {
    if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED_DTYPE;
    if (B < 0 || gamma < 0 || gamma > kMaxGammaApi || V <= 0) return SPEC_ERR_INVALID_ARG;
    if (!(temperature >= kMinTemperature) || !isfinite(temperature)) return SPEC_ERR_INVALID_ARG;
    if (B == 0) return SPEC_OK;
    if (!target_logits || (gamma > 0 && !draft_logits)) return SPEC_ERR_INVALID_ARG;
    if (finish && (!uniforms || !out_tokens || !out_num_accepted || (gamma > 0 && !draft_tokens)))
        return SPEC_ERR_INVALID_ARG;
    if (!aligned(target_logits, 16) || (gamma > 0 && !aligned(draft_logits, 16)))
        return SPEC_ERR_MISALIGNED;
    if (finish && !sample_supported_vocab(V)) return SPEC_ERR_INVALID_ARG;
    return SPEC_OK;
}

static spec_status_t check_ws(void* ws, size_t bytes, int B, int g, int V) {
    if (!ws) return SPEC_ERR_INVALID_ARG;
    if (!aligned(ws, 256)) return SPEC_ERR_MISALIGNED;
    if (bytes < ws_layout(B, g, V).total) return SPEC_ERR_WORKSPACE_TOO_SMALL;
    return SPEC_OK;
}

static spec_status_t to_status(cudaError_t e) { return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA; }

}  // namespace sv

using namespace sv;

extern "C" {

size_t spec_verify_workspace_size(int B, int gamma_or_nodes, int V) {
    if (B < 0 || gamma_or_nodes < 0 || V <= 0) return 0;
    return ws_layout(B, gamma_or_nodes, V).total;
}

spec_status_t spec_verify_workspace_init(void* workspace, size_t workspace_bytes,
                                         cudaStream_t stream) {
    if (!workspace) return SPEC_ERR_INVALID_ARG;
    return to_status(cudaMemsetAsync(workspace, 0, workspace_bytes, stream));
}

static spec_status_t sample_common(const void* target_logits, const void* draft_logits,
                                   spec_dtype_t dtype, const int32_t* draft_tokens,
                                   const float* uniforms, float temperature, int B, int gamma,
                                   int V, int32_t* out_tokens, int32_t* out_num_accepted,
                                   float* out_logprobs, void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream, int parts) {
    const bool finish = (parts & (kSampleFinish | kSampleLazy)) != 0;
    spec_status_t s = check_sample_args(target_logits, draft_logits, dtype, draft_tokens, uniforms,
                                        temperature, B, gamma, V, out_tokens, out_num_accepted,
                                        finish);
    if (s != SPEC_OK || B == 0) return s;
    s = check_ws(workspace, workspace_bytes, B, gamma, V);
    if (s != SPEC_OK) return s;
    return to_status(launch_sample(target_logits, draft_logits, dtype, draft_tokens, uniforms,
                                   temperature, B, gamma, V, out_tokens, out_num_accepted,
                                   out_logprobs, workspace, stream, parts));
}

spec_status_t spec_verify_sample(const void* target_logits, const void* draft_logits,
                                 spec_dtype_t dtype, const int32_t* draft_tokens,
                                 const float* uniforms, float temperature, int B, int gamma,
                                 int V, int32_t* out_tokens, int32_t* out_num_accepted,
                                 float* out_logprobs, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream) {
    return sample_common(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                         B, gamma, V, out_tokens, out_num_accepted, out_logprobs, workspace,
                         workspace_bytes, stream, kSampleStats | kSampleFinish);
}

spec_status_t spec_verify_sample_lazy(const void* target_logits, const void* draft_logits,
                                      spec_dtype_t dtype, const int32_t* draft_tokens,
                                      const float* uniforms, float temperature, int B, int gamma,
                                      int V, int32_t* out_tokens, int32_t* out_num_accepted,
                                      float* out_logprobs, void* workspace, size_t workspace_bytes,
                                      cudaStream_t stream) {
    return sample_common(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                         B, gamma, V, out_tokens, out_num_accepted, out_logprobs, workspace,
                         workspace_bytes, stream, kSampleLazy);
}

int spec_verify_lazy_groups(int B, int gamma, int V, spec_dtype_t dtype, int32_t* ends) {
    if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return 0;
    if (B < 1 || gamma < 0 || gamma > kMaxGammaApi || V < 1 || !ends) return 0;
    int e[kLazyGroups];
    const int n = lazy_groups_host(B, gamma, (size_t)V * elt_size(dtype), e);
    for (int g = 0; g < n; ++g) ends[g] = e[g];
    return n;
}

spec_status_t spec_verify_sample_stats(const void* target_logits, const void* draft_logits,
                                       spec_dtype_t dtype, float temperature, int B, int gamma,
                                       int V, void* workspace, size_t workspace_bytes,
                                       cudaStream_t stream) {
    return sample_common(target_logits, draft_logits, dtype, nullptr, nullptr, temperature, B,
                         gamma, V, nullptr, nullptr, nullptr, workspace, workspace_bytes, stream,
                         kSampleStats);
}

spec_status_t spec_verify_sample_finish(const void* target_logits, const void* draft_logits,
                                        spec_dtype_t dtype, const int32_t* draft_tokens,
                                        const float* uniforms, float temperature, int B,
                                        int gamma, int V, int32_t* out_tokens,
                                        int32_t* out_num_accepted, float* out_logprobs,
                                        void* workspace, size_t workspace_bytes,
                                        cudaStream_t stream) {
    return sample_common(target_logits, draft_logits, dtype, draft_tokens, uniforms, temperature,
                         B, gamma, V, out_tokens, out_num_accepted, out_logprobs, workspace,
                         workspace_bytes, stream, kSampleFinish);
}

spec_status_t spec_verify_greedy(const void* target_logits, spec_dtype_t dtype,
                                 const int32_t* draft_tokens, int B, int gamma, int V,
                                 int32_t* out_tokens, int32_t* out_num_accepted, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream) {
    if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED_DTYPE;
    if (B < 0 || gamma < 0 || gamma + 1 > kMaxNodesApi || V <= 0)
        return SPEC_ERR_INVALID_ARG;
    if (B == 0) return SPEC_OK;
    if (!target_logits || !out_tokens || !out_num_accepted || (gamma > 0 && !draft_tokens))
        return SPEC_ERR_INVALID_ARG;
    if (!aligned(target_logits, 16)) return SPEC_ERR_MISALIGNED;
    spec_status_t s = check_ws(workspace, workspace_bytes, B, gamma, V);
    if (s != SPEC_OK) return s;
    return to_status(launch_greedy(target_logits, dtype, draft_tokens, B, gamma, V, out_tokens,
                                   out_num_accepted, workspace, stream));
}

spec_status_t spec_verify_tree_greedy(const void* target_logits, spec_dtype_t dtype,
                                      const int32_t* node_tokens, const int32_t* parents, int B,
                                      int N, int V, int32_t* out_path_nodes, int32_t* out_tokens,
                                      int32_t* out_num_accepted, void* workspace,
                                      size_t workspace_bytes, cudaStream_t stream) {
    if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED_DTYPE;
    if (B < 0 || N <= 0 || N > kMaxNodesApi || V <= 0) return SPEC_ERR_INVALID_ARG;
    if (B == 0) return SPEC_OK;
    if (!target_logits || !node_tokens || !parents || !out_path_nodes || !out_tokens ||
        !out_num_accepted)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned(target_logits, 16)) return SPEC_ERR_MISALIGNED;
    spec_status_t s = check_ws(workspace, workspace_bytes, B, N, V);
    if (s != SPEC_OK) return s;
    return to_status(launch_tree(target_logits, dtype, node_tokens, parents, B, N, V,
                                 out_path_nodes, out_tokens, out_num_accepted, workspace, stream));
}

size_t spec_topk_workspace_size(int rows, int V, int K) {
    if (rows < 0 || V <= 0 || K < 1 || K > 8) return 0;
    return topk_workspace_size(rows, V, K);
}

spec_status_t spec_topk_exclude(const void* logits, spec_dtype_t dtype, int rows, int V, int K,
                                const int32_t* exclude, int32_t* out_idx, float* out_val,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED_DTYPE;
    if (rows < 0 || V <= 0 || K < 1 || K > 8) return SPEC_ERR_INVALID_ARG;
    if ((long long)rows * nseg(V, elt_size(dtype)) >= (1LL << 31)) return SPEC_ERR_INVALID_ARG;
    if (rows == 0) return SPEC_OK;
    if (!logits || !out_idx || !workspace) return SPEC_ERR_INVALID_ARG;
    if (!aligned(logits, 16)) return SPEC_ERR_MISALIGNED;
    if (!aligned(workspace, 256)) return SPEC_ERR_MISALIGNED;
    if (workspace_bytes < topk_workspace_size(rows, V, K)) return SPEC_ERR_WORKSPACE_TOO_SMALL;
    return to_status(launch_topk(logits, dtype, rows, V, K, exclude, out_idx, out_val, workspace,
                                 stream));
}

size_t spec_ngram_workspace_size(int B, int n_max, int max_matches) {
    if (B < 0 || n_max < 4 || n_max % 4 != 0 || max_matches < 1 || max_matches > 4096) return 0;
    return ngram_workspace_size(B, n_max, max_matches);
}

spec_status_t spec_ngram_retrieve(const int32_t* tokens, const int32_t* lengths, int B, int n_max,
                                  int w, int L, int max_matches, int32_t* out_count,
                                  int32_t* out_matches, int32_t* out_draft, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream) {
    if (B < 0 || n_max < 4 || w < 1 || w > 8 || L < 0 || L > 1024 || max_matches < 1 ||
        max_matches > 4096)
        return SPEC_ERR_INVALID_ARG;
    if (n_max % 4 != 0) return SPEC_ERR_MISALIGNED;
    if (B == 0) return SPEC_OK;
    if (!tokens || !lengths || !out_count || !out_matches || !workspace) return SPEC_ERR_INVALID_ARG;
    if (!aligned(tokens, 16)) return SPEC_ERR_MISALIGNED;
    if (!aligned(workspace, 256)) return SPEC_ERR_MISALIGNED;
    if (workspace_bytes < ngram_workspace_size(B, n_max, max_matches))
        return SPEC_ERR_WORKSPACE_TOO_SMALL;
    return to_status(launch_ngram(tokens, lengths, B, n_max, w, L, max_matches, out_count,
                                  out_matches, out_draft, workspace, stream));
}

size_t spec_cosine_workspace_size(int B, int W) {
    if (B < 0 || W < 1) return 0;
    return cosine_workspace_size(B, W);
}

spec_status_t spec_cosine_topk(const void* hidden, const void* query, spec_dtype_t dtype, int B,
                               int W, int d, int delta, const int32_t* positions,
                               int32_t* out_idx, int32_t* out_pos, float* out_score,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED_DTYPE;
    if (B < 0 || W < 1 || d < 1 || delta < 1 || delta > 8) return SPEC_ERR_INVALID_ARG;
    if ((d * elt_size(dtype)) % 16 != 0) return SPEC_ERR_MISALIGNED;
    if (B == 0) return SPEC_OK;
    if (!hidden || !query || !out_idx || !workspace) return SPEC_ERR_INVALID_ARG;
    if (!aligned(hidden, 16) || !aligned(query, 16) || !aligned(workspace, 256))
        return SPEC_ERR_MISALIGNED;
    if (workspace_bytes < cosine_workspace_size(B, W)) return SPEC_ERR_WORKSPACE_TOO_SMALL;
    return to_status(launch_cosine(hidden, query, dtype, B, W, d, delta, positions, out_idx,
                                   out_pos, out_score, workspace, stream));
}

spec_status_t spec_verify_read_error(void* workspace, cudaStream_t stream, int32_t* code) {
    if (!workspace || !code) return SPEC_ERR_INVALID_ARG;
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(int32_t), stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return SPEC_ERR_CUDA;
    *code = v;
    return SPEC_OK;
}

void spec_verify_set_lazy_split_bytes(double bytes) { set_lazy_split_bytes(bytes); }

void spec_verify_set_wait_limit(uint32_t polls) {
    g_wait_limit.store(polls, std::memory_order_relaxed);
}

uint32_t spec_verify_default_wait_limit(void) { return kWaitLimitDefault; }

const char* spec_verify_status_string(spec_status_t status) {
    switch (status) {
        case SPEC_OK: return "ok";
        case SPEC_ERR_INVALID_ARG: return "invalid argument";
        case SPEC_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
        case SPEC_ERR_MISALIGNED: return "misaligned pointer (logits need 16 bytes, workspace 256)";
        case SPEC_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case SPEC_ERR_CUDA: return "CUDA runtime error";
        case SPEC_ERR_DEVICE_INPUT: return "bad input detected on the device";
        case SPEC_ERR_EXCEEDS_STATIC_SCRATCH:
            return "problem needs more scratch than the fixed array of spec_verify_sample_noalloc";
    }
    return "unknown status";
}

}  // extern "C"
