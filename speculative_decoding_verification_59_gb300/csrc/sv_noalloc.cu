// spec_verify_sample_noalloc: stochastic verification for callers that cannot
// allocate device memory.
//
// Some callers cannot hand the library a workspace: a plugin whose host
// framework owns every byte of device memory through its own pool and passes
// in nothing but the input and output tensors, or a decode loop that is not
// allowed to call cudaMalloc/cudaFree (both can synchronise the device) in
// the middle of a step.  For them this entry point runs exactly the kernels
// of spec_verify_sample, with the scratch taken from a fixed array that the
// library itself places in device memory (kNoAllocScratchBytes, 8 MiB).
// Every GPU that loads the library holds that array until the process exits.
//
// The array's host-side name is only a stand-in; its device address is looked
// up once per device with cudaGetSymbolAddress (on the first call made while
// that device is current) and passed to the kernels like any workspace.
#include <mutex>

#include "sv_internal.h"

namespace sv {

constexpr size_t kNoAllocScratchBytes = SPEC_VERIFY_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes % 256 == 0, "scratch must keep 256-byte granularity");

// The scratch shared by every call of spec_verify_sample_noalloc on a device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (first call per
// device: symbol lookup, which also loads the library's module there).
cudaError_t noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (p == nullptr) return cudaErrorInvalidSymbol;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace sv

extern "C" spec_status_t spec_verify_sample_noalloc(
    const void* target_logits, const void* draft_logits, spec_dtype_t dtype,
    const int32_t* draft_tokens, const float* uniforms, float temperature, int B, int gamma, int V,
    int32_t* out_tokens, int32_t* out_num_accepted, float* out_logprobs, cudaStream_t stream) {
    using namespace sv;
    // The argument rules of spec_verify_sample (the same check), then the size
    // of the fixed scratch.
    const spec_status_t s = check_sample_args(target_logits, draft_logits, dtype, draft_tokens,
                                              uniforms, temperature, B, gamma, V, out_tokens,
                                              out_num_accepted, true);
    if (s != SPEC_OK || B == 0) return s;
    if (ws_layout(B, gamma, V).total > kNoAllocScratchBytes) return SPEC_ERR_EXCEEDS_STATIC_SCRATCH;
    void* scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return SPEC_ERR_CUDA;
    // Every region the kernels read is written earlier in the same call, so
    // nothing in the scratch has to start at zero; the error word in its first
    // bytes only ever gains bits and is not reported by this entry point (bad
    // sequences still come back with -1).
    cudaError_t e = launch_sample(target_logits, draft_logits, dtype, draft_tokens, uniforms,
                                  temperature, B, gamma, V, out_tokens, out_num_accepted,
                                  out_logprobs, scratch, stream, kSampleStats | kSampleFinish);
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
