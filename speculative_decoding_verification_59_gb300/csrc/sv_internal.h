// Internal declarations shared by the translation units of libspecverify.so:
// the workspace layout, the chunking constants and the launch entry points
// that the C ABI (sv_api.cu) dispatches to.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "spec_verify.h"

namespace sv {

// One warp streams a "warp chunk" of 128 bytes per lane (8 x 16-byte vectors):
// 2048 bf16 or 1024 fp32 logits.  A CTA of kWarps warps covers a "block
// chunk" of kWarps consecutive warp chunks of one row.
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kLaneBytes = 128;
constexpr int kVecPerLane = kLaneBytes / 16;

inline int elt_size(spec_dtype_t dt) { return dt == SPEC_DTYPE_BF16 ? 2 : 4; }
inline int warp_elems(int elt) { return 32 * kLaneBytes / elt; }
inline int block_elems(int elt) { return kWarps * warp_elems(elt); }
inline int nseg(int V, int elt) { return (V + block_elems(elt) - 1) / block_elems(elt); }

// Elements of one row per CTA in the final-sample kernels: 32 contiguous
// elements per thread of a 256-thread CTA (four 16-byte vectors of bf16,
// eight of fp32).
constexpr int kFinalPerThread = 32;
constexpr int kFinalChunkThreads = 256;
constexpr int kFinalChunk = kFinalPerThread * kFinalChunkThreads;
inline int final_chunks(int V) { return (V + kFinalChunk - 1) / kFinalChunk; }
// Each warp of a final-pass CTA sums one "segment" of kFinalChunk / 8
// consecutive elements; the workspace keeps one total per segment.
constexpr int kFinalSegs = kFinalChunkThreads / 32;

// Tagged 64-bit words per SampleDesc (k, mt, md, rt) and per segment's sums
// (Za, Zb, W as float-float pairs, D, and a pad word).
constexpr int kDescWords = 4;
constexpr int kSumWords = 8;

// Per-sequence result of the accept decisions, read by the final-sample kernels.
struct SampleDesc {
    int k;        // rejection index (< gamma), gamma when all drafts were accepted, -1: bad input
    float mt;     // max logit of target row k
    float md;     // max logit of draft row k (rejection only)
    float rt;     // rejection: Z_t / Z_d of row k from the row statistics (~1e-6 accurate)
};

// Lazy sampling streams the positions in groups of doubling size (2, 4, 8,
// ...), the last group ending with target row gamma; gamma <= 256 needs at
// most kLazyGroups of them.  Group g > 0 reads the survivor list that the
// decide step of group g - 1 writes.
constexpr int kLazyGroups = 8;

// Workspace: [error word and the streams' claim counter (256 bytes
// reserved) | per-warp row partials | SampleDesc[B] (kDescWords tagged
// words each) | per-sequence finish tickets (tagged counts) | per-segment
// sums (kSumWords tagged words each) | lazy survivor counts (256 bytes) and
// lists [kLazyGroups, B]].
// A call's sampling partials, SampleDescs and segment sums are tagged words
// (sv_common.cuh) carrying the call's tag, and the tickets carry its launch
// tag; the lazy survivor counts are zeroed by the call's first lazy stream.
// So a workspace carries nothing from one call to the next except the error
// word, which only accumulates error bits until spec_verify_read_error clears
// it, whatever an earlier call (finished or not) left in it.
struct WsLayout {
    size_t err_off, part_off, part_count, desc_off, tick_off, sum_off, lz_off, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Byte offset of the streams' 64-bit claim counter inside the first 256
// bytes of a workspace (the error word is at offset 0).
constexpr size_t kClaimOff = 128;
// The counter holds (launch tag << kClaimIdxBits) | next chunk index.
constexpr int kClaimIdxBits = 24;
constexpr int kClaimTagBits = 64 - kClaimIdxBits;

inline WsLayout ws_layout(int B, int gamma_or_nodes, int V) {
    WsLayout L;
    L.err_off = 0;
    L.part_off = 256;
    // rows: sampling needs 2g+1 per sequence, greedy g+1, trees N (<= 2N+1)
    size_t rows = (size_t)B * (size_t)(2 * (size_t)gamma_or_nodes + 1);
    // fp32 has the smaller warp chunk, hence the most partials per row
    L.part_count = rows * (size_t)nseg(V, 4) * kWarps;
    // 16 bytes a partial: sampling stores them as tagged 64-bit word pairs
    L.desc_off = L.part_off + align256(2 * sizeof(float2) * L.part_count);
    const size_t segs = (size_t)B * (size_t)final_chunks(V) * kFinalSegs;
    L.tick_off = L.desc_off + align256(kDescWords * sizeof(unsigned long long) * (size_t)B);
    L.sum_off = L.tick_off + align256(sizeof(unsigned long long) * (size_t)B);
    L.lz_off = L.sum_off + align256(kSumWords * sizeof(unsigned long long) * segs);
    L.total = L.lz_off + 256 + align256(sizeof(int) * (size_t)kLazyGroups * (size_t)B);
    return L;
}

struct DeviceInfo {
    int sm_count;
    int max_smem_optin;
};
// Cached per-device properties (SM count and shared-memory limit).
cudaError_t device_info(DeviceInfo* out);

// A positive value computed once per device ordinal (a kernel's occupancy
// after its shared-memory opt-in, say) and cached for later calls.  Several
// host threads may race to compute it: setup must be idempotent and give the
// same value each time; the cache slot is atomic.  Devices past kMaxDevices
// are served uncached.
constexpr int kMaxDevices = 64;
using DeviceSlots = std::atomic<int>[kMaxDevices];

template <typename F>
inline cudaError_t device_once(DeviceSlots& slots, int* out, F setup) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) {
        const int v = slots[dev].load(std::memory_order_acquire);
        if (v > 0) { *out = v; return cudaSuccess; }
    }
    int v = 0;
    e = setup(dev, &v);
    if (e != cudaSuccess) return e;
    if (v < 1) v = 1;
    if (dev >= 0 && dev < kMaxDevices) slots[dev].store(v, std::memory_order_release);
    *out = v;
    return cudaSuccess;
}

// Polls of a bounded barrier wait inside the ring kernels before it gives up
// (seconds of wall time), and the value for launches made from now on: this
// default, unless spec_verify_set_wait_limit changed it.
constexpr uint32_t kWaitLimitDefault = 1u << 24;
uint32_t ring_wait_limit();
// A fresh nonzero launch tag (kClaimTagBits bits; process-wide, increasing
// until it wraps) for the claim counter of one stream launch.
uint64_t next_launch_tag();

// Upper ends of the lazy pass's position groups (host only; ends holds
// kLazyGroups entries); returns their count.
int lazy_groups_host(int B, int gamma, size_t rowbytes, int* ends);
// Sets the bytes after a group boundary that make the lazy pass split there
// (negative: the built-in figure).
void set_lazy_split_bytes(double bytes);

// Host-side checks of a sampling call's arguments that do not involve the
// workspace (spec_verify_sample and its variants, spec_verify_sample_noalloc):
// SPEC_OK, or the status to return before anything is launched.  `finish`:
// the call takes decisions (draft tokens, uniforms and outputs required).
// B = 0 passes; the caller returns SPEC_OK without launching.
spec_status_t check_sample_args(const void* target_logits, const void* draft_logits,
                                spec_dtype_t dtype, const int32_t* draft_tokens,
                                const float* uniforms, float temperature, int B, int gamma, int V,
                                const int32_t* out_tokens, const int32_t* out_num_accepted,
                                bool finish);
bool is_aligned(const void* p, size_t a);

// ---- launchers (return the first CUDA error) ------------------------------
// parts: kSampleStats (streaming row statistics), kSampleFinish (the accept
// decisions and the final residual/bonus token), both, or kSampleLazy.
constexpr int kSampleStats = 1;
constexpr int kSampleFinish = 2;
constexpr int kSampleLazy = 4;     // early-exit pass instead of stats + decisions, then the final sample
cudaError_t launch_sample(const void* zt, const void* zd, spec_dtype_t dt, const int32_t* x,
                          const float* u, float T, int B, int gamma, int V, int32_t* out_tok,
                          int32_t* out_acc, float* out_lp, void* ws, cudaStream_t st, int parts);

// Whether the final sampling pass supports this vocabulary size.
bool sample_supported_vocab(int V);

cudaError_t launch_greedy(const void* zt, spec_dtype_t dt, const int32_t* x, int B, int gamma,
                          int V, int32_t* out_tok, int32_t* out_acc, void* ws, cudaStream_t st);

cudaError_t launch_tree(const void* zt, spec_dtype_t dt, const int32_t* tok, const int32_t* par,
                        int B, int N, int V, int32_t* out_nodes, int32_t* out_tok,
                        int32_t* out_acc, void* ws, cudaStream_t st);

// Top-K branch tokens (K <= 8) of rows x V logits, one token per row excluded.
cudaError_t launch_topk(const void* logits, spec_dtype_t dt, int rows, int V, int K,
                        const int32_t* exclude, int32_t* out_idx, float* out_val, void* ws,
                        cudaStream_t st);
size_t topk_workspace_size(int rows, int V, int K);
int topk_list_len(int K);

// Lexical (n-gram) retrieval of reuse positions over B token streams.
cudaError_t launch_ngram(const int32_t* tokens, const int32_t* lengths, int B, int n_max, int w,
                         int L, int max_matches, int32_t* out_count, int32_t* out_matches,
                         int32_t* out_draft, void* ws, cudaStream_t st);
size_t ngram_workspace_size(int B, int n_max, int max_matches);

// Cosine top-delta over windows of hidden states (semantic fallback).
cudaError_t launch_cosine(const void* hidden, const void* query, spec_dtype_t dt, int B, int W,
                          int d, int delta, const int32_t* positions, int32_t* out_idx,
                          int32_t* out_pos, float* out_score, void* ws, cudaStream_t st);
size_t cosine_workspace_size(int B, int W);

}  // namespace sv
