// Greedy verification of draft chains and of draft trees: one streaming
// argmax pass over the target logits (sv_stream.cuh), and one CTA per
// sequence that merges its row partials and decides (sv_decide.cuh).  On
// 16-byte rows the decide kernel starts with the stream and runs beside it,
// taking each sequence once that sequence's (tagged) partials are in; on other
// rows it follows the stream with programmatic dependent launch.
//
// Sources: "Speculative decoding: guess a few tokens first - why the answer
// stays the same", greedy paragraph (accept while the draft equals the target
// argmax, emit the target token at the first mismatch); "AdaPLD: adaptive
// retrieval and reuse for efficient model-free speculative decoding", section
// 3.3 "Tree construction and verification" and Algorithm 1 (VerifyAndAccept
// over the draft tree built from the main chain and top-K branches).
//
// Ties: the lowest index among equal raw logits wins (values compared as
// floats, so -0.0 == +0.0; NaN logits are undefined).
#include "sv_stream.cuh"

namespace sv {

// One CTA per sequence.  Beside the stream: 8 warps of at most 80 registers
// (one CTA fits on an SM with two argmax-stream CTAs), waiting for the
// sequence's tagged partials; the last CTA then waits for the stream to
// complete, so that this kernel's completion covers it.  Behind the stream
// (rows that take the register path, trees of more than 32 nodes): 32 warps,
// a row's partials per warp and round of loads, after the stream completes.
constexpr int kArgmaxDecideThreads = 1024;
constexpr int kArgmaxBesideThreads = 256;

template <int NT>
__global__ void __launch_bounds__(NT, NT == kArgmaxBesideThreads ? 3 : 1) greedy_decide_kernel(const VerifyArgs a) {
    __shared__ ArgmaxDecideSmem sm;
    pdl_trigger();
    prefetch_tokens<NT>(a, blockIdx.x, threadIdx.x, false, sm);   // inputs: before the wait
    if (a.poll_parts) wait_seq_parts<NT>(a, blockIdx.x, threadIdx.x);
    else pdl_wait();
    decide_greedy<NT>(a, blockIdx.x, threadIdx.x, sm);
    if (a.poll_parts && blockIdx.x == gridDim.x - 1) pdl_wait();
}

template <int NT>
__global__ void __launch_bounds__(NT, NT == kArgmaxBesideThreads ? 3 : 1) tree_decide_kernel(const VerifyArgs a) {
    __shared__ ArgmaxDecideSmem sm;
    __shared__ TreeWalkSmem tw;
    pdl_trigger();
    prefetch_tokens<NT>(a, blockIdx.x, threadIdx.x, true, sm);
    if (a.poll_parts) wait_seq_parts<NT>(a, blockIdx.x, threadIdx.x);
    else pdl_wait();
    decide_tree<NT>(a, blockIdx.x, threadIdx.x, sm, tw);
    if (a.poll_parts && blockIdx.x == gridDim.x - 1) pdl_wait();
}

// The decide kernel beside the stream prefers the whole carveout as shared
// memory, as the ring stream does: an SM runs CTAs of several kernels only
// under one carveout.
template <int NT>
static cudaError_t launch_decide(void (*kfn)(VerifyArgs), const VerifyArgs& a, int B, cudaStream_t st,
                                 DeviceSlots& slots) {
    if (NT == kArgmaxBesideThreads) {
        int unused = 0;
        cudaError_t e = device_once(slots, &unused, [&](int, int* o) {
            *o = 1;
            return cudaFuncSetAttribute(kfn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                        cudaSharedmemCarveoutMaxShared);
        });
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(kfn, dim3(B), NT, 0, st, a);
}

static VerifyArgs argmax_args(const void* zt, int elt, int B, int rows, int V, void* ws) {
    const WsLayout L = ws_layout(B, rows, V);
    char* w = static_cast<char*>(ws);
    VerifyArgs a = {};
    a.wait_limit = ring_wait_limit();
    a.zt = static_cast<const char*>(zt);
    a.rows_per_seq = rows;
    a.V = V;
    a.nseg = nseg(V, elt);
    a.total_chunks = (long long)B * rows * a.nseg;
    a.B = B;
    a.parts = reinterpret_cast<float2*>(w + L.part_off);
    a.err = reinterpret_cast<int*>(w + L.err_off);
    const uint64_t tag = next_launch_tag();
    a.ptag = (uint32_t)tag ? (uint32_t)tag : 1u;
    a.poll_parts = ((size_t)V * elt) % 16 == 0 ? 1 : 0;  // ring stream: the decide runs beside it
    return a;
}

cudaError_t launch_greedy(const void* zt, spec_dtype_t dt, const int32_t* x, int B, int gamma,
                          int V, int32_t* out_tok, int32_t* out_acc, void* ws, cudaStream_t st) {
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int elt = elt_size(dt);
    VerifyArgs a = argmax_args(zt, elt, B, gamma + 1, V, ws);
    a.x = x;
    a.gamma = gamma;
    a.out_tok = out_tok;
    a.out_acc = out_acc;
    e = elt == 2 ? launch_stream<2, kModeGreedy>(a, di, st) : launch_stream<4, kModeGreedy>(a, di, st);
    if (e != cudaSuccess) return e;
    static DeviceSlots slots = {};
    if (a.poll_parts)
        return launch_decide<kArgmaxBesideThreads>(greedy_decide_kernel<kArgmaxBesideThreads>, a, B, st, slots);
    return launch_decide<kArgmaxDecideThreads>(greedy_decide_kernel<kArgmaxDecideThreads>, a, B, st, slots);
}

cudaError_t launch_tree(const void* zt, spec_dtype_t dt, const int32_t* tok, const int32_t* par,
                        int B, int N, int V, int32_t* out_nodes, int32_t* out_tok,
                        int32_t* out_acc, void* ws, cudaStream_t st) {
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int elt = elt_size(dt);
    VerifyArgs a = argmax_args(zt, elt, B, N, V, ws);
    a.x = tok;
    a.par = par;
    a.out_nodes = out_nodes;
    a.out_tok = out_tok;
    a.out_acc = out_acc;
    // Beside the stream only while the 8 warps merge every row in one round
    // (four rows a warp): larger trees are decided faster by 32 warps after
    // the stream (a 36-node tree: 56.5 against 58.1 us per call).
    if (N > 4 * kArgmaxBesideThreads / 32) a.poll_parts = 0;
    e = elt == 2 ? launch_stream<2, kModeTree>(a, di, st) : launch_stream<4, kModeTree>(a, di, st);
    if (e != cudaSuccess) return e;
    static DeviceSlots slots = {};
    if (a.poll_parts)
        return launch_decide<kArgmaxBesideThreads>(tree_decide_kernel<kArgmaxBesideThreads>, a, B, st, slots);
    return launch_decide<kArgmaxDecideThreads>(tree_decide_kernel<kArgmaxDecideThreads>, a, B, st, slots);
}

}  // namespace sv
