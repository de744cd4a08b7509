// Greedy verification of draft chains and of draft trees: one streaming
// argmax pass over the target logits (sv_stream.cuh), then one CTA per
// sequence that merges its row partials and decides (sv_decide.cuh), chained
// with programmatic dependent launch.
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

// One CTA per sequence, chained behind the argmax stream (waits in hardware
// until the stream's partials are visible).  32 warps: a row's partials per
// warp and round of loads (a 36-node tree takes two rounds).
constexpr int kArgmaxDecideThreads = 1024;

__global__ void __launch_bounds__(kArgmaxDecideThreads) greedy_decide_kernel(const VerifyArgs a) {
    __shared__ ArgmaxDecideSmem sm;
    prefetch_tokens<kArgmaxDecideThreads>(a, blockIdx.x, threadIdx.x, false, sm);   // inputs: before the wait
    pdl_wait();
    decide_greedy<kArgmaxDecideThreads>(a, blockIdx.x, threadIdx.x, sm);
}

__global__ void __launch_bounds__(kArgmaxDecideThreads) tree_decide_kernel(const VerifyArgs a) {
    __shared__ ArgmaxDecideSmem sm;
    __shared__ TreeWalkSmem tw;
    prefetch_tokens<kArgmaxDecideThreads>(a, blockIdx.x, threadIdx.x, true, sm);
    pdl_wait();
    decide_tree<kArgmaxDecideThreads>(a, blockIdx.x, threadIdx.x, sm, tw);
}

static cudaError_t launch_decide(void (*kfn)(VerifyArgs), const VerifyArgs& a, int B, cudaStream_t st) {
    return launch_pdl(kfn, dim3(B), kArgmaxDecideThreads, 0, st, a);
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
    return launch_decide(greedy_decide_kernel, a, B, st);
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
    e = elt == 2 ? launch_stream<2, kModeTree>(a, di, st) : launch_stream<4, kModeTree>(a, di, st);
    if (e != cudaSuccess) return e;
    return launch_decide(tree_decide_kernel, a, B, st);
}

}  // namespace sv
