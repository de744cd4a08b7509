// Greedy verification of draft chains and draft trees: a streaming argmax
// pass over the target logits (argmax_kernel), then one CTA per sequence that
// merges the row partials and takes the decision (greedy_decide_kernel /
// tree_decide_kernel), chained with programmatic dependent launch.
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
#include "sv_common.cuh"
#include "sv_stream.cuh"

namespace sv {

constexpr int kMaxNodes = 1024;
constexpr int kDecideThreads = 256;

struct ArgmaxArgs {
    const char* zt;
    int V, nseg;
    long long total_chunks;
    float2* parts;      // (value, index bits) per warp chunk
};

struct DecideArgs {
    int rows_per_seq, V, nseg;
    const float2* parts;
    // greedy chains
    const int32_t* x;
    int gamma;
    // trees
    const int32_t* tok;
    const int32_t* par;
    int32_t* out_nodes;
    // both
    int32_t* out_tok;
    int32_t* out_acc;
    int* err;
};

template <int ELT, bool VEC>
__global__ void __launch_bounds__(kThreads) argmax_kernel(const ArgmaxArgs a) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int WE = 32 * kLaneBytes / ELT;
    const int P = a.nseg * kWarps;
    const size_t rowbytes = (size_t)a.V * ELT;

    for (long long c = blockIdx.x; c < a.total_chunks; c += gridDim.x) {
        if (c + gridDim.x >= a.total_chunks) pdl_trigger();
        const int seg = (int)(c % a.nseg);
        const long long rr = c / a.nseg;                 // global row: b * rows_per_seq + r
        const char* row = a.zt + (size_t)rr * rowbytes;
        const int base = (seg * kWarps + warp) * WE;

        float bv = kNegInf;
        int bi = 0x7fffffff;
        if (base < a.V) {
            LaneChunk<ELT, VEC> ch;
            ch.load(row, a.V, base, lane);
            // Lane elements come in increasing index order: strict '>' keeps
            // the first maximum.  +0.0f folds -0.0 into +0.0.
            bv = ch.val(0) + 0.0f;
            bi = ch.idx(base, lane, 0);
#pragma unroll
            for (int i = 1; i < LaneChunk<ELT, VEC>::EPL; ++i) {
                const float v = ch.val(i) + 0.0f;
                if (v > bv) { bv = v; bi = ch.idx(base, lane, i); }
            }
            if (bi >= a.V) bi = 0x7fffffff;               // only padding seen
            warp_argmax(bv, bi);
        }
        if (lane == 0) a.parts[(size_t)rr * P + seg * kWarps + warp] = make_float2(bv, __int_as_float(bi));
    }
}

// Merge the warp partials of every row of sequence b into s_g[row].
__device__ void merge_row_argmax(const DecideArgs& a, int b, int* s_g) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int P = a.nseg * kWarps;
    for (int r = warp; r < a.rows_per_seq; r += nwarps) {
        const float2* pr = a.parts + ((size_t)b * a.rows_per_seq + r) * P;
        float bv = kNegInf;
        int bi = 0x7fffffff;
        for (int p = lane; p < P; p += 32) {
            const float2 q = pr[p];
            const int qi = __float_as_int(q.y);
            if (am_better(q.x, qi, bv, bi)) { bv = q.x; bi = qi; }
        }
        warp_argmax(bv, bi);
        if (lane == 0) s_g[r] = bi;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kDecideThreads) greedy_decide_kernel(const DecideArgs a) {
    __shared__ int s_g[kMaxNodes];
    __shared__ int s_k;
    const int b = blockIdx.x;
    const int G = a.gamma;
    pdl_wait();
    merge_row_argmax(a, b, s_g);
    if (threadIdx.x == 0) {
        int bad = 0;
        for (int i = 0; i < G; ++i) {
            const int xi = a.x[(size_t)b * G + i];
            if (xi < 0 || xi >= a.V) bad = 1;
        }
        int k = G;
        if (bad) {
            atomicOr(a.err, SPEC_DEVERR_TOKEN_RANGE);
            k = -1;
        } else {
            for (int i = 0; i < G; ++i)
                if (a.x[(size_t)b * G + i] != s_g[i]) { k = i; break; }
        }
        s_k = k;
        a.out_acc[b] = k;
    }
    __syncthreads();
    const int k = s_k;
    for (int i = threadIdx.x; i <= G; i += blockDim.x) {
        int v = -1;
        if (k >= 0) v = i < k ? a.x[(size_t)b * G + i] : (i == k ? s_g[k] : -1);
        a.out_tok[(size_t)b * (G + 1) + i] = v;
    }
}

__global__ void __launch_bounds__(kDecideThreads) tree_decide_kernel(const DecideArgs a) {
    __shared__ int s_g[kMaxNodes];
    __shared__ int s_depth[kMaxNodes];
    __shared__ int s_best[kMaxNodes];
    __shared__ int s_len, s_bad;
    const int b = blockIdx.x;
    const int N = a.rows_per_seq;
    const int32_t* tok = a.tok + (size_t)b * N;
    const int32_t* par = a.par + (size_t)b * N;
    if (threadIdx.x == 0) s_bad = 0;
    pdl_wait();
    merge_row_argmax(a, b, s_g);          // ends with __syncthreads
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
        const int p = par[n];
        if (n == 0 ? p != -1 : (p < 0 || p >= n)) atomicOr(&s_bad, SPEC_DEVERR_TREE_PARENT);
        if (n > 0) {
            const int t = tok[n];
            if (t < 0 || t >= a.V) atomicOr(&s_bad, SPEC_DEVERR_TOKEN_RANGE);
        }
        s_depth[n] = 0;
        s_best[n] = -1;
    }
    __syncthreads();
    int32_t* on = a.out_nodes + (size_t)b * N;
    int32_t* ot = a.out_tok + (size_t)b * N;
    if (threadIdx.x == 0) {
        int len = -1;
        if (s_bad) {
            atomicOr(a.err, s_bad);
        } else {
            // Accepted: parent accepted and token == argmax of the parent's row.
            // Longest accepted continuation below each node, children (larger
            // ids) first; on equal length the lower child id wins.  Nodes whose
            // parent is not accepted are never reached from the root, so
            // acceptance of the parent is enforced by the walk itself.
            for (int n = N - 1; n >= 1; --n) {
                const int p = par[n];
                if (tok[n] != s_g[p]) continue;
                if (1 + s_depth[n] >= s_depth[p]) { s_depth[p] = 1 + s_depth[n]; s_best[p] = n; }
            }
            len = 0;
            int cur = 0;
            while (s_best[cur] >= 0) {
                cur = s_best[cur];
                on[len] = cur;
                ot[len] = tok[cur];
                ++len;
            }
            ot[len] = s_g[cur];
        }
        s_len = len;
        a.out_acc[b] = len;
    }
    __syncthreads();
    const int len = s_len;
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
        if (len < 0 || n >= len) on[n] = -1;
        if (len < 0 || n > len) ot[n] = -1;
    }
}

template <int ELT, bool VEC>
static cudaError_t launch_argmax_t(const ArgmaxArgs& a, cudaStream_t st) {
    static int occ = 0;
    if (occ == 0) {
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, argmax_kernel<ELT, VEC>, kThreads, 0) !=
                cudaSuccess || o < 1)
            o = 1;
        occ = o;
    }
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    long long g = (long long)di.sm_count * occ;
    if (a.total_chunks < g) g = a.total_chunks;
    argmax_kernel<ELT, VEC><<<(int)g, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

static cudaError_t launch_decide(void (*kfn)(DecideArgs), const DecideArgs& d, int B, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B, 1, 1);
    cfg.blockDim = dim3(kDecideThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kfn, d);
}

static cudaError_t stream_argmax(const void* zt, int elt, int B, int rows, int V, float2* parts,
                                 int* err, cudaStream_t st) {
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    // 16-byte rows: bulk-copy ring; otherwise the register path
    RingArgs ra = {};
    ra.zt = static_cast<const char*>(zt);
    ra.zd = nullptr;
    ra.gamma = -1;
    ra.rows_per_seq = rows;
    ra.V = V;
    ra.nseg = nseg(V, elt);
    ra.total_chunks = (long long)B * rows * ra.nseg;
    ra.parts = parts;
    ra.err = err;
    bool used = false;
    e = elt == 2 ? launch_ring<2, true>(ra, di, st, &used) : launch_ring<4, true>(ra, di, st, &used);
    if (e != cudaSuccess || used) return e;
    ArgmaxArgs a;
    a.zt = ra.zt;
    a.V = V;
    a.nseg = ra.nseg;
    a.total_chunks = ra.total_chunks;
    a.parts = parts;
    const bool vec = ((size_t)V * elt) % 16 == 0;
    if (elt == 2) return vec ? launch_argmax_t<2, true>(a, st) : launch_argmax_t<2, false>(a, st);
    return vec ? launch_argmax_t<4, true>(a, st) : launch_argmax_t<4, false>(a, st);
}

static DecideArgs decide_args(int elt, int rows, int V, void* ws, int gamma_or_nodes, int B) {
    const WsLayout L = ws_layout(B, gamma_or_nodes, V);
    char* w = static_cast<char*>(ws);
    DecideArgs d = {};
    d.rows_per_seq = rows;
    d.V = V;
    d.nseg = nseg(V, elt);
    d.parts = reinterpret_cast<const float2*>(w + L.part_off);
    d.err = reinterpret_cast<int*>(w + L.err_off);
    return d;
}

cudaError_t launch_greedy(const void* zt, spec_dtype_t dt, const int32_t* x, int B, int gamma,
                          int V, int32_t* out_tok, int32_t* out_acc, void* ws, cudaStream_t st) {
    const int elt = elt_size(dt);
    DecideArgs d = decide_args(elt, gamma + 1, V, ws, gamma, B);
    cudaError_t e = stream_argmax(zt, elt, B, gamma + 1, V, const_cast<float2*>(d.parts), d.err, st);
    if (e != cudaSuccess) return e;
    d.x = x;
    d.gamma = gamma;
    d.out_tok = out_tok;
    d.out_acc = out_acc;
    return launch_decide(greedy_decide_kernel, d, B, st);
}

cudaError_t launch_tree(const void* zt, spec_dtype_t dt, const int32_t* tok, const int32_t* par,
                        int B, int N, int V, int32_t* out_nodes, int32_t* out_tok,
                        int32_t* out_acc, void* ws, cudaStream_t st) {
    const int elt = elt_size(dt);
    DecideArgs d = decide_args(elt, N, V, ws, N, B);
    cudaError_t e = stream_argmax(zt, elt, B, N, V, const_cast<float2*>(d.parts), d.err, st);
    if (e != cudaSuccess) return e;
    d.tok = tok;
    d.par = par;
    d.out_nodes = out_nodes;
    d.out_tok = out_tok;
    d.out_acc = out_acc;
    return launch_decide(tree_decide_kernel, d, B, st);
}

}  // namespace sv
