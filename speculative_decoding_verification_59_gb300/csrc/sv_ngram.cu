// Lexical retrieval of a reuse position: every earlier position of a
// sequence's context whose w-token window equals the context's last w tokens,
// and the draft that copies the tokens after the most recent such position.
//
// Source: "AdaPLD: adaptive retrieval and reuse for efficient model-free
// speculative decoding", section 3.2 (lexical retrieval stage: candidates are
// the positions where the most recent token occurs with the preceding tokens
// matching too), section 3.3 (strict hit path: the main draft copies the span
// after the reuse position) and Algorithm 1 (LexicalRetrieval, d_main).  The
// pages rank candidates by hidden-state similarity; that rerank is outside
// this library, and the most recent match is the reuse position here.
//
// Pass 1 (ngram_scan_kernel<W>, the window length a template argument):
// each sequence's context is split into S segments (one 4096-position tile
// each, up to 64 segments), one CTA each, so that many short CTAs overlap
// their load latencies.  A CTA walks its segment in tiles of 4096 positions;
// thread t tests the 16 positions of four 16-byte loads, holding the tokens
// before them from one or two more loads (L1 hits: the neighbouring thread's
// own vectors), against the query reversed in registers -- W compares per
// position, every index a compile-time constant.  Block scans of the
// per-thread match counts keep the segment's match list in position order.
// Pass 2 (ngram_merge_kernel, one warp per sequence) concatenates the
// segments' lists, counts, and copies the draft.
#include "sv_common.cuh"

namespace sv {

constexpr int kNgThreads = 256;
constexpr int kNgPer = 16;                       // positions per thread and tile
constexpr int kNgTile = kNgThreads * kNgPer;     // positions per tile
constexpr int kNgMaxW = 8;
constexpr int kNgMaxSeg = 64;

struct NgArgs {
    const int32_t* tok;      // [B, n_max]
    const int32_t* len;      // [B]
    int B, n_max, w, L, max_matches, S, seg_len;
    int32_t* seg_count;      // [B, S]: matches in the segment, -1: bad sequence
    int32_t* seg_last;       // [B, S]: last match in the segment, -1: none
    int32_t* seg_matches;    // [B, S, max_matches]
    int32_t* out_count;      // [B]
    int32_t* out_matches;    // [B, max_matches]
    int32_t* out_draft;      // [B, L]
    int* err;
};

// Exclusive block scan of one int per thread (kNgThreads); *total gets the sum.
__device__ __forceinline__ int block_excl_scan_int(int v, int* wsum, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int y = lane < kNgThreads / 32 ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int z = __shfl_up_sync(0xffffffffu, y, o);
            if (lane >= o) y += z;
        }
        if (lane < kNgThreads / 32) wsum[lane] = y;
    }
    __syncthreads();
    const int before = warp > 0 ? wsum[warp - 1] : 0;
    *total = wsum[kNgThreads / 32 - 1];
    __syncthreads();
    return before + x - v;
}

__device__ __forceinline__ int4 ld_tok4(const int32_t* p) {
    return __ldg(reinterpret_cast<const int4*>(p));
}

template <int W>
__global__ void __launch_bounds__(kNgThreads) ngram_scan_kernel(const NgArgs a) {
    static_assert(W >= 1 && W <= kNgMaxW, "window length");
    __shared__ int q[kNgMaxW];
    __shared__ int wsum[kNgThreads / 32];
    __shared__ int s_last;
    pdl_wait();
    const int b = blockIdx.x / a.S, s = blockIdx.x % a.S, tid = threadIdx.x;
    const int32_t* t = a.tok + (size_t)b * a.n_max;
    const int n = a.len[b];
    const size_t so = (size_t)b * a.S + s;
    if (n < 1 || n > a.n_max) {                           // block-uniform
        if (tid == 0) {
            a.seg_count[so] = -1;
            a.seg_last[so] = -1;
            if (s == 0) atomicOr(a.err, SPEC_DEVERR_TOKEN_RANGE);
        }
        return;
    }
    if (tid < W) q[tid] = n >= W ? t[n - W + tid] : 0;
    if (tid == 0) s_last = -1;
    __syncthreads();
    // the query reversed: qr[j] must equal the token j places before a candidate's end
    int qr[W];
#pragma unroll
    for (int j = 0; j < W; ++j) qr[j] = q[W - 1 - j];
    // positions of this segment that can match: [lo, hi)
    const int lo = max(s * a.seg_len, W - 1);
    const int hi = min((s + 1) * a.seg_len, n - 1);
    int count = 0;
    int32_t* segm = a.seg_matches + so * a.max_matches;
    for (int p0 = s * a.seg_len; p0 < hi; p0 += kNgTile) {
        const int p = p0 + kNgPer * tid;
        unsigned mask = 0u;
        if (p < hi && p + kNgPer - 1 >= lo) {
            // x[k] = token at p - 8 + k, k = 0..8+kNgPer-1 (-1 outside [0, n_max))
            int x[8 + kNgPer];
            const int4 none = make_int4(-1, -1, -1, -1);
            const int4 m2 = (W > 5 && p >= 8) ? ld_tok4(t + p - 8) : none;
            const int4 m1 = (W > 1 && p >= 4) ? ld_tok4(t + p - 4) : none;
            x[0] = m2.x; x[1] = m2.y; x[2] = m2.z; x[3] = m2.w;
            x[4] = m1.x; x[5] = m1.y; x[6] = m1.z; x[7] = m1.w;
            int4 c[kNgPer / 4];
            if (p + kNgPer <= a.n_max) {                   // all four loads issue together
#pragma unroll
                for (int v = 0; v < kNgPer / 4; ++v) c[v] = ld_tok4(t + p + 4 * v);
            } else {
#pragma unroll
                for (int v = 0; v < kNgPer / 4; ++v) c[v] = p + 4 * v < a.n_max ? ld_tok4(t + p + 4 * v) : none;
            }
#pragma unroll
            for (int v = 0; v < kNgPer / 4; ++v) {
                x[8 + 4 * v] = c[v].x;
                x[9 + 4 * v] = c[v].y;
                x[10 + 4 * v] = c[v].z;
                x[11 + 4 * v] = c[v].w;
            }
#pragma unroll
            for (int e = 0; e < kNgPer; ++e) {
                bool eq = p + e >= lo && p + e < hi;
#pragma unroll
                for (int j = 0; j < W; ++j) eq = eq && x[8 + e - j] == qr[j];
                mask |= (eq ? 1u : 0u) << e;
            }
        }
        if (!__syncthreads_or(mask != 0u)) continue;       // most tiles hold no match
        int total;
        const int off = block_excl_scan_int(__popc(mask), wsum, &total);
        int k = count + off;
        for (unsigned m = mask; m; m &= m - 1u) {
            if (k < a.max_matches) segm[k] = p + __ffs(m) - 1;
            ++k;
        }
        if (mask) atomicMax(&s_last, p + 31 - __clz(mask));
        count += total;
    }
    __syncthreads();
    if (tid == 0) {
        a.seg_count[so] = count;
        a.seg_last[so] = s_last;
    }
}

constexpr int kNgMergeWarps = 8;

// One warp per sequence: lane l owns segments l and l + 32 (S <= 64).  A warp
// scan of the segment counts places every segment's list, the lanes copy in
// parallel, and the highest segment with a match gives the reuse position.
__global__ void __launch_bounds__(kNgMergeWarps * 32) ngram_merge_kernel(const NgArgs a) {
    static_assert(kNgMaxSeg <= 64, "two segments per lane");
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kNgMergeWarps + (threadIdx.x >> 5);
    if (b >= a.B) return;                                 // warp-uniform
    int32_t* om = a.out_matches + (size_t)b * a.max_matches;
    int32_t* od = a.out_draft ? a.out_draft + (size_t)b * a.L : nullptr;
    const int32_t* sc = a.seg_count + (size_t)b * a.S;
    const int s0 = lane, s1 = lane + 32;
    const int c0 = s0 < a.S ? __ldcg(sc + s0) : 0;
    const int c1 = s1 < a.S ? __ldcg(sc + s1) : 0;
    if (__shfl_sync(0xffffffffu, c0, 0) < 0) {           // bad sequence (every segment says so)
        if (lane == 0) a.out_count[b] = -1;
        for (int k = lane; k < a.max_matches; k += 32) om[k] = -1;
        if (od) for (int k = lane; k < a.L; k += 32) od[k] = -1;
        return;
    }
    int i0 = c0, i1 = c1;                                 // inclusive scans
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y0 = __shfl_up_sync(0xffffffffu, i0, o);
        const int y1 = __shfl_up_sync(0xffffffffu, i1, o);
        if (lane >= o) { i0 += y0; i1 += y1; }
    }
    const int t0 = __shfl_sync(0xffffffffu, i0, 31);
    const int total = t0 + __shfl_sync(0xffffffffu, i1, 31);
    const int off0 = i0 - c0, off1 = t0 + i1 - c1;
    // Lane l copies the lists of its segments l and l + 32, four loads in
    // flight at a time.
    auto copy_list = [&](const int32_t* m, int cnt, int off) {
        for (int k0 = 0; k0 < cnt && off + k0 < a.max_matches; k0 += 4) {
            int v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int k = k0 + u;
                v[u] = (k < cnt && off + k < a.max_matches) ? __ldcg(m + k) : 0;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int k = k0 + u;
                if (k < cnt && off + k < a.max_matches) om[off + k] = v[u];
            }
        }
    };
    copy_list(a.seg_matches + ((size_t)b * a.S + s0) * a.max_matches, c0, off0);
    copy_list(a.seg_matches + ((size_t)b * a.S + s1) * a.max_matches, c1, off1);
    for (int k = total + lane; k < a.max_matches; k += 32) om[k] = -1;
    if (lane == 0) a.out_count[b] = total;
    const unsigned h1 = __ballot_sync(0xffffffffu, c1 > 0), h0 = __ballot_sync(0xffffffffu, c0 > 0);
    // the reuse position: the last match of the highest segment with one
    int last = -1;
    if (h1 || h0) {
        const int sl = h1 ? 32 + 31 - __clz(h1) : 31 - __clz(h0);
        last = __ldcg(a.seg_last + (size_t)b * a.S + sl);
    }
    if (od) {
        const int n = a.len[b];
        const int32_t* t = a.tok + (size_t)b * a.n_max;
        for (int k = lane; k < a.L; k += 32)
            od[k] = (last >= 0 && last + 1 + k <= n - 1) ? t[last + 1 + k] : -1;
    }
}

int ngram_segments_max(int n_max) {
    return min(kNgMaxSeg, (n_max + kNgTile - 1) / kNgTile);
}

size_t ngram_workspace_size(int B, int n_max, int max_matches) {
    const size_t segs = (size_t)B * ngram_segments_max(n_max);
    return 256 + align256(sizeof(int32_t) * segs * (size_t)(max_matches + 2));
}

cudaError_t launch_ngram(const int32_t* tokens, const int32_t* lengths, int B, int n_max, int w,
                         int L, int max_matches, int32_t* out_count, int32_t* out_matches,
                         int32_t* out_draft, void* ws, cudaStream_t st) {
    cudaError_t e;
    // one tile per segment up to kNgMaxSeg segments: many short CTAs, whose
    // load latencies overlap
    const int tiles = (n_max + kNgTile - 1) / kNgTile;
    const int smax = ngram_segments_max(n_max);
    const int seg_len = ((tiles + smax - 1) / smax) * kNgTile;
    const int S = (n_max + seg_len - 1) / seg_len;
    char* wsb = static_cast<char*>(ws);
    const size_t segs = (size_t)B * S;
    NgArgs a;
    a.tok = tokens;
    a.len = lengths;
    a.B = B;
    a.n_max = n_max;
    a.w = w;
    a.L = L;
    a.max_matches = max_matches;
    a.S = S;
    a.seg_len = seg_len;
    a.err = reinterpret_cast<int*>(wsb);
    a.seg_count = reinterpret_cast<int32_t*>(wsb + 256);
    a.seg_last = a.seg_count + segs;
    a.seg_matches = a.seg_last + segs;
    a.out_count = out_count;
    a.out_matches = out_matches;
    a.out_draft = out_draft;
    const dim3 grid((unsigned)(B * S));
    switch (w) {
        case 1: e = launch_pdl(ngram_scan_kernel<1>, grid, kNgThreads, 0, st, a); break;
        case 2: e = launch_pdl(ngram_scan_kernel<2>, grid, kNgThreads, 0, st, a); break;
        case 3: e = launch_pdl(ngram_scan_kernel<3>, grid, kNgThreads, 0, st, a); break;
        case 4: e = launch_pdl(ngram_scan_kernel<4>, grid, kNgThreads, 0, st, a); break;
        case 5: e = launch_pdl(ngram_scan_kernel<5>, grid, kNgThreads, 0, st, a); break;
        case 6: e = launch_pdl(ngram_scan_kernel<6>, grid, kNgThreads, 0, st, a); break;
        case 7: e = launch_pdl(ngram_scan_kernel<7>, grid, kNgThreads, 0, st, a); break;
        default: e = launch_pdl(ngram_scan_kernel<8>, grid, kNgThreads, 0, st, a); break;
    }
    if (e != cudaSuccess) return e;
    return launch_pdl(ngram_merge_kernel, dim3((B + kNgMergeWarps - 1) / kNgMergeWarps),
                      kNgMergeWarps * 32, 0, st, a);
}

}  // namespace sv
