// Stochastic verification: the two kernels behind spec_verify_sample.
//
// Source: "Speculative decoding: guess a few tokens first - why the answer
// stays the same", section "What happens in one round" (steps 1-4) and section
// "Why fixing wrong guesses does not leave the target distribution" (residual
// p'(x) = norm(max(0, p(x) - q(x)))).
//
// Pass 1 (sample_rowstats_kernel) streams every logit once.  A persistent
// grid walks block chunks (row, segment) of the 2*gamma+1 rows of every
// sequence; each warp reduces its warp chunk to (max m, sum 2^((z - m)
// log2(e)/T)) and writes that pair to the workspace.  Nothing else happens
// in this pass, so it is a pure HBM stream.
//
// Pass 2 (sample_final_kernel) runs one thread-block cluster per sequence.
// Every CTA of the cluster first merges the sequence's partials into row
// statistics and takes the accept decisions left to right (u_i <
// p_i(x_i)/q_i(x_i), in the log domain, in double); all CTAs reach the same
// rejection index k.  The cluster then draws the final token from the single
// row pair it comes from: target and draft row k after a rejection (weights
// max(0, p_k - q_k)), or target row gamma when every draft was accepted
// (weights p_gamma).  Because the token is an inverse CDF over ~10^5 entries,
// both normalisers are recomputed from the very exponentials that form the
// weights, summed in float-float / double and combined across the cluster
// through distributed shared memory; the search walks exactly the prefix sums
// whose totals picked the owning thread.
#include <cooperative_groups.h>

#include "sv_common.cuh"

namespace cg = cooperative_groups;

namespace sv {

constexpr int kMaxGamma = 256;                 // rows per sequence <= 2*256+1
constexpr int kFinalThreads = 512;
constexpr int kFinalStaticSmem = 16384;        // static shared memory reserve of pass 2

struct StatsArgs {
    const char* zt;
    const char* zd;
    float s;            // log2(e) / T
    int gamma, V;
    int nseg;           // block chunks per row
    int rows_per_seq;   // 2 * gamma + 1
    long long total_chunks;
    float2* parts;
};

struct FinalArgs {
    const char* zt;
    const char* zd;
    const int32_t* x;
    const float* u;
    float T, invT, s;
    int B, gamma, V;
    int nseg, rows_per_seq;
    int L;              // elements per CTA slice (multiple of 8)
    const float2* parts;
    int32_t* out_tok;
    int32_t* out_acc;
    float* out_lp;
    int* err;
};

// Row r of sequence b: r <= gamma is target row r, r > gamma is draft row r-gamma-1.
__device__ __forceinline__ const char* seq_row(const char* zt, const char* zd, int gamma, int b,
                                               int r, size_t rowbytes) {
    return r <= gamma ? zt + ((size_t)b * (gamma + 1) + r) * rowbytes
                      : zd + ((size_t)b * gamma + (r - gamma - 1)) * rowbytes;
}

template <int ELT, bool VEC>
__global__ void __launch_bounds__(kThreads) sample_rowstats_kernel(const StatsArgs a) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int WE = 32 * kLaneBytes / ELT;              // elements per warp chunk
    const int P = a.nseg * kWarps;
    const size_t rowbytes = (size_t)a.V * ELT;

    for (long long c = blockIdx.x; c < a.total_chunks; c += gridDim.x) {
        if (c + gridDim.x >= a.total_chunks) pdl_trigger();
        const int seg = (int)(c % a.nseg);
        const long long rr = c / a.nseg;
        const int b = (int)(rr / a.rows_per_seq);
        const int r = (int)(rr % a.rows_per_seq);
        const char* row = seq_row(a.zt, a.zd, a.gamma, b, r, rowbytes);
        const int base = (seg * kWarps + warp) * WE;

        float m = kNegInf, z = 0.f;
        if (base < a.V) {
            LaneChunk<ELT, VEC> ch;
            ch.load(row, a.V, base, lane);
#pragma unroll
            for (int i = 0; i < LaneChunk<ELT, VEC>::EPL; ++i) m = fmaxf(m, ch.val(i));
            m = warp_max(m);
            if (m != kNegInf) {
#pragma unroll
                for (int i = 0; i < LaneChunk<ELT, VEC>::EPL; ++i)
                    z += ex2_approx((ch.val(i) - m) * a.s);
                z = warp_sum(z);
            }
        }
        if (lane == 0) a.parts[(size_t)rr * P + seg * kWarps + warp] = make_float2(m, z);
    }
}

// ---------------------------------------------------------------- pass 2
// exp((z - m) / T) with the argument carried in two floats, so the only
// roundings left are expf's own and the final product.  -inf logits give 0.
template <int ELT>
__device__ __forceinline__ float exp_scaled(float z, float m, float T, float invT) {
    float d_hi, d_lo;
    if constexpr (ELT == 2) {
        d_hi = z - m;                  // exact: both are bfloat16 values
        d_lo = 0.f;
    } else {
        d_hi = z - m;
        const float bb = d_hi - z;
        d_lo = (z - (d_hi - bb)) + (-m - bb);
    }
    if (d_hi == kNegInf) return 0.f;
    const float y = d_hi * invT;
    const float rem = fmaf(-y, T, d_hi) + d_lo;
    const float ylo = rem * invT;
    const float e = expf(y);
    return fmaf(e, ylo, e);
}

__device__ __forceinline__ double block_sum_double(double v, double* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum(v);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    double t = 0.0;
    if (warp == 0) {
        t = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.0;
        t = warp_sum(t);
        if (lane == 0) red[0] = t;
    }
    __syncthreads();
    t = red[0];
    __syncthreads();
    return t;
}

// Inclusive scan of one double per thread (block of kFinalThreads) into incl[].
__device__ __forceinline__ void block_incl_scan_double(double v, double* incl, double* wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    double x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        double w = lane < kFinalThreads / 32 ? wsum[lane] : 0.0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kFinalThreads / 32) wsum[lane] = w;    // inclusive warp totals
    }
    __syncthreads();
    incl[threadIdx.x] = (warp > 0 ? wsum[warp - 1] : 0.0) + x;
    __syncthreads();
}

// Per-thread float-float sum over a contiguous segment [lo, hi) of w.
__device__ __forceinline__ double seg_sum(const float* w, int lo, int hi) {
    FF acc{0.f, 0.f};
    for (int j = lo; j < hi; ++j) ff_add(acc, w[j]);
    return ff_value(acc);
}

struct DecideSmem {
    float M[2 * kMaxGamma + 1];       // row max
    double lnZ[2 * kMaxGamma + 1];    // ln sum exp((z - M)/T)
    double lp[kMaxGamma], lq[kMaxGamma];
    int bad, k;
};

// Row statistics of sequence b from the pass-1 partials and the accept
// decisions.  Identical in every CTA of the cluster (same data, same order).
template <int ELT>
__device__ void sample_decide(const FinalArgs& a, int b, DecideSmem& sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int P = a.nseg * kWarps;
    const size_t rowbytes = (size_t)a.V * ELT;
    if (threadIdx.x == 0) sm.bad = 0;
    __syncthreads();

    // M = max m_p, Z = sum Z_p 2^((m_p - M) s) over the row's warp partials.
    for (int r = warp; r < a.rows_per_seq; r += nwarps) {
        const float2* pr = a.parts + ((size_t)b * a.rows_per_seq + r) * P;
        float m = kNegInf;
        for (int p = lane; p < P; p += 32) m = fmaxf(m, pr[p].x);
        m = warp_max(m);
        double z = 0.0;
        if (m != kNegInf) {
            for (int p = lane; p < P; p += 32) {
                const float2 q = pr[p];
                if (q.x != kNegInf) z += (double)q.y * (double)ex2_approx((q.x - m) * a.s);
            }
        }
        z = warp_sum(z);
        if (lane == 0) {
            sm.M[r] = m;
            sm.lnZ[r] = m == kNegInf ? 0.0 : log(z);
        }
    }
    __syncthreads();

    // Validate the drafts, gather z[x_i] and form ln p_i(x_i), ln q_i(x_i).
    const double invT = 1.0 / (double)a.T;
    for (int i = threadIdx.x; i < a.gamma; i += blockDim.x) {
        const int xi = a.x[(size_t)b * a.gamma + i];
        if (xi < 0 || xi >= a.V) {
            atomicOr(&sm.bad, SPEC_DEVERR_TOKEN_RANGE);
            sm.lp[i] = sm.lq[i] = 0.0;
        } else {
            const float ztx = load_logit<ELT>(seq_row(a.zt, a.zd, a.gamma, b, i, rowbytes), xi);
            const float zdx = load_logit<ELT>(seq_row(a.zt, a.zd, a.gamma, b, a.gamma + 1 + i, rowbytes), xi);
            sm.lp[i] = ((double)ztx - (double)sm.M[i]) * invT - sm.lnZ[i];
            sm.lq[i] = ((double)zdx - (double)sm.M[a.gamma + 1 + i]) * invT - sm.lnZ[a.gamma + 1 + i];
        }
    }
    for (int r = threadIdx.x; r < a.rows_per_seq; r += blockDim.x)
        if (sm.M[r] == kNegInf) atomicOr(&sm.bad, SPEC_DEVERR_EMPTY_ROW);
    __syncthreads();

    if (threadIdx.x == 0) {
        int k = -1;
        if (!sm.bad) {
            // Left to right; the first rejection voids the remaining drafts.
            k = a.gamma;
            for (int i = 0; i < a.gamma; ++i) {
                const double lp = sm.lp[i], lq = sm.lq[i];
                double r;
                if (lp == -CUDART_INF) r = 0.0;
                else if (lq == -CUDART_INF) r = CUDART_INF;
                else r = exp(lp - lq);
                if (!((double)a.u[(size_t)b * (a.gamma + 1) + i] < r)) { k = i; break; }
            }
        }
        sm.k = k;
    }
    __syncthreads();
}

template <int ELT, bool VEC>
__global__ void __launch_bounds__(kFinalThreads) sample_final_kernel(const FinalArgs a) {
    extern __shared__ float4 dyn_smem[];
    float* ea = reinterpret_cast<float*>(dyn_smem);       // exp of target row (weights p)
    float* eb = ea + a.L;                                 // exp of draft row, then residual weights
    __shared__ DecideSmem dsm;
    __shared__ double s_red[32];
    __shared__ double s_incl[kFinalThreads];
    __shared__ double s_wsum[32];
    __shared__ double s_za, s_zb, s_S[2];

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int CS = (int)cluster.num_blocks();
    const int b = blockIdx.y;
    const int tid = threadIdx.x;

    pdl_wait();                                           // pass-1 partials are visible from here
    sample_decide<ELT>(a, b, dsm);
    const int k = dsm.k;
    if (rank == 0) {
        // Accepted drafts, count, padding and log-probabilities; the final
        // slot k is written by the thread that owns the sampled token.
        if (tid == 0) {
            a.out_acc[b] = k;
            if (dsm.bad) atomicOr(a.err, dsm.bad);
        }
        for (int i = tid; i <= a.gamma; i += kFinalThreads)
            if (k < 0 || i != k)
                a.out_tok[(size_t)b * (a.gamma + 1) + i] = (k >= 0 && i < k) ? a.x[(size_t)b * a.gamma + i] : -1;
        if (a.out_lp)
            for (int i = tid; i < a.gamma; i += kFinalThreads) {
                float* o = a.out_lp + ((size_t)b * a.gamma + i) * 2;
                o[0] = k >= 0 ? (float)dsm.lp[i] : CUDART_NAN_F;
                o[1] = k >= 0 ? (float)dsm.lq[i] : CUDART_NAN_F;
            }
    }
    if (k < 0) return;                                    // bad sequence: the whole cluster leaves

    const bool rej = k < a.gamma;
    const float mt = dsm.M[k];
    const float md = rej ? dsm.M[a.gamma + 1 + k] : 0.f;
    const size_t rowbytes = (size_t)a.V * ELT;
    const char* rt = a.zt + ((size_t)b * (a.gamma + 1) + k) * rowbytes;
    const char* rd = rej ? a.zd + ((size_t)b * a.gamma + k) * rowbytes : nullptr;
    const int j0 = rank * a.L;
    const int n = max(0, min(a.V - j0, a.L));

    // Phase A: stage exponentials of the slice and sum them.
    FF sa{0.f, 0.f}, sb{0.f, 0.f};
    int jtail = 0;
    if constexpr (VEC) {
        constexpr int PV = 16 / ELT;
        const int nv = n / PV;                            // n is a multiple of PV except at the row end
        for (int v = tid; v < nv; v += kFinalThreads) {
            const uint4 qt = ld_stream16(rt + (size_t)(j0 + v * PV) * ELT);
            uint4 qd = make_uint4(0, 0, 0, 0);
            if (rej) qd = ld_stream16(rd + (size_t)(j0 + v * PV) * ELT);
#pragma unroll
            for (int e = 0; e < PV; ++e) {
                float zt_, zd_;
                if constexpr (ELT == 4) {
                    zt_ = __uint_as_float(u4_get(qt, e));
                    zd_ = __uint_as_float(u4_get(qd, e));
                } else {
                    const uint32_t wt = u4_get(qt, e >> 1), wd = u4_get(qd, e >> 1);
                    zt_ = __uint_as_float((e & 1) ? (wt & 0xffff0000u) : (wt << 16));
                    zd_ = __uint_as_float((e & 1) ? (wd & 0xffff0000u) : (wd << 16));
                }
                const float et = exp_scaled<ELT>(zt_, mt, a.T, a.invT);
                ea[v * PV + e] = et;
                ff_add(sa, et);
                if (rej) {
                    const float ed = exp_scaled<ELT>(zd_, md, a.T, a.invT);
                    eb[v * PV + e] = ed;
                    ff_add(sb, ed);
                }
            }
        }
        jtail = nv * PV;
    }
    for (int j = jtail + tid; j < n; j += kFinalThreads) {
        const float et = exp_scaled<ELT>(load_logit<ELT>(rt, j0 + j), mt, a.T, a.invT);
        ea[j] = et;
        ff_add(sa, et);
        if (rej) {
            const float ed = exp_scaled<ELT>(load_logit<ELT>(rd, j0 + j), md, a.T, a.invT);
            eb[j] = ed;
            ff_add(sb, ed);
        }
    }
    const double za_part = block_sum_double(ff_value(sa), s_red);
    const double zb_part = rej ? block_sum_double(ff_value(sb), s_red) : 0.0;
    if (tid == 0) { s_za = za_part; s_zb = zb_part; }
    cluster.sync();
    double Za = 0.0, Zb = 0.0;
    for (int r = 0; r < CS; ++r) {                        // same order in every CTA
        Za += *cluster.map_shared_rank(&s_za, r);
        Zb += *cluster.map_shared_rank(&s_zb, r);
    }

    // Phase B: weights.  p_k - q_k scaled by Za is ea - (Za/Zb) eb; the ratio is
    // applied as a float-float pair so the subtraction sees it to ~1e-14.
    float* w = ea;
    if (rej) {
        const double R = Za / Zb;
        const float Rhi = (float)R;
        const float Rlo = (float)(R - (double)Rhi);
        for (int j = tid; j < n; j += kFinalThreads) {
            const float t = fmaf(-Rhi, eb[j], ea[j]);
            eb[j] = fmaxf(fmaf(-Rlo, eb[j], t), 0.f);
        }
        w = eb;
    }
    __syncthreads();

    const int E = (n + kFinalThreads - 1) / kFinalThreads;   // contiguous elements per thread
    const int lo = min(n, tid * E), hi = min(n, lo + E);
    int slot = 0;
    double S = 0.0, P = 0.0;
    for (int attempt = 0; attempt < 2; ++attempt) {
        const double ts = seg_sum(w, lo, hi);
        block_incl_scan_double(ts, s_incl, s_wsum);
        if (tid == 0) s_S[slot] = s_incl[kFinalThreads - 1];
        cluster.sync();
        double acc = 0.0;
        P = 0.0;
        for (int r = 0; r < CS; ++r) {
            const double Sr = *cluster.map_shared_rank(&s_S[slot], r);
            if (r == rank) P = acc;
            acc = acc + Sr;
        }
        S = acc;
        if (S > 0.0 || !rej || attempt == 1) break;
        // No positive residual mass (p_k equals q_k to rounding): fall back to p_k.
        w = ea;
        slot = 1;
    }

    // Inverse CDF: the token is the first j whose prefix sum exceeds u * S.
    // Thread intervals [P + incl(t-1), P + incl(t)) tile [0, S) exactly.
    if (S > 0.0) {
        double target = (double)a.u[(size_t)b * (a.gamma + 1) + a.gamma] * S;
        if (!(target < S)) target = nextafter(S, 0.0);    // u >= 1 clamps to the last token with mass
        const double Bt = P + (tid > 0 ? s_incl[tid - 1] : 0.0);
        const double Et = P + s_incl[tid];
        if (Et > Bt && Bt <= target && target < Et) {
            FF run{0.f, 0.f};
            int pick = -1, last = -1;
            for (int j = lo; j < hi; ++j) {
                ff_add(run, w[j]);
                if (w[j] > 0.f) {
                    last = j;
                    if (pick < 0 && Bt + ff_value(run) > target) pick = j;
                }
            }
            if (pick < 0) pick = last;
            if (pick >= 0) a.out_tok[(size_t)b * (a.gamma + 1) + k] = j0 + pick;
        }
    }
    cluster.sync();                                       // keep shared memory alive for remote readers
}

// ---------------------------------------------------------------- launch
template <int ELT, bool VEC>
static cudaError_t launch_stats_t(const StatsArgs& sa, const DeviceInfo& di, cudaStream_t st) {
    static int occ = 0;                                   // blocks per SM, per template instance
    if (occ == 0) {
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, sample_rowstats_kernel<ELT, VEC>,
                                                          kThreads, 0) != cudaSuccess || o < 1)
            o = 1;
        occ = o;
    }
    long long g = (long long)di.sm_count * occ;
    if (sa.total_chunks < g) g = sa.total_chunks;
    sample_rowstats_kernel<ELT, VEC><<<(int)g, kThreads, 0, st>>>(sa);
    return cudaGetLastError();
}

template <int ELT, bool VEC>
static cudaError_t launch_final_t(const FinalArgs& fa, int CS, size_t smem, bool pdl, cudaStream_t st) {
    auto kfn = sample_final_kernel<ELT, VEC>;
    static size_t smem_set = 0;                           // largest opt-in requested so far
    if (smem > smem_set) {
        cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kfn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        smem_set = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CS, fa.B, 1);
    cfg.blockDim = dim3(kFinalThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kfn, fa);
}

// Cluster size for the final pass: enough CTAs per sequence to fill the GPU
// when B is small, and slices (two float rows each) that fit in shared memory.
static bool final_geometry(int B, int V, const DeviceInfo& di, int* CS_out, int* L_out) {
    const int max_L = (di.max_smem_optin - kFinalStaticSmem) / 8;
    int CS = 1;
    while (CS < 16 && ((long long)CS * max_L < V ||
                       ((long long)CS * B < di.sm_count && V / (CS * 2) >= 4096)))
        CS *= 2;
    int Ls = (V + CS - 1) / CS;
    Ls = (Ls + 7) & ~7;
    if (Ls > max_L) return false;
    *CS_out = CS;
    *L_out = Ls;
    return true;
}

cudaError_t launch_sample(const void* zt, const void* zd, spec_dtype_t dt, const int32_t* x,
                          const float* u, float T, int B, int gamma, int V, int32_t* out_tok,
                          int32_t* out_acc, float* out_lp, void* ws, cudaStream_t st, int parts) {
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int elt = elt_size(dt);
    const bool vec = ((size_t)V * elt) % 16 == 0;
    const WsLayout L = ws_layout(B, gamma, V);
    char* w = static_cast<char*>(ws);
    float2* parts_buf = reinterpret_cast<float2*>(w + L.part_off);
    const float s = (float)(1.4426950408889634 / (double)T);

    if (parts & kSampleStats) {
        StatsArgs sa;
        sa.zt = static_cast<const char*>(zt);
        sa.zd = static_cast<const char*>(zd);
        sa.s = s;
        sa.gamma = gamma;
        sa.V = V;
        sa.nseg = nseg(V, elt);
        sa.rows_per_seq = 2 * gamma + 1;
        sa.total_chunks = (long long)B * sa.rows_per_seq * sa.nseg;
        sa.parts = parts_buf;
        if (elt == 2) e = vec ? launch_stats_t<2, true>(sa, di, st) : launch_stats_t<2, false>(sa, di, st);
        else e = vec ? launch_stats_t<4, true>(sa, di, st) : launch_stats_t<4, false>(sa, di, st);
        if (e != cudaSuccess) return e;
    }
    if (parts & kSampleFinish) {
        int CS = 1, Ls = 0;
        if (!final_geometry(B, V, di, &CS, &Ls)) return cudaErrorInvalidValue;
        FinalArgs fa;
        fa.zt = static_cast<const char*>(zt);
        fa.zd = static_cast<const char*>(zd);
        fa.x = x;
        fa.u = u;
        fa.T = T;
        fa.invT = 1.0f / T;
        fa.s = s;
        fa.B = B;
        fa.gamma = gamma;
        fa.V = V;
        fa.nseg = nseg(V, elt);
        fa.rows_per_seq = 2 * gamma + 1;
        fa.L = Ls;
        fa.parts = parts_buf;
        fa.out_tok = out_tok;
        fa.out_acc = out_acc;
        fa.out_lp = out_lp;
        fa.err = reinterpret_cast<int*>(w + L.err_off);
        const size_t smem = (size_t)Ls * 2 * sizeof(float);
        const bool pdl = (parts & kSampleStats) != 0;     // chained right behind pass 1
        if (elt == 2) e = vec ? launch_final_t<2, true>(fa, CS, smem, pdl, st) : launch_final_t<2, false>(fa, CS, smem, pdl, st);
        else e = vec ? launch_final_t<4, true>(fa, CS, smem, pdl, st) : launch_final_t<4, false>(fa, CS, smem, pdl, st);
    }
    return e;
}

bool sample_supported_vocab(int V) {
    DeviceInfo di;
    if (device_info(&di) != cudaSuccess) return true;     // reported by the launch instead
    int CS, Ls;
    return final_geometry(1, V, di, &CS, &Ls);
}

}  // namespace sv
