/*
 * fp64 CPU oracle for the speculative-decoding verification step.
 *
 * TEST INFRASTRUCTURE ONLY (tests, the smoke check and the benchmark's CPU
 * baseline).  It is written from the definitions on the source pages, in their
 * order and notation, with no blocking or reordering beyond them: every sum is
 * taken in index order with Neumaier compensation, every logit is widened to
 * double first.  It shares nothing with the CUDA library.  The citation keys
 * [SD] and [AdaPLD] are spelled out in oracle.h.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- compensated summation (Neumaier), index order ---------------------- */
typedef struct { double s, c; } ksum_t;

static void ks_add(ksum_t* a, double x) {
    double t = a->s + x;
    if (fabs(a->s) >= fabs(x)) a->c += (a->s - t) + x;
    else a->c += (x - t) + a->s;
    a->s = t;
}
static double ks_val(const ksum_t* a) { return a->s + a->c; }

/* ---- temperature softmax of one row ------------------------------------- */
/* ln p_j = (z_j - m)/T - lnZ with m = max_j z_j and Z = sum_j exp((z_j - m)/T).
 * [SD] "What happens in one round", step 2: the target (and, step 1, the draft)
 * distribution at each position.  A row whose logits are all -inf has no
 * distribution: m = -inf is returned and the caller treats it as bad input. */
typedef struct { double m, lnZ; } rowstat_t;

static rowstat_t row_stats(const float* z, int V, double T) {
    rowstat_t st;
    double m = -INFINITY;
    for (int j = 0; j < V; ++j)
        if ((double)z[j] > m) m = (double)z[j];
    st.m = m;
    st.lnZ = 0.0;
    if (m == -INFINITY) return st;
    ksum_t acc = {0.0, 0.0};
    for (int j = 0; j < V; ++j) ks_add(&acc, exp(((double)z[j] - m) / T));
    st.lnZ = log(ks_val(&acc));
    return st;
}

static double log_prob(const float* z, rowstat_t st, double T, int j) {
    return ((double)z[j] - st.m) / T - st.lnZ;     /* -inf when z_j = -inf */
}

static double prob(const float* z, rowstat_t st, double T, int j) {
    return exp(log_prob(z, st, T, j));
}

/* ---- stochastic verification of one chain ------------------------------ */
static void fill_bad(int32_t* tok, int n, int32_t* acc) {
    for (int i = 0; i < n; ++i) tok[i] = -1;
    *acc = -1;
}

/* Returns 0 on success, 1 on bad input.  w is scratch of V doubles. */
static int verify_one_sample(const float* zt, const float* zd, const int32_t* x, const float* u,
                             double T, int gamma, int V, int32_t* out_tok, int32_t* out_acc,
                             double* out_lp, double* out_ratio, double* out_cdf, double* w,
                             rowstat_t* st_t, rowstat_t* st_d) {
    const size_t V_ = (size_t)V;
    for (int i = 0; i < gamma; ++i)
        if (x[i] < 0 || x[i] >= V) { fill_bad(out_tok, gamma + 1, out_acc); return 1; }

    /* Every position's distribution is computed ([SD] step 2: the target
     * scores the whole draft in one batch). */
    for (int i = 0; i <= gamma; ++i) {
        st_t[i] = row_stats(zt + (size_t)i * V_, V, T);
        if (st_t[i].m == -INFINITY) { fill_bad(out_tok, gamma + 1, out_acc); return 1; }
    }
    for (int i = 0; i < gamma; ++i) {
        st_d[i] = row_stats(zd + (size_t)i * V_, V, T);
        if (st_d[i].m == -INFINITY) { fill_bad(out_tok, gamma + 1, out_acc); return 1; }
    }

    /* [SD] step 3: x_i is accepted with probability min(1, p_i(x_i)/q_i(x_i)),
     * i.e. when u_i < p_i(x_i)/q_i(x_i) for u_i uniform on [0, 1).  p = 0 never
     * accepts; q = 0 < p always accepts. */
    int k = gamma;
    for (int i = 0; i < gamma; ++i) {
        double lp = log_prob(zt + (size_t)i * V_, st_t[i], T, x[i]);
        double lq = log_prob(zd + (size_t)i * V_, st_d[i], T, x[i]);
        double r;
        if (lp == -INFINITY) r = 0.0;
        else if (lq == -INFINITY) r = INFINITY;
        else r = exp(lp - lq);
        if (out_lp) { out_lp[2 * i] = lp; out_lp[2 * i + 1] = lq; }
        if (out_ratio) out_ratio[i] = r;
        if (k == gamma && !((double)u[i] < r)) k = i;   /* first rejection; later drafts void */
    }

    /* [SD] step 4 and "Why fixing wrong guesses ...": after a rejection at
     * position k sample from norm(max(0, p_k - q_k)); if all gamma drafts were
     * accepted sample the bonus token from p_gamma. */
    const float* zp = zt + (size_t)k * V_;
    if (k < gamma) {
        const float* zq = zd + (size_t)k * V_;
        for (int j = 0; j < V; ++j) {
            double p = prob(zp, st_t[k], T, j);
            double q = prob(zq, st_d[k], T, j);
            w[j] = p > q ? p - q : 0.0;
        }
    } else {
        for (int j = 0; j < V; ++j) w[j] = prob(zp, st_t[k], T, j);
    }
    ksum_t tot = {0.0, 0.0};
    for (int j = 0; j < V; ++j) ks_add(&tot, w[j]);
    double S = ks_val(&tot);
    if (!(S > 0.0)) {
        /* The residual has no positive mass (p_k equals q_k to double
         * precision); the rejected position then falls back to p_k itself. */
        tot.s = tot.c = 0.0;
        for (int j = 0; j < V; ++j) { w[j] = prob(zp, st_t[k], T, j); ks_add(&tot, w[j]); }
        S = ks_val(&tot);
    }

    /* Inverse CDF in index order: the token is the first j whose inclusive
     * prefix sum exceeds u_gamma * S.  Zero-mass tokens are never chosen; if
     * rounding leaves u_gamma * S at or above the total, the last token with
     * positive mass is chosen. */
    const double target = (double)u[gamma] * S;
    ksum_t c = {0.0, 0.0};
    int t = -1, last_pos = -1;
    for (int j = 0; j < V; ++j) {
        if (w[j] > 0.0) last_pos = j;
        ks_add(&c, w[j]);
        double Cj = ks_val(&c);
        if (t < 0 && w[j] > 0.0 && Cj > target) t = j;
        if (out_cdf) out_cdf[j] = Cj / S;
    }
    if (t < 0) t = last_pos;

    for (int i = 0; i < k; ++i) out_tok[i] = x[i];
    out_tok[k] = t;
    for (int i = k + 1; i <= gamma; ++i) out_tok[i] = -1;
    *out_acc = k;
    return 0;
}

static int threads_for(int nthreads) {
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

int oracle_verify_sample(const float* target, const float* draft, const int32_t* tokens,
                         const float* uniforms, double T, int B, int gamma, int V,
                         int32_t* out_tokens, int32_t* out_accepted, double* out_logprob,
                         double* out_ratio, double* out_cdf, int nthreads) {
    if (B < 0 || gamma < 0 || V <= 0 || !(T > 0.0) || !isfinite(T)) return -1;
    if (B == 0) return 0;
    if (!target || !uniforms || !out_tokens || !out_accepted) return -1;
    if (gamma > 0 && (!draft || !tokens)) return -1;
    const size_t V_ = (size_t)V;
    int bad = 0;
    int nt = threads_for(nthreads);
#pragma omp parallel num_threads(nt) reduction(+ : bad)
    {
        double* w = (double*)malloc(sizeof(double) * V_);
        rowstat_t* st = (rowstat_t*)malloc(sizeof(rowstat_t) * (size_t)(2 * gamma + 1));
#pragma omp for schedule(dynamic, 1)
        for (int b = 0; b < B; ++b) {
            bad += verify_one_sample(
                target + (size_t)b * (size_t)(gamma + 1) * V_,
                gamma > 0 ? draft + (size_t)b * (size_t)gamma * V_ : NULL,
                gamma > 0 ? tokens + (size_t)b * (size_t)gamma : NULL,
                uniforms + (size_t)b * (size_t)(gamma + 1), T, gamma, V,
                out_tokens + (size_t)b * (size_t)(gamma + 1), out_accepted + b,
                out_logprob ? out_logprob + (size_t)b * (size_t)gamma * 2 : NULL,
                out_ratio ? out_ratio + (size_t)b * (size_t)gamma : NULL,
                out_cdf ? out_cdf + (size_t)b * V_ : NULL, w, st, st + gamma + 1);
        }
        free(st);
        free(w);
    }
    return bad;
}

/* ---- greedy verification ------------------------------------------------- */
/* Row argmax on the raw logits; the lowest index wins among equal values. */
static int argmax_row(const float* z, int V) {
    int best = 0;
    for (int j = 1; j < V; ++j)
        if ((double)z[j] > (double)z[best]) best = j;
    return best;
}

int oracle_verify_greedy(const float* target, const int32_t* tokens, int B, int gamma, int V,
                         int32_t* out_tokens, int32_t* out_accepted, int32_t* out_argmax,
                         int nthreads) {
    if (B < 0 || gamma < 0 || V <= 0) return -1;
    if (B == 0) return 0;
    if (!target || !out_tokens || !out_accepted || (gamma > 0 && !tokens)) return -1;
    const size_t V_ = (size_t)V;
    int bad = 0;
    int nt = threads_for(nthreads);
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1) reduction(+ : bad)
    for (int b = 0; b < B; ++b) {
        const float* zt = target + (size_t)b * (size_t)(gamma + 1) * V_;
        const int32_t* x = gamma > 0 ? tokens + (size_t)b * (size_t)gamma : NULL;
        int32_t* ot = out_tokens + (size_t)b * (size_t)(gamma + 1);
        int ok = 1;
        for (int i = 0; i < gamma; ++i)
            if (x[i] < 0 || x[i] >= V) ok = 0;
        if (!ok) {
            fill_bad(ot, gamma + 1, out_accepted + b);
            if (out_argmax)
                for (int i = 0; i <= gamma; ++i) out_argmax[(size_t)b * (size_t)(gamma + 1) + i] = -1;
            bad += 1;
            continue;
        }
        int k = gamma, gk = -1;
        for (int i = 0; i <= gamma; ++i) {
            int g = argmax_row(zt + (size_t)i * V_, V);
            if (out_argmax) out_argmax[(size_t)b * (size_t)(gamma + 1) + i] = g;
            if (i < k && i < gamma && x[i] != g) { k = i; gk = g; }
            if (i == gamma && k == gamma) gk = g;
        }
        for (int i = 0; i < k; ++i) ot[i] = x[i];
        ot[k] = gk;
        for (int i = k + 1; i <= gamma; ++i) ot[i] = -1;
        out_accepted[b] = k;
    }
    return bad;
}

/* ---- greedy tree verification ------------------------------------------- */
int oracle_verify_tree_greedy(const float* target, const int32_t* tokens, const int32_t* parents,
                              int B, int N, int V, int32_t* out_nodes, int32_t* out_tokens,
                              int32_t* out_accepted, int nthreads) {
    if (B < 0 || N <= 0 || V <= 0) return -1;
    if (B == 0) return 0;
    if (!target || !tokens || !parents || !out_nodes || !out_tokens || !out_accepted) return -1;
    const size_t V_ = (size_t)V, N_ = (size_t)N;
    int bad = 0;
    int nt = threads_for(nthreads);
#pragma omp parallel num_threads(nt) reduction(+ : bad)
    {
        int* g = (int*)malloc(sizeof(int) * N_);
        int* acc = (int*)malloc(sizeof(int) * N_);
        int* depth = (int*)malloc(sizeof(int) * N_);
        int* best = (int*)malloc(sizeof(int) * N_);
#pragma omp for schedule(dynamic, 1)
        for (int b = 0; b < B; ++b) {
            const int32_t* tok = tokens + (size_t)b * N_;
            const int32_t* par = parents + (size_t)b * N_;
            int32_t* on = out_nodes + (size_t)b * N_;
            int32_t* ot = out_tokens + (size_t)b * N_;
            int ok = par[0] == -1;
            for (int n = 1; n < N && ok; ++n)
                if (par[n] < 0 || par[n] >= n || tok[n] < 0 || tok[n] >= V) ok = 0;
            if (!ok) {
                for (int n = 0; n < N; ++n) on[n] = -1;
                fill_bad(ot, N, out_accepted + b);
                bad += 1;
                continue;
            }
            for (int n = 0; n < N; ++n) g[n] = argmax_row(target + ((size_t)b * N_ + (size_t)n) * V_, V);
            /* A node is accepted when its parent is accepted and its token is
             * the target's greedy choice after the parent ([AdaPLD] 3.3: the
             * tree is verified in one target pass; greedy acceptance as in
             * [SD]'s greedy paragraph applied along every root path). */
            acc[0] = 1;
            for (int n = 1; n < N; ++n) acc[n] = acc[par[n]] && tok[n] == g[par[n]];
            /* Longest accepted downward path below each node; children have
             * larger ids than their parent, so one descending sweep finalises
             * every node before its parent reads it.  Among equally long
             * continuations the lower child id wins (visited later). */
            for (int n = 0; n < N; ++n) { depth[n] = 0; best[n] = -1; }
            for (int n = N - 1; n >= 1; --n) {
                if (!acc[n]) continue;
                int p = par[n];
                if (1 + depth[n] >= depth[p]) { depth[p] = 1 + depth[n]; best[p] = n; }
            }
            int len = 0, cur = 0;
            while (best[cur] >= 0) {
                cur = best[cur];
                on[len] = cur;
                ot[len] = tok[cur];
                ++len;
            }
            ot[len] = g[cur];
            for (int n = len; n < N; ++n) on[n] = -1;
            for (int n = len + 1; n < N; ++n) ot[n] = -1;
            out_accepted[b] = len;
        }
        free(best); free(depth); free(acc); free(g);
    }
    return bad;
}

/* ---- top-K branch tokens --------------------------------------------------- */
/* [AdaPLD] 3.3 and Algorithm 1: TopKNextTokens(...) \ {d_main[1]}.  The top K
 * of a row by (larger logit, then lower index): a scan in index order that
 * keeps the best K seen so far, sorted; an element enters only when its logit
 * is strictly larger than the current K-th (so among equal logits the earlier
 * index stays ahead), then the excluded token is dropped from the list. */
int oracle_topk_exclude(const float* logits, const int32_t* exclude, int R, int V, int K,
                        int32_t* out_idx, float* out_val, int nthreads) {
    if (R < 0 || V <= 0 || K <= 0 || K > 64) return -1;
    if (R == 0) return 0;
    if (!logits || !out_idx) return -1;
    int nt = threads_for(nthreads);
#pragma omp parallel for num_threads(nt) schedule(dynamic, 4)
    for (int r = 0; r < R; ++r) {
        const float* z = logits + (size_t)r * (size_t)V;
        int32_t* oi = out_idx + (size_t)r * (size_t)K;
        float* ov = out_val ? out_val + (size_t)r * (size_t)K : NULL;
        int idx[64];
        double val[64];
        int n = 0;                                       /* entries held, <= K */
        for (int j = 0; j < V; ++j) {
            const double x = (double)z[j];
            if (n == K && !(x > val[K - 1])) continue;
            int pos = n < K ? n : K - 1;                 /* slot it takes before sifting up */
            if (n < K) ++n;
            while (pos > 0 && x > val[pos - 1]) {
                val[pos] = val[pos - 1];
                idx[pos] = idx[pos - 1];
                --pos;
            }
            val[pos] = x;
            idx[pos] = j;
        }
        const int ex = exclude ? exclude[r] : -1;
        int o = 0;
        for (int i = 0; i < n; ++i) {
            if (idx[i] == ex) continue;
            oi[o] = idx[i];
            if (ov) ov[o] = (float)val[i];
            ++o;
        }
        for (; o < K; ++o) {
            oi[o] = -1;
            if (ov) ov[o] = -INFINITY;
        }
    }
    return 0;
}

/* ---- lexical (n-gram) retrieval -------------------------------------------- */
/* [AdaPLD] 3.2: the candidates are every earlier position where the most
 * recent token occurs with the preceding tokens matching too (a window of w
 * tokens equal to the query); 3.3: the main draft copies the span after the
 * chosen position.  Plain loops over positions and window offsets. */
int oracle_ngram_retrieve(const int32_t* tokens, const int32_t* lengths, int B, int n_max, int w,
                          int L, int max_matches, int32_t* out_count, int32_t* out_matches,
                          int32_t* out_draft, int nthreads) {
    if (B < 0 || n_max <= 0 || w < 1 || w > 8 || L < 0 || max_matches < 0) return -1;
    if (B == 0) return 0;
    if (!tokens || !lengths || !out_count) return -1;
    int bad = 0;
    int nt = threads_for(nthreads);
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1) reduction(+ : bad)
    for (int b = 0; b < B; ++b) {
        const int32_t* t = tokens + (size_t)b * (size_t)n_max;
        const int n = lengths[b];
        int32_t* om = out_matches ? out_matches + (size_t)b * (size_t)max_matches : NULL;
        int32_t* od = out_draft ? out_draft + (size_t)b * (size_t)L : NULL;
        for (int k = 0; k < max_matches && om; ++k) om[k] = -1;
        for (int k = 0; k < L && od; ++k) od[k] = -1;
        if (n < 1 || n > n_max) {
            out_count[b] = -1;
            bad += 1;
            continue;
        }
        int count = 0, last = -1;
        if (n >= w) {
            const int32_t* q = t + (n - w);               /* the query: the last w tokens */
            for (int p = w - 1; p <= n - 2; ++p) {
                int eq = 1;
                for (int o = 0; o < w; ++o)
                    if (t[p - w + 1 + o] != q[o]) { eq = 0; break; }
                if (!eq) continue;
                if (om && count < max_matches) om[count] = p;
                ++count;
                last = p;
            }
        }
        out_count[b] = count;
        if (od && last >= 0)
            for (int k = 0; k < L && last + 1 + k <= n - 1; ++k) od[k] = t[last + 1 + k];
    }
    return bad;
}
