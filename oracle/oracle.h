/*
 * fp64 CPU oracle for the speculative-decoding verification step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this code: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * Sources (the pages this restates):
 *   [SD]    "Speculative decoding: guess a few tokens first - why the answer
 *           stays the same" (explainer blog).  Section "What happens in one
 *           round" (the four steps), section "Why fixing wrong guesses does
 *           not leave the target distribution" (the min(p,q) identity and the
 *           residual p'(x) = norm(max(0, p(x) - q(x)))), and its paragraph on
 *           greedy decoding (accept while the draft equals the target argmax).
 *   [AdaPLD] "AdaPLD: adaptive retrieval and reuse for efficient model-free
 *           speculative decoding", section 3.3 "Tree construction and
 *           verification" and Algorithm 1 (BuildDraftTree, VerifyAndAccept).
 *
 * Logits are float32 arrays (bfloat16 inputs are passed as their exact float32
 * values); every value is widened to double before any arithmetic.
 *
 * Return value of every call: the number of sequences rejected as bad input
 * (those get num_accepted = -1 and all output tokens -1), or -1 when the
 * arguments themselves are invalid.
 */
#ifndef SPEC_ORACLE_H
#define SPEC_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Stochastic verification of B independent draft chains ([SD] "What happens
 * in one round" steps 1-4).
 *   target   [B, gamma+1, V]  target-model logits z^t
 *   draft    [B, gamma,   V]  draft-model logits z^d (may be NULL if gamma == 0)
 *   tokens   [B, gamma]       drafted tokens x_0..x_{gamma-1}
 *   uniforms [B, gamma+1]     u_0..u_{gamma-1} decide acceptance, u_gamma drives
 *                             the one final (residual or bonus) sample
 *   T                         temperature (> 0) applied to both models
 * Outputs:
 *   out_tokens   [B, gamma+1] accepted drafts, then the final token, then -1
 *   out_accepted [B]          number of accepted drafts k (0..gamma)
 *   out_logprob  [B, gamma, 2] (nullable) ln p_i(x_i), ln q_i(x_i)
 *   out_ratio    [B, gamma]   (nullable) p_i(x_i)/q_i(x_i) for every position
 *   out_cdf      [B, V]       (nullable) normalised inclusive CDF C_j / S of the
 *                             distribution the final token was drawn from
 *   nthreads                  OpenMP threads over sequences (<= 0: default)
 */
int oracle_verify_sample(const float* target, const float* draft, const int32_t* tokens,
                         const float* uniforms, double T, int B, int gamma, int V,
                         int32_t* out_tokens, int32_t* out_accepted, double* out_logprob,
                         double* out_ratio, double* out_cdf, int nthreads);

/*
 * Greedy verification ([SD], greedy paragraph): accept x_i while it equals the
 * argmax of target row i (lowest index among equal logits); at the first
 * mismatch emit the target argmax; if all match emit the argmax of row gamma.
 *   out_argmax [B, gamma+1] (nullable): the per-row argmax.
 */
int oracle_verify_greedy(const float* target, const int32_t* tokens, int B, int gamma, int V,
                         int32_t* out_tokens, int32_t* out_accepted, int32_t* out_argmax,
                         int nthreads);

/*
 * Greedy verification of a draft tree ([AdaPLD] 3.3, Algorithm 1 VerifyAndAccept).
 *   target  [B, N, V]  target logits of every tree node (node 0 is the root)
 *   tokens  [B, N]     drafted token of each node (node 0 ignored)
 *   parents [B, N]     parents[0] = -1, 0 <= parents[n] < n for n >= 1
 * A node is accepted when its parent is accepted and its token equals the
 * argmax of its parent's row; the root is accepted.  The result is the longest
 * root path of accepted nodes (ties: lexicographically smallest node ids)
 * plus the bonus token argmax(row of the path's last node).
 *   out_nodes    [B, N] path node ids (root excluded), then -1
 *   out_tokens   [B, N] path tokens, then the bonus token, then -1
 *   out_accepted [B]    path length
 */
int oracle_verify_tree_greedy(const float* target, const int32_t* tokens, const int32_t* parents,
                              int B, int N, int V, int32_t* out_nodes, int32_t* out_tokens,
                              int32_t* out_accepted, int nthreads);

/*
 * Branch tokens of a draft tree ([AdaPLD] 3.3, "strict hit path", and
 * Algorithm 1, TopKNextTokens(M, x_{<=p*}, K) \ {d_main[1]}): for each of R
 * rows of V logits, the K tokens with the largest logits (larger logit first,
 * lower index first among equal logits, -0.0 equal to +0.0), then the row's
 * excluded token removed from that list if it is in it.  The list keeps its
 * order and is padded with -1 at the end (value -inf); it is also padded when
 * V < K.
 *   logits   [R, V]
 *   exclude  [R] (nullable: no exclusion); -1 excludes nothing
 *   out_idx  [R, K]
 *   out_val  [R, K] (nullable) the logits of out_idx
 * K is at most 64.
 */
int oracle_topk_exclude(const float* logits, const int32_t* exclude, int R, int V, int K,
                        int32_t* out_idx, float* out_val, int nthreads);

/*
 * Lexical retrieval of a reuse position ([AdaPLD] 3.2 "lexical retrieval
 * stage", 3.3 "strict hit path", Algorithm 1 LexicalRetrieval and d_main).
 * Sequence b's context is tokens[b, 0..len[b]-1]; its query is its last w
 * tokens.  A match is a position p <= len[b]-2 whose window
 * tokens[p-w+1..p] equals the query (p >= w-1).
 *   tokens      [B, n_max] int32 context streams (entries past len[b] ignored)
 *   lengths     [B] context lengths, 1..n_max
 *   out_count   [B] number of matches
 *   out_matches [B, max_matches] the first max_matches match positions in
 *               ascending order, then -1
 *   out_draft   [B, L] the continuation after the most recent match p*:
 *               tokens[p*+1 .. min(p*+L, len[b]-1)], then -1 (all -1 when
 *               there is no match)
 * 1 <= w <= 8.
 */
int oracle_ngram_retrieve(const int32_t* tokens, const int32_t* lengths, int B, int n_max, int w,
                          int L, int max_matches, int32_t* out_count, int32_t* out_matches,
                          int32_t* out_draft, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
