/*
 * spec_verify.h - C ABI of the GB300 (sm_103a) speculative-decoding
 * verification library (libspecverify.so).
 *
 * The operation is the target-model verification step of speculative
 * decoding as defined in:
 *   [SD]     "Speculative decoding: guess a few tokens first - why the answer
 *            stays the same" (explainer blog).  Section "What happens in one
 *            round": the target scores all gamma drafts (plus one position)
 *            in one batch, drafts are checked left to right and accepted with
 *            probability min(1, p_i(x_i)/q_i(x_i)), the first rejection voids
 *            the rest and is replaced by a sample from the residual; when all
 *            drafts are accepted a bonus token is sampled from the next
 *            position.  Section "Why fixing wrong guesses does not leave the
 *            target distribution": residual p'(x) = norm(max(0, p(x) - q(x))).
 *            The greedy paragraph: accept while the draft equals the target
 *            argmax, replace the first mismatch by the target token.
 *   [AdaPLD] "AdaPLD: adaptive retrieval and reuse for efficient model-free
 *            speculative decoding", section 3.3 "Tree construction and
 *            verification" and Algorithm 1 (BuildDraftTree / VerifyAndAccept):
 *            a draft tree (main chain plus top-K branches) verified by the
 *            target in one pass.
 *
 * Conventions shared by every call
 *   - Every pointer is a DEVICE pointer owned by the caller; the library never
 *     allocates and keeps no per-call state.  Calls are asynchronous on
 *     `stream`; results are valid once the stream reaches them.  The
 *     library's kernels are launched with programmatic dependent launch: a
 *     call's first kernel may start while the kernel before it on `stream`
 *     finishes, and may then prefetch logits into L2, but it reads the
 *     inputs and the workspace only after that kernel has completed.  Inputs
 *     written by the kernel just before the call on the same stream are
 *     therefore read as written.
 *   - Logits are row-major with V contiguous, dtype SPEC_DTYPE_F32 or
 *     SPEC_DTYPE_BF16.  Logit base pointers must be 16-byte aligned
 *     (SPEC_ERR_MISALIGNED otherwise).  V need not be a multiple of anything.
 *     -inf logits are legal (masked tokens); NaN/+inf logits are undefined.
 *   - `workspace` is caller-owned device scratch of at least
 *     spec_verify_workspace_size() bytes, 256-byte aligned.  Its first 4
 *     bytes are the device error word (below): zero-fill the workspace once
 *     (spec_verify_workspace_init) so that word starts clear.  Everything
 *     else in it is rewritten by each call before it is read, so one
 *     workspace serves calls of any mode and size in turn.  Calls that share
 *     a workspace must be ordered on the device (same stream, or events);
 *     overlapping calls on one workspace race.
 *   - Host-side argument checks return immediately without touching the
 *     device.  Bad input that only the device can see (a draft token outside
 *     [0, V), a row with every logit -inf, a malformed tree) marks that
 *     sequence with num_accepted = -1 and every output token -1, and sets a
 *     bit in the workspace error word (see spec_verify_read_error).
 *   - B = 0 is an empty batch: SPEC_OK, nothing is launched.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1,          /* null pointer, negative size, bad temperature */
    SPEC_ERR_UNSUPPORTED_DTYPE = 2,
    SPEC_ERR_MISALIGNED = 3,           /* logits or workspace not aligned as required */
    SPEC_ERR_WORKSPACE_TOO_SMALL = 4,
    SPEC_ERR_CUDA = 5,                 /* a CUDA runtime call or launch failed */
    SPEC_ERR_DEVICE_INPUT = 6,         /* reported by spec_verify_read_error only */
    SPEC_ERR_EXCEEDS_STATIC_SCRATCH = 7 /* spec_verify_sample_noalloc: the problem needs more than
                                           SPEC_VERIFY_NOALLOC_SCRATCH_BYTES of scratch */
} spec_status_t;

typedef enum { SPEC_DTYPE_F32 = 0, SPEC_DTYPE_BF16 = 1 } spec_dtype_t;

/* Bits of the device error word. */
#define SPEC_DEVERR_TOKEN_RANGE  1   /* a draft / node token outside [0, V) */
#define SPEC_DEVERR_EMPTY_ROW    2   /* a logits row whose every entry is -inf (sampling) */
#define SPEC_DEVERR_TREE_PARENT  4   /* parents[0] != -1 or parents[n] not in [0, n) */
#define SPEC_DEVERR_TIMEOUT      8   /* a bounded wait inside a kernel ran out (internal error;
                                        the affected results are not valid) */

/*
 * Bytes of workspace any of the three verification calls needs for B
 * sequences of `gamma_or_nodes` drafts (chains) or nodes (trees) over a
 * vocabulary of V, for either dtype.  Returns 0 for invalid sizes.
 */
size_t spec_verify_workspace_size(int B, int gamma_or_nodes, int V);

/* Zero-fills a workspace (cudaMemsetAsync on `stream`). */
spec_status_t spec_verify_workspace_init(void* workspace, size_t workspace_bytes,
                                         cudaStream_t stream);

/*
 * Stochastic verification of B independent draft chains ([SD] "What happens in
 * one round", steps 1-4, and the residual of "Why fixing wrong guesses ...").
 *
 *   target_logits [B, gamma+1, V]  target logits z^t; row i scores position i
 *   draft_logits  [B, gamma, V]    draft logits z^d (NULL allowed if gamma == 0)
 *   draft_tokens  [B, gamma] int32 drafted tokens x_0..x_{gamma-1}
 *   uniforms      [B, gamma+1] f32 in [0, 1): u_i decides draft i (accepted iff
 *                                  u_i < p_i(x_i)/q_i(x_i)); u_gamma drives the
 *                                  single final sample (residual or bonus) by
 *                                  inverse CDF in index order
 *   temperature   finite, >= 1e-20; p = softmax(z^t / T), q = softmax(z^d / T)
 *   0 <= gamma <= 256, 1 <= V <= 2097152, B >= 0.  (The final sample scans
 *   the 8192-element chunk totals of a row in one 256-thread CTA, hence the
 *   bound on V; larger V returns SPEC_ERR_INVALID_ARG.)
 * Outputs (device):
 *   out_tokens       [B, gamma+1] int32: the k accepted drafts, the final
 *                    token, then -1
 *   out_num_accepted [B] int32: k in [0, gamma] (emitted tokens = k + 1)
 *   out_logprobs     [B, gamma, 2] f32, nullable: ln p_i(x_i), ln q_i(x_i)
 *
 * A streaming pass over every logit row (row max and sum-exp partials) is
 * followed by two kernels: the accept decisions, then the chunk sums of the
 * exponentials and of the residual weights of the one rejected (or bonus)
 * row pair, in which the last chunk of each sequence to finish runs the
 * inverse-CDF search.
 */
spec_status_t spec_verify_sample(const void* target_logits, const void* draft_logits,
                                 spec_dtype_t dtype, const int32_t* draft_tokens,
                                 const float* uniforms, float temperature, int B, int gamma,
                                 int V, int32_t* out_tokens, int32_t* out_num_accepted,
                                 float* out_logprobs, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/*
 * Lazy (early-exit) stochastic verification ([SD] "What happens in one
 * round", step 3: the first rejection discards every later draft, so a
 * position's rows are only needed while every earlier draft was accepted).
 * Same arguments, workspace and outputs as spec_verify_sample, with the same
 * tokens and accept counts.  The positions are streamed in groups of
 * doubling size -- [0, 2), [2, 6), [6, 14), ... -- each group one pass over
 * the GPU for the sequences whose drafts before it were all accepted, so
 * after a rejection at k only the rows of the groups up to k's are read (at
 * most positions 0..2k+1), all 2 gamma + 1 rows when every draft is
 * accepted.  A group runs on to the end (at most 128 positions) when the
 * rows after it, for all B sequences, hold fewer than 96 MB: a pass then
 * costs more than it can save.  spec_verify_set_lazy_split_bytes, or the
 * environment variable SPEC_VERIFY_LAZY_SPLIT_BYTES read once at the first
 * lazy call or groups query of the process, overrides that figure (0: split
 * at every boundary); the outputs do not depend on it.  out_logprobs (nullable)
 * holds the log-probabilities of positions 0..min(k, gamma - 1); later
 * positions, and every position of a bad sequence, are NaN.  Rows whose
 * byte length is not a multiple of 16 take the full pass (every row read)
 * with the same outputs.  Device-side bad-input detection covers the rows
 * decided: positions 0..k.
 */
spec_status_t spec_verify_sample_lazy(const void* target_logits, const void* draft_logits,
                                      spec_dtype_t dtype, const int32_t* draft_tokens,
                                      const float* uniforms, float temperature, int B, int gamma,
                                      int V, int32_t* out_tokens, int32_t* out_num_accepted,
                                      float* out_logprobs, void* workspace, size_t workspace_bytes,
                                      cudaStream_t stream);

/*
 * The position groups that spec_verify_sample_lazy streams for B sequences of
 * gamma drafts over V logits of the given dtype ([SD] "What happens in one
 * round", step 3, read as in spec_verify_sample_lazy): writes the groups'
 * upper ends, exclusive, to ends[0 .. count) in ascending order (group g
 * covers positions ends[g-1] .. ends[g]-1, from 0; the last end is gamma + 1)
 * and returns count, at most 8.  The sizes double from 2 -- [0,2), [2,6),
 * [6,14), ... -- and a group runs on to the end (at most 128 positions) when
 * the rows after it, for all B sequences, hold fewer than 96 MB (or the
 * figure set as described for spec_verify_sample_lazy).  Host only, no CUDA
 * call; returns 0 for invalid arguments (B < 1, gamma outside 0..256, V < 1,
 * an unknown dtype, ends NULL).  ends must hold 8 entries.  The groups of a
 * lazy call are those this function returns with the same figure in force.
 */
int spec_verify_lazy_groups(int B, int gamma, int V, spec_dtype_t dtype, int32_t* ends);

/*
 * Sets the figure of spec_verify_sample_lazy's group rule: a group runs on to
 * the end when the rows after it hold fewer than `bytes` (0: split at every
 * boundary; negative: back to the built-in 96 MB).  Process-wide, for calls
 * and queries made afterwards from any thread; it replaces the value of
 * SPEC_VERIFY_LAZY_SPLIT_BYTES.  Host only.
 */
void spec_verify_set_lazy_split_bytes(double bytes);

/*
 * The two halves of spec_verify_sample, for callers that want to overlap or
 * time them separately; spec_verify_sample is exactly _stats then _finish on
 * the same stream with the same arguments and workspace.
 *   _stats:  streams every logit row once and leaves per-row partial
 *            statistics (running max and sum of exponentials) in the
 *            workspace.  Writes no output.
 *   _finish: takes the accept decisions from those statistics and draws the
 *            final token of every sequence (residual after a rejection, bonus
 *            otherwise); writes every output of spec_verify_sample.
 * The workspace and the logits must stay unchanged between the two calls.
 */
spec_status_t spec_verify_sample_stats(const void* target_logits, const void* draft_logits,
                                       spec_dtype_t dtype, float temperature, int B, int gamma,
                                       int V, void* workspace, size_t workspace_bytes,
                                       cudaStream_t stream);
spec_status_t spec_verify_sample_finish(const void* target_logits, const void* draft_logits,
                                        spec_dtype_t dtype, const int32_t* draft_tokens,
                                        const float* uniforms, float temperature, int B,
                                        int gamma, int V, int32_t* out_tokens,
                                        int32_t* out_num_accepted, float* out_logprobs,
                                        void* workspace, size_t workspace_bytes,
                                        cudaStream_t stream);

/*
 * Greedy verification ([SD] greedy paragraph): g_i = argmax_j z^t[b,i,j]
 * (lowest index among equal logits), k = first i with x_i != g_i, else gamma.
 * Draft logits are not needed.
 *   target_logits [B, gamma+1, V], draft_tokens [B, gamma] (NULL if gamma == 0)
 *   out_tokens [B, gamma+1]: x_0..x_{k-1}, g_k, then -1;  out_num_accepted [B]: k
 */
spec_status_t spec_verify_greedy(const void* target_logits, spec_dtype_t dtype,
                                 const int32_t* draft_tokens, int B, int gamma, int V,
                                 int32_t* out_tokens, int32_t* out_num_accepted, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream);

/*
 * Greedy verification of a draft tree ([AdaPLD] 3.3, Algorithm 1).
 *   target_logits [B, N, V]: row n scores the continuation after node n
 *   node_tokens   [B, N] int32: token of node n (node 0, the root, is ignored)
 *   parents       [B, N] int32: parents[0] = -1, 0 <= parents[n] < n
 * A node is accepted when its parent is accepted and its token equals the
 * argmax of the parent's row (the root is accepted).  Result: the longest
 * root path of accepted nodes (ties: lexicographically smallest node ids) and
 * the bonus token argmax(row of the path's last node).
 *   out_path_nodes   [B, N]: path node ids (root excluded), then -1
 *   out_tokens       [B, N]: path tokens, then the bonus token, then -1
 *   out_num_accepted [B]: path length
 */
spec_status_t spec_verify_tree_greedy(const void* target_logits, spec_dtype_t dtype,
                                      const int32_t* node_tokens, const int32_t* parents, int B,
                                      int N, int V, int32_t* out_path_nodes, int32_t* out_tokens,
                                      int32_t* out_num_accepted, void* workspace,
                                      size_t workspace_bytes, cudaStream_t stream);

/*
 * Branch tokens of a draft tree ([AdaPLD] 3.3 "strict hit path" and
 * Algorithm 1: TopKNextTokens(M, x_{<=p*}, K) \ {d_main[1]}): for each of
 * `rows` rows of V logits, the K tokens with the largest logits (larger logit
 * first, lower index first among equal logits, -0.0 equal to +0.0), then the
 * row's excluded token removed from that list when it is in it.  The list
 * keeps its order and is padded with -1 (value -inf), also when V < K.
 *   logits   [rows, V], row-major, 16-byte aligned, bf16 or fp32; -inf
 *            (masked) logits are ordinary values, NaN is undefined
 *   exclude  [rows] int32 (NULL: no exclusion); -1, or any value outside
 *            [0, V), excludes nothing
 *   out_idx  [rows, K] int32
 *   out_val  [rows, K] float (NULL: not written): the logits of out_idx
 * 1 <= K <= 8.  Workspace: spec_topk_workspace_size(rows, V, K) bytes,
 * 256-byte aligned, its first 256 bytes zero-filled once (the error word, as
 * for the verification calls); nothing else is carried between calls.
 */
size_t spec_topk_workspace_size(int rows, int V, int K);
spec_status_t spec_topk_exclude(const void* logits, spec_dtype_t dtype, int rows, int V, int K,
                                const int32_t* exclude, int32_t* out_idx, float* out_val,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Lexical retrieval of a reuse position ([AdaPLD] 3.2 "lexical retrieval
 * stage", 3.3 "strict hit path", Algorithm 1 LexicalRetrieval and d_main):
 * sequence b's context is tokens[b, 0 .. lengths[b]-1] and its query its last
 * w tokens.  A match is a position p with w-1 <= p <= lengths[b]-2 whose
 * window tokens[b, p-w+1 .. p] equals the query.  The pages choose among the
 * matches by hidden-state similarity; here the most recent match p* is the
 * reuse position.
 *   tokens      [B, n_max] int32, 16-byte aligned, n_max a multiple of 4;
 *               entries at or past lengths[b] are ignored
 *   lengths     [B] int32 in 1..n_max (device); another value marks the
 *               sequence bad: out_count -1, every output -1, error bit
 *               SPEC_DEVERR_TOKEN_RANGE
 *   out_count   [B]: number of matches
 *   out_matches [B, max_matches]: the first max_matches match positions in
 *               ascending order, then -1
 *   out_draft   [B, L] (NULL: not written): tokens[b, p*+1 .. min(p*+L,
 *               lengths[b]-1)], then -1; all -1 without a match
 * 1 <= w <= 8, 0 <= L <= 1024, 1 <= max_matches <= 4096.  Workspace:
 * spec_ngram_workspace_size(B, n_max, max_matches) bytes, 256-byte aligned,
 * first 256 bytes zero-filled once (the error word).
 */
size_t spec_ngram_workspace_size(int B, int n_max, int max_matches);
spec_status_t spec_ngram_retrieve(const int32_t* tokens, const int32_t* lengths, int B, int n_max,
                                  int w, int L, int max_matches, int32_t* out_count,
                                  int32_t* out_matches, int32_t* out_draft, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream);

/*
 * Semantic fallback of the reuse-position search ([AdaPLD] 3.2 "semantic
 * fallback stage", Algorithm 1 SemanticFallback): for each sequence b,
 * score(j) = h . H_j / (|h| |H_j|) over its window of W hidden states (the
 * states of the most recent forward steps), then the delta largest scores,
 * larger first, lower window index first among equal scores.  A zero norm
 * gives score 0.  Scores are accumulated in fp32 (|error| ~1e-6).
 *   hidden     [B, W, d] bf16 or fp32, 16-byte aligned, d a multiple of 8
 *              (bf16) or 4 (fp32)
 *   query      [B, d] same dtype, 16-byte aligned
 *   positions  [B, W] int32 (NULL: the window index): the context position of
 *              each window row
 *   out_idx    [B, delta] window rows, -1 padded when W < delta
 *   out_pos    [B, delta] (NULL: not written) their positions, -1 padded
 *   out_score  [B, delta] (NULL: not written) their scores, -inf padded
 * 1 <= delta <= 8, W >= 1.  Workspace: spec_cosine_workspace_size(B, W)
 * bytes, 256-byte aligned.
 */
size_t spec_cosine_workspace_size(int B, int W);
spec_status_t spec_cosine_topk(const void* hidden, const void* query, spec_dtype_t dtype, int B,
                               int W, int d, int delta, const int32_t* positions,
                               int32_t* out_idx, int32_t* out_pos, float* out_score,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * spec_verify_sample for callers that cannot allocate device memory.
 *
 * The source pages have no counterpart to this call; it exists for callers
 * that cannot provide a workspace: a plugin whose host framework owns all
 * device memory in its own pool and passes in only input and output buffers,
 * or a decode loop that must not call cudaMalloc/cudaFree (which can
 * synchronise the device) in the middle of a step.  Arguments, outputs and
 * results are those of spec_verify_sample without the workspace; the same
 * kernels run.  The call allocates nothing and calls no allocating routine.
 *
 * Scratch: a fixed array of SPEC_VERIFY_NOALLOC_SCRATCH_BYTES (8 MiB) that the
 * library places in the device memory of every GPU it is loaded on, held
 * until the process exits.  Problems whose scratch need,
 * spec_verify_workspace_size(B, gamma, V), exceeds it are rejected with
 * SPEC_ERR_EXCEEDS_STATIC_SCRATCH before anything is launched (B = 256
 * sequences of 4 drafts over 128256 fp32 logits need 6.8 MB).
 *
 * The first call on each device, made while that device is current, looks up
 * the array's device address (cudaGetSymbolAddress, which may also load the
 * library's kernels onto that device); make that first call before any stream
 * capture.  The address is kept for the life of the process: after
 * cudaDeviceReset (or any other reset of the device's primary context) in the
 * same process, this entry point must not be called again on that device.  Every call on a device shares the one array, so calls whose work
 * overlaps on the GPU (different streams without ordering, or host threads
 * racing on one device) race on it and give undefined results; order them.
 * Bad input is reported per sequence (num_accepted = -1, tokens -1) only: the
 * device error word of the workspace calls is not readable for this entry.
 */
#define SPEC_VERIFY_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
spec_status_t spec_verify_sample_noalloc(const void* target_logits, const void* draft_logits,
                                         spec_dtype_t dtype, const int32_t* draft_tokens,
                                         const float* uniforms, float temperature, int B,
                                         int gamma, int V, int32_t* out_tokens,
                                         int32_t* out_num_accepted, float* out_logprobs,
                                         cudaStream_t stream);

/*
 * Test hook for the kernels' bounded waits (the source pages have no
 * counterpart).  Every wait of the streaming kernels on a shared-memory
 * barrier of their bulk-copy ring gives up after a number of polls (seconds of
 * wall time by default: spec_verify_default_wait_limit()), sets
 * SPEC_DEVERR_TIMEOUT in the workspace error word and lets the kernel return
 * instead of hanging.  spec_verify_set_wait_limit sets that number for every
 * launch made afterwards in the process, from any thread; 0 makes such waits
 * give up without polling, so a test can drive the timeout path without
 * breaking a kernel.  Results of a call whose wait gave up are not valid; the
 * workspace stays usable for later calls.  A kernel's final wait for its own
 * bulk copies in flight always keeps the default bound.  Host only; set it
 * back to the default after the test.
 */
void spec_verify_set_wait_limit(uint32_t polls);
uint32_t spec_verify_default_wait_limit(void);

/*
 * Synchronises `stream`, returns the accumulated SPEC_DEVERR_* bits of the
 * workspace in *code and clears them.  SPEC_OK when the read succeeded (code
 * may still be nonzero).
 */
spec_status_t spec_verify_read_error(void* workspace, cudaStream_t stream, int32_t* code);

/* Static description of a status code. */
const char* spec_verify_status_string(spec_status_t status);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
