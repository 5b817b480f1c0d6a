/*
 * tsv.h -- C ABI of libtsv, the GB300 (sm_103a) target-side verification step of
 * tree-based speculative decoding.
 *
 * One verification step is three calls on one CUDA stream, with no host
 * synchronisation between them:
 *   1. tsv_tree_verify_attn    -- attention of the flattened draft tree over the
 *                                 paged KV cache under the ancestor-only tree mask;
 *   2. tsv_tree_reject_sample  -- rejection-sampling walk of the tree (Sequoia-style
 *                                 sampling without replacement) plus a bonus token;
 *   3. tsv_kv_compact_accepted -- KV-cache rewrite of the accepted path
 *      (tsv_tree_reject_sample_compact runs 2 and 3 in one launch).
 * (Step 2 consumes target logits, which in a full model are produced from step
 * 1's output by the layers above attention; the library takes them as input.)
 *
 * Conventions for every entry point
 *  - All array pointers are caller-owned DEVICE memory on the current device,
 *    except where a comment says otherwise.  The library allocates no device
 *    memory and keeps no state between calls; calls are thread-safe.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default).
 *  - Host-side argument errors return TSV_ERR_ARG / TSV_ERR_UNSUPPORTED at once and
 *    launch nothing.  A failed launch returns TSV_ERR_CUDA.  tsv_last_error()
 *    gives a message for the calling thread's last failure.
 *  - Data errors found on the device never trap: they are written as bit masks to
 *    `seq_err[b]` (one int32 per sequence, overwritten by each call) and the
 *    sequence's outputs are poisoned as documented per call.
 *  - Layouts are row-major:  q/out [B, N, Hq, D];  caches [num_blocks, block_size,
 *    Hkv, D];  block_table [B, max_blocks];  seq_lens/ new_seq_lens [B];  parent,
 *    draft_tokens, u_accept, accepted_nodes, out_tokens [B, N];  target_logits,
 *    draft_probs [B, N, V];  u_bonus, accept_len, bonus_token, seq_err [B].
 *  - Logical slot t of sequence b lives at physical row
 *    block_table[b, t / block_size] * block_size + t % block_size of the caches.
 *
 * The tree (sglang report "Speculative decoding on sglang", sections "What is
 * Tree-Attention?" and "Tree-based Speculative Decoding (EAGLE) Implementation
 * Summary": draft candidates flattened to 1-D, verified in one pass under a tree
 * mask) is given per sequence as parent[b, i]: node 0 is the root, i.e. the last
 * accepted token (parent -1), and 0 <= parent[i] < i for i >= 1.  Node i's K/V is
 * already in the cache at logical slot seq_lens[b] + i (written by the caller's
 * projection, as serving engines do); the caller preallocates the blocks, so
 * seq_lens[b] + N <= max_blocks * block_size ("preallocated slots", vLLM PR #2188,
 * "Guide for reviewers").
 */
#ifndef TSV_H
#define TSV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TSV_OK = 0,
    TSV_ERR_ARG = 1,         /* null pointer, bad size, workspace too small */
    TSV_ERR_UNSUPPORTED = 2, /* valid but not built: e.g. D not in {64, 128} */
    TSV_ERR_CUDA = 3         /* a CUDA runtime/driver call or launch failed */
} tsv_status;

typedef enum { TSV_BF16 = 0, TSV_F32 = 1 } tsv_dtype;

/* Device-side data error bits written to seq_err[b]. */
enum {
    TSV_DERR_PARENT = 1,    /* parent array (or accepted path) is not a valid tree/path */
    TSV_DERR_BLOCK = 2,     /* a block id covering slots [0, L_b + N) is outside [0, num_blocks) */
    TSV_DERR_CAPACITY = 4,  /* L_b < 0 or L_b + N > max_blocks * block_size */
    TSV_DERR_TOKEN = 8,     /* a tried draft token is outside [0, V) */
    TSV_DERR_NONFINITE = 16, /* a visited logits row, or a draft row that is read, is not finite */
    TSV_DERR_TIMEOUT = 32,   /* internal: a bounded device-side wait gave up; outputs of the
                                sequence are not valid (never expected; reported, not trapped) */
    TSV_DERR_INTERNAL = 64   /* checked builds only (-DTSV_CHECKED, a test build): a device-side
                                index check failed and the access was skipped -- a library bug */
};

/* Message for the calling thread's most recent failed call ("" if none). */
const char *tsv_last_error(void);

/* ---------------------------------------------------------------------------
 * Tree-masked GQA attention (sglang report, "What is Tree-Attention?"; the EAGLE
 * "Tree Decoding" step with attention_mask + tree_attention_mask).
 *
 * For query row (b, n, h), kv head g = h / (Hq / Hkv):
 *   keys = prefix slots 0 .. L_b-1  (all visible)
 *        + tree slots L_b + j for every node j on the root-to-n path, n included;
 *   out[b,n,h,:] = softmax_t(scale * q[b,n,h,:] . k[t,g,:]) @ v[t,g,:].
 * q, caches and out share `dtype` (bf16: tensor-core tiles, fp32 accumulation;
 * fp32: exact fp32 FMA path).  D in {64, 128}; 1 <= N <= 128; Hq % Hkv == 0;
 * block_size a power of two in [8, 128].
 * bf16: persistent CTAs split the 128-key tiles of all (sequence, kv head) pairs
 * evenly; a pair that straddles CTAs leaves partial (max, sum, output) in
 * `workspace`, combined by a merge kernel.  fp32: long prefixes are split into key
 * chunks whose partials are merged by a second kernel.  The call's kernels are
 * chained with programmatic dependent launch; each waits for the kernel before it
 * in the stream to complete before reading its inputs.
 * `workspace` must hold tsv_attn_workspace_size(...) bytes (may be NULL when that
 * is 0); it is scratch owned by the caller, and every byte the call reads there is
 * written earlier in the same call (no clearing needed between calls).
 * Rows of a sequence with seq_err != 0 are written as NaN.
 * Cache slots from L_b + N to the end of the sequence's last block are never
 * read into the result (they may hold anything, NaN included).
 * ------------------------------------------------------------------------- */
size_t tsv_attn_workspace_size(int B, int N, int Hq, int Hkv, int D, int block_size, int max_blocks,
                               tsv_dtype dtype);

tsv_status tsv_tree_verify_attn(const void *q, const void *k_cache, const void *v_cache,
                                const int32_t *block_table, const int32_t *seq_lens,
                                const int32_t *parent, void *out, int B, int N, int Hq, int Hkv,
                                int D, int block_size, int max_blocks, int num_blocks, float scale,
                                tsv_dtype dtype, void *workspace, size_t workspace_bytes,
                                int32_t *seq_err, void *stream);

/* ---------------------------------------------------------------------------
 * tsv_tree_verify_attn with the tree's own K/V appended in the same call (sglang
 * report, "Tree-based Speculative Decoding (EAGLE) Implementation Summary": the KV
 * cache is updated for the tree's tokens before they are verified; vLLM PR #2188,
 * "Guide for reviewers": no host synchronisation inside the step).
 *
 * k_new, v_new [B, N, Hkv, D] (dtype as q) are the tree nodes' K/V rows; node j's row
 * is written to logical slot seq_lens[b] + j of k_cache / v_cache (all kv heads), and
 * the attention then reads it there, exactly as tsv_tree_verify_attn does once the
 * caller has written the rows: same results, same workspace, same errors.  A sequence
 * whose capacity or block ids fail the checks (TSV_DERR_CAPACITY / TSV_DERR_BLOCK)
 * gets no rows written.  The rows are written by the sequence-check kernel, and the
 * attention kernel waits for that kernel (programmatic dependent launch) before its
 * first tile that reaches the tree keys, so the append adds no launch on the bf16
 * path (fp32: one small kernel before the attention).  k_new / v_new must be 16-byte
 * aligned and must not overlap the caches.
 * ------------------------------------------------------------------------- */
tsv_status tsv_tree_verify_attn_append(const void *q, const void *k_new, const void *v_new, void *k_cache,
                                       void *v_cache, const int32_t *block_table,
                                       const int32_t *seq_lens, const int32_t *parent, void *out, int B,
                                       int N, int Hq, int Hkv, int D, int block_size, int max_blocks,
                                       int num_blocks, float scale, tsv_dtype dtype, void *workspace,
                                       size_t workspace_bytes, int32_t *seq_err, void *stream);

/* ---------------------------------------------------------------------------
 * tsv_tree_verify_attn without a caller workspace (the pages have no counterpart
 * of this call; it is an interface convenience).
 *
 * For callers that cannot allocate device memory -- e.g. a plugin inside an engine
 * that owns all device memory and passes only inputs and outputs, or a loop that
 * must not call cudaMalloc because it can synchronise the device.  Same arguments
 * and result as tsv_tree_verify_attn, minus the workspace: the split-K partials go
 * to a scratch array of tsv_noalloc_scratch_bytes() (64 MiB) that the library
 * defines in device memory; every GPU that loads the library holds it until the
 * process exits.  Nothing is allocated per call.
 *  - Shapes whose tsv_attn_workspace_size exceeds the array are rejected with
 *    TSV_ERR_UNSUPPORTED before anything is launched.
 *  - The array used is the CURRENT device's: the current device must be the device
 *    of `stream` and of every buffer (a stream of another device is refused with
 *    TSV_ERR_ARG).
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current; again only if the device's context changes,
 *    e.g. after cudaDeviceReset, which reloads the array with the module); make that
 *    first call before any stream capture.  A failed lookup returns TSV_ERR_CUDA and
 *    is retried by the next call.
 *  - All calls share the array: calls that overlap on the GPU race on it and must
 *    be ordered by the caller.  Each call rewrites every scratch byte it reads.
 * ------------------------------------------------------------------------- */
size_t tsv_noalloc_scratch_bytes(void);

tsv_status tsv_tree_verify_attn_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                        const int32_t *block_table, const int32_t *seq_lens,
                                        const int32_t *parent, void *out, int B, int N, int Hq,
                                        int Hkv, int D, int block_size, int max_blocks,
                                        int num_blocks, float scale, tsv_dtype dtype,
                                        int32_t *seq_err, void *stream);

/* ---------------------------------------------------------------------------
 * Rejection-sampling verification of the tree (statistical-learning-notes ch.07
 * "Speculative Decoding", section "Draft Token Validation"; Sequoia summary,
 * sections "Scalable Speculative Decoding" and "Robust Sampling").
 *
 * Per sequence, starting at the root i = 0:
 *   p = softmax(target_logits[b,i,:] / T), q = draft_probs[b,i,:];
 *   children c of i are tried in increasing index with x = draft_tokens[b,c]:
 *     accept iff u_accept[b,c] < p(x)/q(x)   (q(x) == 0: accept iff p(x) > 0);
 *     on rejection p <- normalize(max(0, p - q)) (kept if that sum is 0),
 *                  q(x) <- 0, q <- normalize(q) (kept if that sum is 0);
 *   the first accepted child becomes i; when no child is accepted (or i is a
 *   leaf) the walk stops and the bonus token is the smallest t with
 *   u_bonus[b] < sum_{v<=t} p(v) over the current p; if there is none (u_bonus >= 1
 *   or NaN, outside the stated [0, 1)), the last t with p(t) > 0.
 * T == 0: a child is accepted iff its token is argmax target_logits[b,i,:]
 * (lowest index on ties) and the bonus is that argmax; draft_probs and the
 * uniforms are not read (draft_probs may be NULL).
 * Outputs: accepted_nodes[b,:] = root-first path, -1 padded; accept_len[b] =
 * drafts accepted (path length - 1); bonus_token[b]; out_tokens[b,:] = accepted
 * draft tokens then the bonus, -1 padded.  A sequence with seq_err != 0 gets
 * accept_len = bonus_token = -1 and all-(-1) rows.
 * Uniforms are pre-drawn by the caller in [0, 1).  T == 0 or T >= 1e-6 (smaller
 * positive T is refused with TSV_ERR_UNSUPPORTED).  Vocabulary-wide sums use fp32
 * per thread and float-float pairs (about 44 significant bits) across threads, warps
 * and CTAs; the ratio p(x)/q(x) is formed in float-float from a compensated exponent
 * argument (relative error a few 1e-7).  V <= 16 * 512 * 32.
 * ------------------------------------------------------------------------- */
tsv_status tsv_tree_reject_sample(const float *target_logits, const float *draft_probs,
                                  const int32_t *draft_tokens, const int32_t *parent,
                                  const float *u_accept, const float *u_bonus, float temperature,
                                  int B, int N, int V, int32_t *accepted_nodes, int32_t *accept_len,
                                  int32_t *bonus_token, int32_t *out_tokens, int32_t *seq_err,
                                  void *stream);

/* ---------------------------------------------------------------------------
 * Variants of the walk (a host struct, read during the call; NULL = the defaults
 * {0, TSV_F32, 0, 1.0f}, i.e. tsv_tree_reject_sample).
 *
 * with_replacement: how the caller's drafter drew the siblings of a node.
 *   0 -- without replacement (Sequoia summary, "Robust Sampling"): the walk above.
 *   1 -- independently from q (the SpecInfer verification that the Sequoia summary's
 *        figure of rejection rates compares against, "More on figures"): after a
 *        rejected sibling only p takes the residual update, p <- normalize(max(0,
 *        p - q)); q is kept (no q(x) <- 0), so siblings may repeat a token.
 *   The walk must match the drafting: each is lossless only for its own drafts.
 * logits_dtype: element type of target_logits, TSV_F32 or TSV_BF16 (the target
 *   model's own output dtype; a bf16 row is half the bytes of an fp32 one).  A bf16
 *   logit is decoded exactly to fp32; everything after the load is the fp32 walk.
 * top_k, top_p: filtered target (the Sequoia summary's table of robustness to
 *   top-p sampling, "More on tables"): at every visited node p is first restricted
 *   to its top_k most probable tokens (top_k = 0: all), then to the smallest prefix
 *   of them, by decreasing p with ties to the lower index, whose mass reaches top_p
 *   (top_p = 1: all), and renormalised; q is the drafter's own (filtered)
 *   distribution as given.  top_k >= V keeps every token.  The cut is found by
 *   bisection over the logits' order (about 35 cluster reductions per visited node,
 *   a few more when the boundary falls inside a run of equal logits), so a filtered
 *   walk costs several times the plain one.  Mass sums are float-float; a cut whose
 *   cumulative mass lies within ~1e-7 of top_p may differ from an exact computation.
 * ------------------------------------------------------------------------- */
typedef struct {
    int with_replacement;
    tsv_dtype logits_dtype;
    int top_k;
    float top_p;
} tsv_walk_options;

/* tsv_tree_reject_sample with options; target_logits has opts->logits_dtype. */
tsv_status tsv_tree_reject_sample_ex(const void *target_logits, const float *draft_probs,
                                     const int32_t *draft_tokens, const int32_t *parent,
                                     const float *u_accept, const float *u_bonus, float temperature,
                                     const tsv_walk_options *opts, int B, int N, int V,
                                     int32_t *accepted_nodes, int32_t *accept_len, int32_t *bonus_token,
                                     int32_t *out_tokens, int32_t *seq_err, void *stream);

/* ---------------------------------------------------------------------------
 * KV-cache rewrite for the accepted path (sglang report: the KV cache must be
 * updated selectively for accepted indices and trees require a rewrite; SGLang
 * "SpeculativeDecoding", prefix match: rejected tokens' KV cache is evicted).
 *
 * For j = 1 .. accept_len[b]: the K and V rows (all kv heads) at logical slot
 * L_b + accepted_nodes[b,j] move to logical slot L_b + j; new_seq_lens[b] =
 * L_b + 1 + accept_len[b].  Slots at or past the new length are evicted by the
 * length cut (their bytes are not cleared; freeing blocks is the caller's).
 * seq_lens is read only, so a repeated call gives the same result.
 * accept_len[b] < 0 leaves the sequence untouched (new_seq_lens[b] = L_b).
 * The path must satisfy 0 = a_0 < a_1 < ... < a_A < N (else TSV_DERR_PARENT).
 * ------------------------------------------------------------------------- */
tsv_status tsv_kv_compact_accepted(void *k_cache, void *v_cache, const int32_t *block_table,
                                   const int32_t *seq_lens, const int32_t *accepted_nodes,
                                   const int32_t *accept_len, int32_t *new_seq_lens, int B, int N,
                                   int Hkv, int D, int block_size, int max_blocks, int num_blocks,
                                   tsv_dtype dtype, int32_t *seq_err, void *stream);

/* ---------------------------------------------------------------------------
 * The walk and the KV-cache rewrite in one launch: the same arguments and results as
 * tsv_tree_reject_sample(...) followed by tsv_kv_compact_accepted(k_cache, v_cache,
 * block_table, seq_lens, accepted_nodes, accept_len, new_seq_lens, ..., compact_err)
 * on the same stream (the rewrite runs in the walk kernel's tail, one CTA per
 * sequence, so it costs no launch of its own).  Walk errors go to seq_err, rewrite
 * errors to compact_err, with the same codes as the two calls.
 * ------------------------------------------------------------------------- */
tsv_status tsv_tree_reject_sample_compact(const float *target_logits, const float *draft_probs,
                                          const int32_t *draft_tokens, const int32_t *parent,
                                          const float *u_accept, const float *u_bonus,
                                          float temperature, int B, int N, int V,
                                          int32_t *accepted_nodes, int32_t *accept_len,
                                          int32_t *bonus_token, int32_t *out_tokens, int32_t *seq_err,
                                          void *k_cache, void *v_cache, const int32_t *block_table,
                                          const int32_t *seq_lens, int32_t *new_seq_lens, int Hkv,
                                          int D, int block_size, int max_blocks, int num_blocks,
                                          tsv_dtype dtype, int32_t *compact_err, void *stream);

/* tsv_tree_reject_sample_compact with the walk options above. */
tsv_status tsv_tree_reject_sample_compact_ex(const void *target_logits, const float *draft_probs,
                                             const int32_t *draft_tokens, const int32_t *parent,
                                             const float *u_accept, const float *u_bonus, float temperature,
                                             const tsv_walk_options *opts, int B, int N, int V,
                                             int32_t *accepted_nodes, int32_t *accept_len,
                                             int32_t *bonus_token, int32_t *out_tokens, int32_t *seq_err,
                                             void *k_cache, void *v_cache, const int32_t *block_table,
                                             const int32_t *seq_lens, int32_t *new_seq_lens, int Hkv, int D,
                                             int block_size, int max_blocks, int num_blocks, tsv_dtype dtype,
                                             int32_t *compact_err, void *stream);

/* ---------------------------------------------------------------------------
 * Tree construction (host side).  Sequoia summary, sections "Scalable Speculative
 * Decoding" and "Dynamic Programming": the tree of speculated tokens is built by
 * dynamic programming to an optimal shape; the figure of forward-pass time against
 * input length: the tree size trades the draft model's time against the target's
 * verification time (hardware-aware).  The pages state neither the objective nor the
 * recurrence; this library reads them as follows.
 *
 * accept[k], k = 0 .. K-1: probability that the (k+1)-th drafted sibling is the one
 * the walk accepts at a node it has reached (positional acceptance, the same at every
 * node; accept[k] >= 0, sum <= 1 + 1e-9); siblings of rank > K are never accepted.
 * A node is reached with the product of accept[rank - 1] over the edges of its root
 * path (rank = 1 + the number of earlier siblings), so the expected number of tokens
 * a verification step generates -- accepted drafts plus the bonus -- is
 *     E(tree) = sum over the tree's nodes of that product   (the root counts 1).
 *
 * These calls read and write HOST memory, run synchronously on the calling thread,
 * need no GPU, and use O(min(d_max, n_max) * min(K, n_max) * n_max) bytes of
 * temporary host memory.  Argument errors return TSV_ERR_ARG.
 * ------------------------------------------------------------------------- */

/* values[n * (d_max + 1) + d] = the largest E over trees of n nodes (root included)
 * and depth <= d (root at depth 0), for 1 <= n <= n_max, 0 <= d <= d_max; row n = 0
 * is 0, and -INFINITY where no tree exists (n > 1 with d = 0).
 * 1 <= n_max <= 128, d_max >= 0, K >= 1; values holds (n_max + 1) * (d_max + 1). */
tsv_status tsv_sequoia_values(const double *accept, int K, int n_max, int d_max, double *values);

/* One tree of n nodes and depth <= max_depth attaining the largest E: parent[0..n-1]
 * in breadth-first order with siblings by rank (parent[0] = -1, parent[i] < i, a
 * node's children have increasing indices in draft order, the order in which the walk
 * tries them); *expected = its E.  1 <= n <= 128; max_depth >= 1 unless n == 1. */
tsv_status tsv_sequoia_tree(const double *accept, int K, int n, int max_depth, int32_t *parent,
                            double *expected);

/* Hardware-aware size and depth: the (n, d) with 1 <= n <= n_max, 0 <= d <= d_max that
 * maximises  speedup(n, d) = E_best(n, d) * t_verify[1] / (t_verify[n] + d * t_draft),
 * where t_verify[n] > 0 is the time of one target forward over n tree tokens
 * (t_verify[1]: one incremental decoding step; t_verify[0] is not read) and
 * t_draft >= 0 the time of one draft forward, run once per tree level.  Ties go to
 * the smaller n, then the smaller d. */
tsv_status tsv_sequoia_plan(const double *accept, int K, int n_max, int d_max, const double *t_verify,
                            double t_draft, int *n_best, int *d_best, double *speedup);

/* Acceptance statistics for the planner, accumulated from verification outputs (HOST
 * copies of parent, accepted_nodes and accept_len, layouts as above).  For every
 * sequence with accept_len[b] >= 0 and every node on its accepted path
 * accepted_nodes[b, 0 .. accept_len[b]] -- the nodes the walk reached -- with c
 * children: reached[k] += 1 for every rank k + 1 <= min(c, K), and accepted[r - 1] += 1
 * when the path goes on to the child of rank r <= K.  Under the positional model above,
 * accepted[k] / reached[k] estimates accept[k].  The counts are added to the arrays
 * (int64 [K]), so steps can be accumulated; sequences with accept_len < 0 are skipped.
 * TSV_ERR_ARG for a parent array that is not a tree or a path that does not follow it. */
tsv_status tsv_sequoia_accept_counts(const int32_t *parent, const int32_t *accepted_nodes,
                                     const int32_t *accept_len, int B, int N, int K, int64_t *reached,
                                     int64_t *accepted);

#ifdef __cplusplus
}
#endif

#endif /* TSV_H */
