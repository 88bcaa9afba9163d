/*
 * spec_verify.h — C ABI of the speculative-decoding verification library
 * (libspecverify.so, sm_103a).
 *
 * One call verifies the draft tokens of B requests against the target model's
 * logits on the caller's CUDA stream.  Sources of each operation:
 *
 *   chain verify   vLLM anatomy page ("Inside vLLM", part 3), section
 *                  "Speculative Decoding": accept/reject left to right, stop
 *                  at the first rejection, sample the rebalanced distribution
 *                  max(0, p_large - p_draft) normalised, or the bonus token
 *                  from the extra row when all k drafts are accepted.  The
 *                  vLLM learning book, section 2 (Leviathan 2023 flowchart),
 *                  gives the test r < min(1, p(x_i)/q(x_i)).  The TensorRT-LLM
 *                  walkthrough (part 10), rejection-sampling section, fixes the
 *                  shapes draft [batch, D, vocab], target [batch, D+1, vocab]
 *                  and the output accepted_tokens [batch, D+1] padded with -1.
 *   greedy verify  Kestrel article 32, section 3.3: accept while the target's
 *                  argmax equals the draft; the emitted stream is the target's
 *                  own argmax chain.  TensorRT-LLM walkthrough, rejection-
 *                  sampling section: an all-greedy batch takes the base path.
 *   tree verify    TensorRT-LLM deployment page ("05-TensorRT-LLM 推测解码"),
 *                  section "Eagle-2 多层级树状草稿生成": paths tensor
 *                  [batch, max_decoding_tokens, max_path_len].
 *   rollback       TensorRT-LLM walkthrough, update_requests section
 *                  (py_rewind_len = verified_len - accepted) and the paged
 *                  rewind_cache section (only the logical length moves; rows
 *                  are not cleared).  Kestrel article 32, section 3.1
 *                  (truncate = move the cursor, copy nothing).
 *
 * Conventions for every call
 *   - All array pointers are DEVICE pointers owned by the caller; the library
 *     never allocates or frees memory.  It keeps no global state apart from
 *     the fixed scratch array of spec_verify_chain_noalloc.  Arrays are
 *     dense, row-major, with the shapes given below.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     A host-detectable error (bad size, null pointer, small workspace)
 *     returns before any launch and writes nothing.  A failed launch returns
 *     SPEC_ECUDA.
 *   - Data-dependent errors (a token or node id out of range) do not stop the
 *     call: the affected request fails closed (its num_accepted is -1, its
 *     token row is all -1, its seq_len is left unchanged) and the status word
 *     in the workspace records SPEC_EBADINDEX; read it with spec_last_error().
 *   - Logits must be finite or -inf (masked), with at least one finite value
 *     per row; NaN and +inf are outside the contract and are not checked.
 *   - One workspace serves one stream at a time: calls that overlap on the GPU
 *     must not share a workspace.
 *   - The second phase of a verify waits (bounded, about one second) for
 *     words the first phase publishes.  A wait that runs out records
 *     SPEC_ETIMEOUT in the status word and fails the requests that depended
 *     on it closed, as above; it cannot happen unless the GPU is broken or
 *     another kernel starves the call.
 *   - Every call leaves its workspace ready for the next.  After a call that
 *     returned SPEC_ECUDA, or whose status word reads SPEC_ETIMEOUT, zero the
 *     workspace again with spec_workspace_init before reusing it.
 *   - Calls run on the device that is current for the calling thread; the
 *     arrays and the stream must belong to it.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st *spec_stream_t;

typedef enum {
    SPEC_OK = 0,
    SPEC_EINVAL = -1,      /* bad size, dtype, temperature or null pointer */
    SPEC_EBADINDEX = -2,   /* a token or node id was out of range (device status) */
    SPEC_ECUDA = -3,       /* a CUDA launch or copy failed */
    SPEC_EWORKSPACE = -4,  /* workspace missing or smaller than spec_workspace_size() */
    SPEC_ETIMEOUT = -5,    /* a bounded device wait ran out (device status) */
    SPEC_ELIMIT = -6       /* a filtered row's cut search found its bins inconsistent
                              (an internal check, not expected; device status) */
} spec_status_t;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype_t;

/* Largest supported draft length k of a chain call, and the largest tree
 * (N nodes, L path length) of a tree call. */
#define SPEC_MAX_DRAFT 64
/* Largest batch B of any call. */
#define SPEC_MAX_BATCH 8192
/* Largest top_k the filtered chain verify serves with explicit kept lists;
 * a larger top_k (and top-p or min_p without top-k) takes per-row cuts. */
#define SPEC_MAX_TOPK 256
#define SPEC_MAX_TREE_NODES 1024
#define SPEC_MAX_PATH_LEN 64

/* Bytes of scratch one call needs for B requests of `rows_per_request` logit
 * rows of width V (chain: 2k+1, greedy: k+1, tree: N).  Returns 0 for invalid
 * sizes.  The same workspace may be reused by any call whose own size is not
 * larger.  Every workspace starts with a fixed 512 KB block of per-request
 * sync lines (SPEC_MAX_BATCH of them). */
size_t spec_workspace_size(int B, int rows_per_request, int V);

/* Bytes of scratch of a filtered chain verify (spec_chain_params with
 * top_k > 0, or top_k = 0 with top_p < 1 or min_p > 0) of B requests, k
 * drafts, width V: the chain's, plus for 1 <= top_k <= SPEC_MAX_TOPK each
 * row's kept list (top_k words), 2k probabilities per request and two bytes
 * per 2048 logits of each row; for top_k = 0 or top_k > SPEC_MAX_TOPK
 * (per-row cuts) each row's 2048-bin mass histogram and counts (24 KB), a
 * 64-byte record and a 4096-entry candidate list (16 KB).  Returns 0 for
 * invalid sizes (top_k < 0 included). */
size_t spec_workspace_size_filtered(int B, int k, int V, int top_k);

/* Zero a workspace (asynchronously, on `stream`).  Call once after allocating
 * it; every verify call leaves it ready for the next. */
int spec_workspace_init(void *workspace, size_t workspace_bytes, spec_stream_t stream);

/* Chain rejection-sampling verify.
 *   target_logits  [B, k+1, V] of `dtype`: row i (i < k) is the target
 *                  distribution of draft position i, row k the bonus row.
 *   draft_logits   [B, k, V] of `dtype`: row i is the draft distribution
 *                  that draft token i was sampled from.
 *   draft_tokens   [B, k] int32 in [0, V).
 *   uniforms       [B, k+1] float32 in [0, 1): column i < k is the accept
 *                  test of position i, column k drives the final sample.
 *   temperature    > 0 and finite; both rows are softmax(logits / T).
 * Accepts x_i while uniforms[b,i] < p_i(x_i) / q_i(x_i) (q == 0 accepts).
 * At the first rejection j the last token is drawn from max(0, p_j - q_j)
 * normalised; when all k are accepted it is drawn from p_k.  The draw takes
 * the smallest t whose cumulative weight exceeds uniforms[b,k] times the
 * total.
 *   out_tokens       [B, k+1] int32: x_0..x_{n-1}, the final token, -1 pad.
 *   out_num_accepted [B] int32: n in [0, k] (-1 for a failed request).
 *   out_probs        [B, k, 2] float32 or NULL: p_i(x_i), q_i(x_i) for every i.
 *   seq_lens         [B] int32 or NULL: KV cursor, updated in place to
 *                    seq_len + n + 1 (see spec_rollback_lengths).
 * Probabilities are accumulated in fp32. */
int spec_verify_chain(const void *target_logits, const void *draft_logits, int dtype,
                      const int32_t *draft_tokens, const float *uniforms, float temperature,
                      int B, int k, int V,
                      int32_t *out_tokens, int32_t *out_num_accepted, float *out_probs,
                      int32_t *seq_lens,
                      void *workspace, size_t workspace_bytes, spec_stream_t stream);

/* Chain verify with each request's uniforms drawn inside the kernel from a
 * per-request Philox state (TensorRT-LLM walkthrough, rejection-sampling
 * section: chain_speculative_sampling takes a seed and an offset per request,
 * the offset keeping each request's stream apart so that the seed can stay
 * constant).  Arguments and results are those of spec_verify_chain, with
 *   seeds    [B] uint64: Philox4x32-10 key (low word first);
 *   offsets  [B] uint64: counter, advanced by the caller between steps;
 * in place of uniforms.  Uniform i of request b (i = 0..k; i < k are the
 * accept tests, i = k drives the final draw) is word i % 4 of
 * Philox4x32-10(counter = (low word of offset, high word of offset, i / 4, 0),
 * key = seed) (Salmon et al., SC'11), shifted right by 8 and scaled by 2^-24.
 * The pages fix the state, not this mapping: it is this library's reading. */
int spec_verify_chain_philox(const void *target_logits, const void *draft_logits, int dtype,
                             const int32_t *draft_tokens, const uint64_t *seeds,
                             const uint64_t *offsets, float temperature, int B, int k, int V,
                             int32_t *out_tokens, int32_t *out_num_accepted, float *out_probs,
                             int32_t *seq_lens, void *workspace, size_t workspace_bytes,
                             spec_stream_t stream);

/* Parameters of spec_verify_chain_ex: those of spec_verify_chain and
 * spec_verify_chain_philox in one struct, plus ragged draft lengths and
 * top-k / top-p filtering.  Set size = sizeof(spec_chain_params); fields a
 * later version adds go at the end, and a smaller size (an earlier version
 * of the struct, ending at seq_lens) leaves the added fields at their
 * defaults (no filtering).
 *   draft_lens [B] int32 or NULL: request b has k_b <= k real drafts in the
 *     buffers padded to k (TensorRT-LLM walkthrough: the real draft count is
 *     kept apart from the padded buffer, pad_draft_tokens_for_cuda_graph; the
 *     verified window is per request, verify_lens).  It is verified as a chain
 *     of k_b: accept tests on positions 0..k_b-1, the final draw uses uniform
 *     column (or Philox index) k_b and target row k_b is its bonus row.  Rows
 *     past k_b are not read (pass 1 skips them) and their draft tokens are not
 *     checked; out_probs there is NaN.  A length outside [0, k] fails the
 *     request closed (SPEC_EBADINDEX in the status word).
 *   uniforms or (seeds, offsets): exactly as in the two calls above; when
 *     uniforms is NULL both seeds and offsets are required. */
typedef struct spec_chain_params {
    size_t size;
    const void *target_logits;  /* [B, k+1, V] */
    const void *draft_logits;   /* [B, k, V] */
    int dtype;
    const int32_t *draft_tokens; /* [B, k] */
    const int32_t *draft_lens;   /* [B] or NULL */
    const float *uniforms;       /* [B, k+1] or NULL */
    const uint64_t *seeds;       /* [B] when uniforms is NULL */
    const uint64_t *offsets;     /* [B] when uniforms is NULL */
    float temperature;
    int B, k, V;
    int32_t *out_tokens;         /* [B, k+1] */
    int32_t *out_num_accepted;   /* [B] */
    float *out_probs;            /* [B, k, 2] or NULL */
    int32_t *seq_lens;           /* [B] or NULL */
    /* Symmetric filtering (TensorRT-LLM walkthrough, rejection-sampling
     * section: target and draft are filtered by the same backend and
     * parameters, or the accept test is silently wrong).  top_k = 0: none.
     * top_k >= 1: every target and draft row keeps its top_k tokens by
     * (logit descending, token ascending) (top_k >= V: all), then the
     * shortest prefix of them whose softmax mass (over those top_k, at
     * temperature T) reaches top_p (top_p = 1: all top_k); p and q are the
     * softmax over the kept set, and the chain verify above runs on them
     * (the final draw takes u * Z over the kept tokens in token order).
     * out_probs holds the filtered p and q.  Logits of -inf carry weight 0
     * (they change no probability, no top-p prefix and no draw); logits must
     * not be NaN or +inf.  top_p in (0, 1].  top_k = 0 with top_p < 1 keeps
     * the shortest prefix of the whole row whose mass reaches top_p.  Kept
     * sets of any size are exact: 1 <= top_k <= SPEC_MAX_TOPK uses explicit
     * kept lists, top_k = 0 (with top_p < 1 or min_p > 0) and top_k >
     * SPEC_MAX_TOPK a per-row cut found from a mass histogram and a radix
     * selection over the tokens of the bins the cut can fall in.  The
     * workspace must hold spec_workspace_size_filtered(B, k, V, top_k)
     * bytes. */
    int top_k;
    float top_p;
    /* min_p in [0, 1] (0: off), applied after top-p (the walkthrough names
     * temperature, top-k, top-p and min_p in that order): a token of the
     * kept set stays when its probability is at least min_p times the
     * largest, 2^((x - x_max) log2(e) / T) >= min_p.  A struct ending at
     * top_p leaves it at 0. */
    float min_p;
} spec_chain_params;
int spec_verify_chain_ex(const spec_chain_params *params, void *workspace,
                         size_t workspace_bytes, spec_stream_t stream);

/* Parameters of spec_verify_greedy_ex: spec_verify_greedy's plus ragged
 * draft lengths (as in spec_chain_params: a request with k_b drafts is
 * greedy-verified over positions 0..k_b-1 and its bonus token is the argmax
 * of target row k_b; rows past k_b are not read). */
typedef struct spec_greedy_params {
    size_t size;
    const void *target_logits;   /* [B, k+1, V] */
    int dtype;
    const int32_t *draft_tokens; /* [B, k] */
    const int32_t *draft_lens;   /* [B] or NULL */
    int B, k, V;
    int32_t *out_tokens;         /* [B, k+1] */
    int32_t *out_num_accepted;   /* [B] */
    int32_t *seq_lens;           /* [B] or NULL */
} spec_greedy_params;
int spec_verify_greedy_ex(const spec_greedy_params *params, void *workspace,
                          size_t workspace_bytes, spec_stream_t stream);

/* Rollback with ragged draft lengths and paged block accounting
 * (TensorRT-LLM walkthrough: update_requests sets rewind = verified_len -
 * accepted; rewind_cache recomputes the blocks needed from tokens_per_block
 * and returns only whole surplus blocks, clearing nothing).
 *   k_b = draft_lens[b] (or k when NULL); new_lens = old_lens + n + 1;
 *   rewind_lens (nullable) = k_b - n; free_blocks (nullable) = max(0,
 *   blocks_held[b] - ceil(new_len / tokens_per_block)), 0 when blocks_held is
 *   NULL.  new_lens may alias old_lens.  An entry with k_b outside [0, k] or
 *   n outside [0, k_b] (a failed request reads n = -1) keeps its length; its
 *   rewind reads -1 and its free count 0. */
int spec_rollback_paged(const int32_t *old_lens, const int32_t *num_accepted,
                        const int32_t *draft_lens, int k, const int32_t *blocks_held,
                        int tokens_per_block, int B, int32_t *new_lens, int32_t *rewind_lens,
                        int32_t *free_blocks, spec_stream_t stream);

/* The uniforms spec_verify_chain_philox draws: out[b, i] for i = 0..n-1
 * (n <= SPEC_MAX_DRAFT + 1), from the same per-request Philox streams, so a
 * caller can log or replay a step's randomness. */
int spec_philox_uniforms(const uint64_t *seeds, const uint64_t *offsets, int B, int n,
                         float *out, spec_stream_t stream);

/* Greedy chain verify.
 *   target_logits [B, k+1, V], draft_tokens [B, k] in [0, V).
 * g_i = argmax_t target[b,i,t] on the stored values, lowest id on ties;
 * n = the longest prefix with g_i == d_i; out_tokens [B, k+1] =
 * d_0..d_{n-1}, g_n, -1 pad; out_num_accepted [B]; seq_lens as above. */
int spec_verify_greedy(const void *target_logits, int dtype, const int32_t *draft_tokens,
                       int B, int k, int V,
                       int32_t *out_tokens, int32_t *out_num_accepted, int32_t *seq_lens,
                       void *workspace, size_t workspace_bytes, spec_stream_t stream);

/* Greedy tree verify over EAGLE-style paths.
 *   target_logits [B, N, V]: row n is the target distribution after node n;
 *                 node 0 is the root (the last committed token).
 *   tree_tokens   [B, N] int32 in [0, V): node n's token.
 *   paths         [B, P, L] int32 in [-1, N): root-to-leaf node lists padded
 *                 with -1; a used path starts with 0, an unused one with -1.
 * For every used path, step j = 1..L-1 is accepted while its node is >= 0 and
 * its token equals argmax of its parent's row; the path with the most
 * accepted steps wins (lowest path index on ties).
 *   out_tokens         [B, L] int32: accepted tokens, then argmax of the last
 *                      accepted node's row, -1 pad.
 *   out_num_accepted   [B] int32 (-1 for a failed request).
 *   out_best_path      [B] int32 or NULL (-1 when no path is used).
 *   out_accepted_nodes [B, L] int32 or NULL: the root and the accepted node
 *                      ids (the KV rows to keep), -1 pad.
 *   seq_lens           [B] int32 or NULL, updated to seq_len + n + 1. */
int spec_verify_tree(const void *target_logits, int dtype, const int32_t *tree_tokens,
                     const int32_t *paths, int B, int N, int P, int L, int V,
                     int32_t *out_tokens, int32_t *out_num_accepted, int32_t *out_best_path,
                     int32_t *out_accepted_nodes, int32_t *seq_lens,
                     void *workspace, size_t workspace_bytes, spec_stream_t stream);

/* Stochastic tree verify (TensorRT-LLM deployment page, "目标模型验证：树注意力
 * 与批量并行": the tree's tokens are judged against the target logits by
 * rejection sampling; children are chosen by top-K per level, "Eagle-2
 * 多层级树状草稿生成").  A chosen child is a point-mass proposal on its token,
 * so the rejection-sampling rule becomes: at each node, try its children in
 * increasing node id; accept child c iff uniforms[b, c] < p'(token of c), the
 * current residual of the node's softmax(row / T); on a rejection remove that
 * token from the residual and renormalise; when no child is accepted (or the
 * node has none, or L - 1 steps were taken) draw the final token from the
 * residual by inverse CDF at uniforms[b, 0] (from the node's own row if the
 * residual's mass vanished).  The emitted tokens follow the target rows.
 *   target_logits [B, N, V], tree_tokens [B, N], paths [B, P, L]: as for
 *                 spec_verify_tree; a node's children are the entries d + 1
 *                 of the used paths whose first d + 1 entries are the
 *                 accepted prefix.  P * L <= 4096.
 *   uniforms      [B, N] float32 in [0, 1): column n >= 1 is node n's accept
 *                 test, column 0 drives the final draw.
 *   temperature   > 0 and finite.
 *   Outputs as for spec_verify_tree: tokens [B, L] (accepted tokens, the
 *   final token, -1 pad), num_accepted [B], best_path [B] (the lowest used
 *   path holding the accepted nodes, -1 when none), accepted_nodes [B, L];
 *   seq_lens advanced by n + 1.  Workspace: spec_workspace_size(B, N, V). */
int spec_verify_tree_sampled(const void *target_logits, int dtype, const int32_t *tree_tokens,
                             const int32_t *paths, const float *uniforms, float temperature,
                             int B, int N, int P, int L, int V,
                             int32_t *out_tokens, int32_t *out_num_accepted,
                             int32_t *out_best_path, int32_t *out_accepted_nodes,
                             int32_t *seq_lens, void *workspace, size_t workspace_bytes,
                             spec_stream_t stream);

/* KV cursor rollback as length arithmetic only (no KV row is copied or
 * cleared; rows past the new length become invisible and are overwritten
 * later).
 *   old_lens [B]: cursor before the verify window was written.
 *   num_accepted [B]: n per request; k = draft rows in the verify window
 *   (chain: k; tree: N - 1).
 *   new_lens [B] = old_lens + n + 1 (may alias old_lens);
 *   rewind_lens [B] or NULL = k - n (rows written but not kept).
 * An entry with n outside [0, k] (a failed request reads n = -1) keeps its
 * length and its rewind reads -1, so a caller can tell it from a valid
 * rewind (>= 0); the call itself returns SPEC_OK. */
int spec_rollback_lengths(const int32_t *old_lens, const int32_t *num_accepted, int k, int B,
                          int32_t *new_lens, int32_t *rewind_lens, spec_stream_t stream);

/* Accepted-KV relocation after a tree verify (TensorRT-LLM walkthrough, the
 * "moving to the right place" step before update_resources,
 * _update_kv_cache_draft_token_location): the KV rows of the accepted nodes,
 * written in tree order during the draft step, are gathered into consecutive
 * logical positions right after the committed prefix.  As on that page the
 * cache is paged.
 *   kv_pool        [num_blocks * tokens_per_block, row_bytes] device memory,
 *                  16-byte aligned; one row per token (one layer's K and V
 *                  of every KV head, or however the caller lays a token out).
 *                  row_bytes must be a multiple of 16.
 *   block_tables   [B, max_blocks] int32: request b's logical position t is
 *                  pool row block_tables[b][t / tokens_per_block] *
 *                  tokens_per_block + t % tokens_per_block.  Blocks holding
 *                  the window must not be shared between requests.
 *   base_lens      [B] int32: logical position of tree node 0 (the committed
 *                  length before the verify window).
 *   accepted_nodes [B, L] int32 and num_accepted [B]: spec_verify_tree's
 *                  outputs (root, then the n accepted nodes; -1 padded).
 * For j = 1..n, row base + accepted_nodes[b][j] moves to row base + j; rows
 * past base + n are left as they are (the rollback makes them invisible).
 * A request is left untouched when n <= 0 or n >= L (failed closed), or when
 * its path does not start at node 0 with strictly increasing nodes, or a row
 * it would read or write is unmapped (a block id outside [0, num_blocks) or
 * a position past max_blocks * tokens_per_block); no status is recorded.
 * Returns SPEC_EINVAL for null pointers, sizes outside the limits or a
 * misaligned pool. */
int spec_relocate_accepted_kv(void *kv_pool, size_t row_bytes, int tokens_per_block,
                              int num_blocks, const int32_t *block_tables, int max_blocks,
                              const int32_t *base_lens, const int32_t *accepted_nodes,
                              const int32_t *num_accepted, int B, int L, spec_stream_t stream);

/* Chain verify without a caller-provided workspace, for callers that cannot
 * allocate device memory (code whose allocator forbids allocations while a
 * step runs, or host code that owns no CUDA allocator).  The pages have no
 * counterpart: it is an addition of this library.
 *   Arguments and results are those of spec_verify_chain; inputs and outputs
 *   are still the caller's device arrays.
 *   Scratch: a file-scope device array of SPEC_NOALLOC_SCRATCH_BYTES that
 *   every GPU loading the library holds until the process exits.  A problem
 *   whose spec_workspace_size(B, 2k+1, V) exceeds it returns SPEC_EWORKSPACE
 *   before any launch.
 *   Every call on a device shares the one array: calls that can overlap on the
 *   GPU (other streams, other threads) race and must be serialised by the
 *   caller.  Each call clears the array's counters and status word on
 *   `stream` before launching, so there is no status word to read: the only
 *   data-dependent signal is a request that fails closed (num_accepted ==
 *   -1, tokens -1, seq_len unchanged), whether for a bad draft token or for
 *   a device wait that ran out.
 *   The arrays must be device (or managed) memory of the current device:
 *   the array used as scratch is the current device's.  Every argument is
 *   checked before the array is written; a refused call (SPEC_EINVAL,
 *   SPEC_EWORKSPACE) leaves it untouched.  Each call looks up the array's
 *   device address (cudaGetSymbolAddress) with its device current, so no
 *   call needs a set-up step first.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
#define SPEC_NOALLOC_SCRATCH_BYTES (4u << 20)
int spec_verify_chain_noalloc(const void *target_logits, const void *draft_logits, int dtype,
                              const int32_t *draft_tokens, const float *uniforms,
                              float temperature, int B, int k, int V,
                              int32_t *out_tokens, int32_t *out_num_accepted, float *out_probs,
                              int32_t *seq_lens, spec_stream_t stream);

/* Fault injection for tests of the bounded device waits (no counterpart on
 * the pages).  Each runs its call with the first phase left out, so that the
 * words the second phase waits for are never written, and with every device
 * wait bounded by wait_cycles SM clock cycles (>= 1) instead of about one
 * second.  Arguments are those of spec_verify_chain_ex (plain or filtered
 * with kept lists; a filtered call whose rows are wider than one CTA's codes
 * has no wait and returns SPEC_ECUDA, and the per-row-cut filter (top_k = 0
 * with top_p < 1 or min_p > 0, or top_k > SPEC_MAX_TOPK) waits for nothing
 * and returns SPEC_EINVAL) / spec_verify_greedy_ex.  Expected outcome: every
 * request fails closed and the status word reads SPEC_ETIMEOUT.  The
 * workspace may hold stale words afterwards: zero it with
 * spec_workspace_init before its next use. */
int spec_test_timeout_chain(const spec_chain_params *params, long long wait_cycles,
                            void *workspace, size_t workspace_bytes, spec_stream_t stream);
int spec_test_timeout_greedy(const spec_greedy_params *params, long long wait_cycles,
                             void *workspace, size_t workspace_bytes, spec_stream_t stream);

/* Synchronise `stream`, read the workspace status word into *status_out
 * (SPEC_OK, SPEC_EBADINDEX or SPEC_ETIMEOUT) and clear it.  Returns SPEC_OK, SPEC_EINVAL or
 * SPEC_ECUDA. */
int spec_last_error(void *workspace, size_t workspace_bytes, spec_stream_t stream,
                    int *status_out);

/* Static text for a status code. */
const char *spec_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
