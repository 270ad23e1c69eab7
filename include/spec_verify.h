/*
 * spec_verify.h -- C ABI of libspecverify, the GB300 (sm_103a) verify-and-accept
 * step of speculative decoding.
 *
 * What the step computes (the speculative-decoding pages):
 *  - EAGLE-3 review, "Speculative Decoding" (draft, verification, accept or
 *    reject): the target model scores k draft tokens in one forward pass and
 *    returns next-token distributions at k+1 positions; drafts are checked
 *    front to back; the first rejection ends the step and its position is
 *    resampled; when all k drafts pass, the distribution at position k+1 gives
 *    one more (bonus) token, so every step emits at least one token.
 *  - EAGLE-3 review, section on whether a small draft model hurts quality:
 *    greedy decoding accepts a draft iff it equals the target argmax and
 *    otherwise emits that argmax; sampling accepts x with probability
 *    min(1, p(x)/q(x)) and resamples a rejection from norm(max(0, p - q)).
 *  - Serving-book chapter, "acceptance rule that preserves the output
 *    distribution": temperature 0 is the greedy case.
 *  - EAGLE-3 review, "EAGLE-3 inference" steps 3-5 and the vLLM EAGLE
 *    walkthrough, "tree drafting in detail": a token tree is verified in one
 *    forward; greedy verification keeps the longest root-to-node path whose
 *    tokens all match the target's choices; tree_choices gives
 *    num/cu/child drafts per level.
 *  - vLLM EAGLE walkthrough, "handling rejected tokens" and "slot mapping and
 *    KV-cache management": the slot_mapping entries of rejected tokens are
 *    replaced by PADDING_SLOT_ID so their KV never lands in the cache.
 *
 * Conventions for every entry point:
 *  - Ownership: the caller owns every buffer.  The library never allocates or
 *    frees device memory and keeps no pointer after a call returns.
 *  - Execution: device work is enqueued on `stream` (a cudaStream_t passed as
 *    void*, NULL = the legacy default stream) on the calling thread's current
 *    device; there is no host synchronisation inside a call.
 *  - "device" pointers must be device-accessible memory of the current device;
 *    "host" pointers are read during the call only.
 *  - Layouts are dense row-major (C order) with the shapes given below.
 *  - Host-side checks run before any launch; a failed check returns
 *    SPEC_ERR_INVALID_ARG and enqueues nothing.  A device that is not
 *    compute capability 10.3 returns SPEC_ERR_UNSUPPORTED.  A CUDA launch
 *    failure returns SPEC_ERR_CUDA (spec_last_error() gives the text).
 *  - Data problems found on the device never trap: they OR bits into the
 *    caller's int32 status word (SPEC_STATUS_*), which the library never
 *    clears.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1,
    SPEC_ERR_UNSUPPORTED = 2,
    SPEC_ERR_CUDA = 3
} spec_status_t;

typedef enum { SPEC_BF16 = 0, SPEC_FP32 = 1 } spec_dtype_t;

/* Bits OR-ed into the device status word. */
#define SPEC_STATUS_TOKEN_RANGE 1  /* a draft token outside [0, V): treated as a rejection */
#define SPEC_STATUS_NONFINITE 2    /* a NaN or +inf logit was read, or a row was -inf throughout
                                      (results undefined).  A -inf logit alone is a masked
                                      token: probability 0, never the argmax of a finite row. */
#define SPEC_STATUS_WAIT_TIMEOUT 4 /* an inter-block wait gave up (results of that request undefined) */
#define SPEC_STATUS_BAD_OFFSETS 8  /* ragged chains: cu_num_draft_tokens not non-decreasing within
                                      [0, total_drafts] or a count above max_k (clamped; results of
                                      the requests involved undefined) */
#define SPEC_STATUS_SLOT_RANGE 32  /* next-step preparation / KV compaction: a position past the block
                                      table or a negative table entry (the slot is padded), or a KV slot
                                      outside the cache (that row is not moved) */
#define SPEC_STATUS_BAD_TEMPERATURE 16 /* sampled trees: a temperature that is not finite and > 0 (that
                                          request is walked with T = 1; greedy trees go through
                                          spec_verify_tree) */

/* Largest rows per request (k+1 for chains, N+1 for trees). */
#define SPEC_MAX_ROWS 256

/* Workspace bytes needed by spec_verify_chain / spec_verify_tree for B requests
 * of `rows` logits rows (k+1 or N+1) over vocabulary V.  The workspace is
 * device memory owned by the caller, 16-byte aligned.  It must be zero-filled
 * (spec_workspace_init) before its first use and before any call whose
 * (B, rows, V, dtype) differs from the previous call on it: its counter
 * region sits at offsets that depend on those sizes.  Every completed call
 * leaves the counter region of its own layout zero again, so repeated calls
 * (or CUDA-graph replays) with the same sizes need no re-initialisation.
 * Bytes [0, 64) hold eight uint64 diagnostic counters the kernel only adds to
 * (A-row chunks loaded, A chunks skipped, residual chunks loaded, residual
 * chunks skipped, bytes streamed, 3 reserved).  One workspace must not be
 * used by two calls that can run at the same time.
 * Returns 0 for invalid sizes. */
size_t spec_workspace_bytes(int B, int rows, int V, spec_dtype_t dtype);

/* Zero-fills `bytes` of device workspace on `stream` (cudaMemsetAsync). */
spec_status_t spec_workspace_init(void *workspace, size_t bytes, void *stream);

/*
 * Chain verification (draft, verify, accept/reject as summarised above).
 *
 *  target_logits [B, k+1, V] device, dtype bf16 or fp32, 16-byte aligned.
 *      Row i (0-based) is the target's next-token distribution after the
 *      prefix plus drafts 1..i; row k scores the bonus token.
 *  draft_probs   [B, k, V] fp32 device, 16-byte aligned, or NULL when every
 *      request is greedy.  Row i is the draft distribution q that draft
 *      token i+1 was drawn from; it is used as given (no temperature).
 *  draft_tokens  [B, k] int32 device.
 *  temperature   [B] fp32 device, or NULL (every request greedy).  T == 0 is
 *      greedy; T > 0 samples from p = softmax(z / T).  Negative T is invalid.
 *  u_accept      [B, k] fp32 device in [0, 1), or NULL when every request is
 *      greedy.  Draft i+1 is accepted iff q(x) == 0 or u_accept[b,i] < p(x)/q(x).
 *  u_sample      [B, k+1] fp32 device in [0, 1), or NULL when every request is
 *      greedy.  A request rejected at row a draws its token with u_sample[b,a]
 *      (the bonus row k uses u_sample[b,k]) by inverse CDF: the smallest j
 *      whose prefix mass exceeds u * (total mass).
 *  out_tokens    [B, k+1] int32 device: drafts 1..a, then the corrected or
 *      bonus token, then -1 padding.
 *  out_num_accepted [B] int32 device: a in [0, k].
 *  d_status      one int32 device word (may be NULL): SPEC_STATUS_* bits.
 *  workspace / workspace_bytes: see spec_workspace_bytes(B, k+1, V, dtype).
 *  Sizes: 1 <= B, 1 <= k <= SPEC_MAX_ROWS-1, 1 <= V < 2^30.
 */
spec_status_t spec_verify_chain(const void *target_logits, spec_dtype_t dtype,
                                const float *draft_probs, const int32_t *draft_tokens,
                                const float *temperature, const float *u_accept,
                                const float *u_sample, int B, int k, int V,
                                int32_t *out_tokens, int32_t *out_num_accepted,
                                int32_t *d_status, void *workspace, size_t workspace_bytes,
                                void *stream);

/*
 * spec_verify_chain with the slot_mapping fix-up fused into the same launch:
 * slot_mapping [B, k+1] int64 device memory, and entry j of request b becomes
 * padding_slot_id iff j > num_accepted[b] (what spec_fixup_slots in chain mode
 * writes afterwards), written when request b's outcome is known.  Other
 * arguments, sizes and errors as spec_verify_chain; slot_mapping must not be
 * NULL.
 */
spec_status_t spec_verify_chain_fused(const void *target_logits, spec_dtype_t dtype, const float *draft_probs,
                                      const int32_t *draft_tokens, const float *temperature, const float *u_accept,
                                      const float *u_sample, int B, int k, int V, int32_t *out_tokens,
                                      int32_t *out_num_accepted, int64_t *slot_mapping, int64_t padding_slot_id,
                                      int32_t *d_status, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Ragged chain verification: a different number of drafts per request, packed
 * (the vLLM speculative-decoding walkthrough's per-step metadata:
 * cu_num_draft_tokens offsets into packed draft and target rows).  Greedy and
 * sampled requests may be mixed, as in spec_verify_chain.
 *
 *  cu_num_draft_tokens [B+1] int32 device, non-decreasing, cu[0] = 0,
 *      cu[B] = total_drafts: request b has k_b = cu[b+1] - cu[b] drafts
 *      (0 <= k_b <= max_k).
 *  target_logits [total_drafts + B, V] device: request b's k_b + 1 rows start
 *      at row cu[b] + b (row i of the request as in spec_verify_chain).
 *  draft_probs   [total_drafts, V] fp32 device or NULL: request b's rows start
 *      at row cu[b].
 *  draft_tokens, u_accept [total_drafts] packed the same way (u_accept NULL when
 *      every request is greedy).
 *  u_sample      [total_drafts + B], packed like the logits rows.
 *  temperature   [B], as in spec_verify_chain.
 *  out_tokens    [B, max_k+1] int32 device (padded, -1 after the emitted tokens).
 *  out_num_accepted [B] int32 device: a_b in [0, k_b].
 *  workspace: spec_workspace_bytes(B, max_k+1, V, dtype).
 *  Offsets that break the rules above are clamped so nothing is read outside
 *  the packed inputs, and SPEC_STATUS_BAD_OFFSETS is set.
 *  Sizes: 1 <= B, 0 <= max_k <= SPEC_MAX_ROWS-1, 1 <= V < 2^30,
 *  0 <= total_drafts <= B * max_k.
 */
spec_status_t spec_verify_chain_ragged(const void *target_logits, spec_dtype_t dtype,
                                       const float *draft_probs, const int32_t *draft_tokens,
                                       const int32_t *cu_num_draft_tokens, int total_drafts,
                                       const float *temperature, const float *u_accept,
                                       const float *u_sample, int B, int max_k, int V,
                                       int32_t *out_tokens, int32_t *out_num_accepted,
                                       int32_t *d_status, void *workspace, size_t workspace_bytes,
                                       void *stream);

/*
 * spec_verify_chain_ragged with the ragged slot_mapping fix-up fused into the
 * same launch: slot_mapping holds total_drafts + B int64 entries packed as for
 * spec_fixup_slots_ragged, and slot j of request b (entry cu[b] + b + j)
 * becomes padding_slot_id iff j > num_accepted[b].  slot_mapping must not be
 * NULL; everything else as spec_verify_chain_ragged.
 */
spec_status_t spec_verify_chain_ragged_fused(const void *target_logits, spec_dtype_t dtype,
                                             const float *draft_probs, const int32_t *draft_tokens,
                                             const int32_t *cu_num_draft_tokens, int total_drafts,
                                             const float *temperature, const float *u_accept, const float *u_sample,
                                             int B, int max_k, int V, int32_t *out_tokens,
                                             int32_t *out_num_accepted, int64_t *slot_mapping,
                                             int64_t padding_slot_id, int32_t *d_status, void *workspace,
                                             size_t workspace_bytes, void *stream);

/*
 * Greedy token-tree verification (EAGLE-style tree, one verification forward).
 *
 *  target_logits [B, N+1, V] device, bf16 or fp32, 16-byte aligned.  Row n is
 *      the target distribution after the prefix plus the path root..n; row 0
 *      belongs to the root (the last accepted token).
 *  node_tokens   [B, N] int32 device; column n-1 holds node n's token.
 *  parent        [N+1] int32 HOST array, parent[0] = -1, 0 <= parent[n] < n
 *      (level order, as spec_tree_from_choices returns).  Shared by all requests.
 *  max_depth     row stride minus one of out_path / out_tokens; must be at
 *      least the tree's depth.
 *  Node n is accepted iff its parent is accepted and node_tokens[n] equals the
 *  argmax of row parent[n] (lowest index on ties); the root is accepted.  The
 *  chosen node n* is the deepest accepted node, smallest index on ties.
 *  out_path   [B, max_depth+1] int32 device: root, ..., n*, then -1.
 *  out_tokens [B, max_depth+1] int32 device: the path's tokens (excluding the
 *      root), then argmax of row n*, then -1.
 *  out_len    [B] int32 device: tokens emitted = depth(n*) + 1.
 *  Sizes: 1 <= B, 0 <= N <= SPEC_MAX_ROWS-1, 1 <= V < 2^30.
 */
spec_status_t spec_verify_tree(const void *target_logits, spec_dtype_t dtype,
                               const int32_t *node_tokens, const int32_t *parent, int B, int N,
                               int V, int max_depth, int32_t *out_path, int32_t *out_tokens,
                               int32_t *out_len, int32_t *d_status, void *workspace,
                               size_t workspace_bytes, void *stream);

/*
 * Sampled token-tree verification (EAGLE-3 review, "EAGLE-3 inference" step
 * 4: with sampling, min(1, p/q) acceptance and residual correction keep the
 * target distribution).  The pages give no rule for siblings; this one walks
 * from the root and tests the children of the current node c in index order:
 * child n with token x is accepted iff q_c(x) == 0 or u_accept[b, n-1] <
 * p'(x) / q_c(x), where p' starts as softmax(z_c / T) and, after each rejected
 * sibling, becomes norm(max(0, p' - q_c)) (unchanged if that has no mass).
 * An accepted child becomes the current node.  When no child of c is
 * accepted, or c is a leaf, one token is drawn from p' by inverse CDF with
 * u_sample[b, c] (the smallest j whose prefix mass exceeds u * total).  With
 * the children of c drawn i.i.d. from q_c this emits tokens with the target's
 * law.  A child token outside [0, V) is rejected (SPEC_STATUS_TOKEN_RANGE).
 *
 *  target_logits [B, N+1, V] device, bf16 or fp32, 16-byte aligned: row n is
 *      the target distribution after the path root..n.
 *  draft_probs   [B, N+1, V] fp32 device, 16-byte aligned: row c is the
 *      distribution the children of node c were drawn from (rows of leaves
 *      are not read).  NULL allowed only when N == 0.
 *  node_tokens   [B, N] int32 device, column n-1 = node n's token.
 *  parent        [N+1] int32 HOST, parent[0] = -1, 0 <= parent[n] < n.
 *  temperature   [B] fp32 device, T > 0 (otherwise SPEC_STATUS_BAD_TEMPERATURE
 *      and T = 1 for that request).
 *  u_accept      [B, N] fp32 device in [0, 1), column n-1 for node n's test.
 *  u_sample      [B, N+1] fp32 device in [0, 1), indexed by the node where the
 *      walk stops.
 *  out_path / out_tokens [B, max_depth+1] int32 device and out_len [B], as in
 *      spec_verify_tree: the walk's nodes from the root, the accepted tokens
 *      then the drawn one, -1 padded; out_len = accepted + 1.
 *  d_status      one int32 device word or NULL (SPEC_STATUS_* bits).
 *  No workspace.  Sizes: 1 <= B, 0 <= N <= SPEC_MAX_ROWS-1, max_depth at least
 *  the tree's depth, 1 <= V <= 360448 (bf16) or 300288 (fp32).
 */
spec_status_t spec_verify_tree_sampled(const void *target_logits, spec_dtype_t dtype, const float *draft_probs,
                                       const int32_t *node_tokens, const int32_t *parent, const float *temperature,
                                       const float *u_accept, const float *u_sample, int B, int N, int V,
                                       int max_depth, int32_t *out_path, int32_t *out_tokens, int32_t *out_len,
                                       int32_t *d_status, void *stream);

/*
 * Next-step preparation after verification (vLLM EAGLE walkthrough, "slot
 * mapping and KV-cache management", which names the next-step helpers, and
 * the EAGLE-3 review, "EAGLE-3 inference" step 5: drafting restarts from the
 * confirmed prefix).  Request b verified rows 0..k at sequence positions
 * positions[b]..positions[b]+k and accepted a = num_accepted[b] drafts.
 *
 *  out_tokens    [B, out_stride] int32 device: the verify step's output tokens.
 *  num_accepted  [B] int32 device (for a tree: out_len - 1).  An a outside
 *      [0, min(out_stride-1, k_b)] is clamped and sets SPEC_STATUS_BAD_OFFSETS
 *      (k_b = rows_per_req - 1, or cu[b+1] - cu[b] when ragged).
 *  positions     [B] int32 device: sequence position of row 0.
 *  block_table   [B, max_blocks] int32 device (may be NULL when P_next == 0):
 *      block ids of each request's KV cache, block_size slots a block.
 *  rows_per_req / cu_num_draft_tokens: where request b's rows start in the
 *      flat target rows: b * rows_per_req, or cu[b] + b when cu ([B+1] int32
 *      device) is given.
 *  hidden_in     [rows, row_bytes] device or NULL: the target's hidden states,
 *      one row per verified position (all B * rows_per_req, or cu[B] + B, rows).
 *  Outputs (device): next_token[b] = out_tokens[b][a]; next_position[b] =
 *  positions[b] + a + 1; next_slots [B, P_next] int64: slot of position
 *  next_position + j, block_table[b][pos / block_size] * block_size +
 *  pos % block_size, or padding_slot_id past the table or for a negative
 *  entry (SPEC_STATUS_SLOT_RANGE); last_row[b] (may be NULL) = the flat row of
 *  the last accepted position, row0(b) + a; hidden_out [B, row_bytes] = that
 *  row of hidden_in.
 *  Sizes: B >= 0, out_stride >= 1, block_size >= 1, P_next >= 0.
 */
spec_status_t spec_prepare_next_step(const int32_t *out_tokens, int out_stride, const int32_t *num_accepted,
                                     const int32_t *positions, const int32_t *block_table, int max_blocks,
                                     int block_size, int B, int P_next, int rows_per_req,
                                     const int32_t *cu_num_draft_tokens, const void *hidden_in, int64_t row_bytes,
                                     int64_t padding_slot_id, int32_t *next_token, int32_t *next_position,
                                     int64_t *next_slots, int32_t *last_row, void *hidden_out, int32_t *d_status,
                                     void *stream);

/*
 * Tree KV compaction (EAGLE-3 review, "EAGLE-3 inference" step 5: only the
 * accepted path's KV is kept).  After a tree verify whose node n wrote its KV
 * row into slot slot_mapping[b][n], depth i of the accepted path
 * (path[b][i], i = 1 .. out_len[b]-1) moves to slot_mapping[b][i], the slot
 * of chain position i; every destination receives its source's row as it was
 * before the call.  Afterwards the chain-mode slot fix-up with
 * num_accepted = out_len - 1 describes the cache.
 *
 *  kv            [num_slots, row_bytes] device, 16-byte aligned, row_bytes a
 *      multiple of 16 (one token's KV across the layers and heads it covers).
 *  slot_mapping  [B, slot_stride] int64 device (slot_stride = N + 1).
 *  path          [B, path_stride] int32 device, out_len [B] int32 device, as
 *      spec_verify_tree / spec_verify_tree_sampled return them.  A path whose
 *      node indices do not start at 0 and strictly increase leaves its request
 *      untouched (SPEC_STATUS_BAD_OFFSETS); a slot outside [0, num_slots)
 *      skips that row (SPEC_STATUS_SLOT_RANGE).
 *  Sizes: B >= 0, 1 <= path_stride <= SPEC_MAX_ROWS.
 */
spec_status_t spec_compact_tree_kv(void *kv, int64_t num_slots, int64_t row_bytes, const int64_t *slot_mapping,
                                   int slot_stride, const int32_t *path, int path_stride, const int32_t *out_len,
                                   int B, int32_t *d_status, void *stream);

/*
 * KV slot_mapping fix-up, in place on [B, P] int64 device memory.
 *  Chain mode (num_accepted != NULL, path == NULL): entry j of request b keeps
 *    its value iff j <= num_accepted[b] (row 0 is the last accepted token,
 *    whose KV is written this step); other entries become padding_slot_id.
 *  Tree mode (path != NULL): entry j keeps its value iff j == 0 or j occurs in
 *    path[b, 0..path_stride).  Entries of accepted nodes off the chosen path
 *    are padded too.
 *  Kept entries are not written.  num_accepted / path are device arrays.
 */
spec_status_t spec_fixup_slots(int64_t *slot_mapping, int B, int P, const int32_t *num_accepted,
                               const int32_t *path, int path_stride, int64_t padding_slot_id,
                               void *stream);

/*
 * Slot_mapping fix-up for ragged chains, in place on packed int64 device
 * memory of total_drafts + B entries: request b's k_b + 1 slots start at
 * cu_num_draft_tokens[b] + b, and slot j of request b keeps its value iff
 * j <= num_accepted[b]; the others become padding_slot_id.
 */
spec_status_t spec_fixup_slots_ragged(int64_t *slot_mapping, int B, const int32_t *cu_num_draft_tokens,
                                      int total_drafts, const int32_t *num_accepted,
                                      int64_t padding_slot_id, void *stream);

/*
 * n-gram lookup drafting (serving-book chapter, table of draft sources, row
 * "n-gram lookup": find, in the prompt or the text generated so far, a span
 * equal to the current ending and use what follows it as the draft; no model).
 *
 *  tokens  [B, Lmax] int32 device: row b holds sequence b (prompt + generated)
 *      in its first lengths[b] entries.
 *  lengths [B] int32 device (values outside [0, Lmax] are clamped).
 *  For each sequence s of length L: the longest n in [n_min, n_max] such that
 *  the ending s[L-n..L-1] also occurs ending at some e < L-1, and among those
 *  occurrences the latest e; the draft is s[e+1..], at most k tokens.
 *  out_draft [B, k] int32 device: the draft, -1 padded.
 *  out_count [B] int32 device: draft length (0 when nothing matches).
 *  out_match_len, out_match_end [B] int32 device, may be NULL: n and e
 *      (0 and -1 when nothing matches).
 *  Sizes: B, Lmax >= 0; 1 <= n_min <= n_max <= 64; k >= 0.
 */
spec_status_t spec_ngram_propose(const int32_t *tokens, const int32_t *lengths, int B, int Lmax, int n_min,
                                 int n_max, int k, int32_t *out_draft, int32_t *out_count,
                                 int32_t *out_match_len, int32_t *out_match_end, void *stream);

/*
 * Host helper (no device work): tree_choices -> parent[] and level metadata,
 * following the vLLM EAGLE walkthrough ("tree drafting in detail").
 *  flat / lens / n: the n tuples of tree_choices, concatenated in `flat`,
 *      lens[i] = length of tuple i.  Tuples must be in level order and each
 *      tuple's prefix must appear before it.
 *  parent [n+1] (out): parent[0] = -1; node i+1 is tuple i; its parent is the
 *      node of the tuple without its last entry (the root for length 1).
 *  cu_per_level, child_per_level [depth] (out, may be NULL; capacity
 *      SPEC_MAX_ROWS): cumulative node count per level and count[l] /
 *      count[l-1] (count[0] at level 0).
 *  depth (out): length of the last tuple.
 */
spec_status_t spec_tree_from_choices(const int32_t *flat, const int32_t *lens, int n,
                                     int32_t *parent, int32_t *cu_per_level,
                                     int32_t *child_per_level, int *depth);

/*
 * spec_verify_chain_noalloc -- spec_verify_chain for callers that cannot
 * allocate device memory.  (The pages have no counterpart: this is a
 * deployment convenience, not part of the method.)
 *
 * Who needs it: code that owns no device allocator and so cannot create the
 * workspace spec_verify_chain asks for -- for example a plugin inside a serving
 * runtime whose device memory is entirely owned and budgeted by the runtime's
 * own allocator, or a C caller that is handed only device pointers to its
 * inputs and outputs.  Such callers pass inputs and outputs exactly as for
 * spec_verify_chain (same meaning, layout and checks), and the library uses a
 * fixed scratch array of spec_noalloc_scratch_bytes() (16 MiB) that it
 * reserves in its device module: every GPU on which the library is loaded
 * holds that array until the process exits.  The entry point itself calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 *  - Sizes whose workspace would exceed the scratch (see spec_workspace_bytes)
 *    are rejected with SPEC_ERR_INVALID_ARG before any device work.
 *  - The first call on a device does one-time set-up with that device current
 *    (it looks up the scratch's device address and configures the kernels);
 *    make that first call before any stream capture.
 *  - All calls share the one array, which keeps the previous call's contents:
 *    each call clears the counters it needs (an async memset on `stream`), and
 *    calls that can overlap on the GPU (other streams, other threads) race on
 *    the scratch and must be serialised by the caller.
 */
spec_status_t spec_verify_chain_noalloc(const void *target_logits, spec_dtype_t dtype,
                                        const float *draft_probs, const int32_t *draft_tokens,
                                        const float *temperature, const float *u_accept,
                                        const float *u_sample, int B, int k, int V,
                                        int32_t *out_tokens, int32_t *out_num_accepted,
                                        int32_t *d_status, void *stream);

/* Bytes of the fixed scratch used by spec_verify_chain_noalloc. */
size_t spec_noalloc_scratch_bytes(void);

/* Text of the last error recorded on the calling thread ("" if none). */
const char *spec_last_error(void);

/*
 * Tuning and test settings, process-wide; normal use needs neither.  A call
 * reads them when it sets up its launch, so a call captured in a CUDA graph
 * keeps the values in force at capture time.
 *
 * spec_set_wait_limit_ns: the limit, in nanoseconds, of every wait a kernel of
 * this library makes on other blocks, warps or cluster peers (default
 * 500000000, i.e. 0.5 s; 0 = give up at once unless the awaited event has
 * already happened).  A wait that runs out sets
 * SPEC_STATUS_WAIT_TIMEOUT and the kernel finishes early: the outputs of the
 * requests involved are undefined, bulk copies already in flight are still
 * waited for (with the default limit) before a block exits, and the workspace
 * counters are left zero as after any call.  Returns the previous limit.
 * Tests set the limit to 0 to drive the time-out path; there is no reason to
 * change it otherwise.
 *
 * spec_set_tuning: splits = units each logits row of the persistent chain /
 * greedy-tree kernel is cut into (0 = automatic: whole rows when the batch has
 * about two rows per SM, finer otherwise); ahead = stages that kernel's copy
 * ring keeps in flight (0 = automatic, i.e. all 3; else 2 or 3); path = 0
 * (automatic: sampled padded chains whose per-request thread-block clusters
 * all fit on the GPU at once are verified one cluster per request; greedy
 * trees of at most 64 rows, and greedy padded chains of at most 64 rows with
 * fewer than two rows per SM, by a persistent grid of clusters; the rest by
 * the persistent kernel), 1 (the persistent kernel for every batch) or 2 (as
 * 0, with every greedy padded chain of at most 64 rows on the grid).  Greedy
 * results do not depend on any of them; sampled tokens can differ between the
 * two kernels only where the arithmetic of the accept test or the draw falls
 * within rounding of a decision boundary.  Other values return
 * SPEC_ERR_INVALID_ARG and change nothing.
 */
unsigned long long spec_set_wait_limit_ns(unsigned long long ns);
spec_status_t spec_set_tuning(int splits, int ahead, int path);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
