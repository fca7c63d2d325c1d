/*
 * treespec.h — C ABI of the GB300 tree-attention speculative verification library.
 *
 * One verification step scores a flattened tree of N draft tokens per sequence
 * in a single pass and then accepts the longest draft path the target model
 * agrees with.  The library exposes that step as three calls, each a stream-
 * ordered launch of hand-written sm_103a kernels:
 *
 *   tree_build_ancestry  ancestor bitmasks, depths and positions of the tree
 *   tree_attn_fwd        attention of every tree node over the verified prefix
 *                        (paged KV cache) plus its own ancestors and itself
 *   tree_verify_greedy   greedy argmax of every node's logits and the
 *                        parent-chain acceptance walk
 * and around it:
 *   tree_build_dynamic      rerank a draft's candidate pool into the tree (and
 *                           its masks) in place of tree_build_ancestry
 *   tree_build_ancestry_forest, tree_verify_greedy_forest
 *                           the same for several roots per sequence
 *   tree_verify_stochastic  temperature verification by rejection sampling
 *   tree_commit_accepted    append the accepted path to the paged cache
 *   tree_attn_workspace_size, tree_attn_plan, tree_attn_plan_order, tree_verify_workspace_size
 *                           host-only queries: workspace bytes, split plan
 *
 * Sources (web pages on the method):
 *   [P1] "Tree Attention", inferensys glossary.
 *   [P2] "Tree Attention", zhongzhoutan-coder terms page.
 *   [P3] "Speculative Tree Attention: How Multi-Candidate Draft Models and
 *        Parallel Verification Deliver 4x LLM Speedups", premlal news.
 *
 * Conventions shared by every call
 *   - Every pointer is a DEVICE pointer unless its name ends in _host.
 *   - The caller owns every buffer, workspace included.  The library never
 *     allocates, frees or keeps a pointer past the call.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream) and the call returns without synchronising.
 *   - The return value reports what the host can check before launching:
 *     null pointers, shapes, unsupported sizes, too small a workspace, and
 *     launch errors.  Nothing is launched when it is not TS_OK.
 *   - Data-dependent errors (an invalid tree, a block id outside the pool, an
 *     internal wait that timed out) are written as a ts_status code into the
 *     caller's per-sequence int32 `status` array on the device.  A call never
 *     writes 0 there except tree_build_ancestry(_forest) and tree_build_dynamic,
 *     which (re)initialise it, so one status array can be threaded through a whole
 *     step and read once.
 *   - Index tensors are int32, row-major, densely packed.  bf16 tensors are
 *     16-bit brain-float, row-major, densely packed, 16-byte aligned.
 *   - Supported sizes: 1 <= N <= 256 nodes (W = ceil(N/64) <= 4 mask words),
 *     head_dim D in {64, 128}, Hq = G * Hkv with G in {1, 2, 4, 8, 16},
 *     KV block size any positive multiple of 16.
 *     Anything else returns TS_ERR_UNSUPPORTED.
 */
#ifndef TREESPEC_H_
#define TREESPEC_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TS_API __attribute__((visibility("default")))
#else
#define TS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef int ts_status;

enum {
  TS_OK = 0,
  TS_ERR_NULL = -1,         /* a required pointer is NULL */
  TS_ERR_SHAPE = -2,        /* inconsistent sizes, misaligned pointer, output too short */
  TS_ERR_BAD_TREE = -3,     /* parent array is not a topologically ordered single-root tree */
  TS_ERR_UNSUPPORTED = -4,  /* sizes outside the supported set above */
  TS_ERR_BAD_BLOCK = -5,    /* block table entry outside [0, num_blocks) for a used block */
  TS_ERR_TIMEOUT = -6,      /* an internal pipeline wait gave up (kernel exited early) */
  TS_ERR_CUDA = -7,         /* a CUDA runtime call failed */
  TS_ERR_WORKSPACE = -8     /* workspace NULL or smaller than the *_workspace_size query */
};

/* A cudaStream_t, passed as an opaque pointer so that this header needs no CUDA headers. */
typedef void* ts_stream;

/* Human-readable name of a status code (static string, never NULL). */
TS_API const char* ts_status_str(ts_status st);

/*
 * tree_build_ancestry — tree-causal mask, depths and positions.
 *
 * Defines the ancestry ("tree-causal") mask of [P1] Key Mechanisms > Modified
 * Causal Attention Mask (a node sees its ancestral path to the root and
 * itself, no sibling branch), [P2] How It Works (prefix, self and ancestors
 * only), built as in [P3]'s code listing (build_tree_attention_mask: walk
 * parent pointers to the root), and the "position bookkeeping" of [P2]
 * Tradeoffs.
 *
 *   parent_idx  [B, N] int32.  Node 0 is the root (parent -1); every other node
 *               i has 0 <= parent_idx[i] < i (topological flattening).
 *   prefix_len  [B] int32, verified-prefix length P_b >= 0 of each sequence.
 *   anc_mask    [B, N, W] uint64 out, W = ceil(N/64).  Bit (j mod 64) of word
 *               (j div 64) of row i is set iff node j is i or an ancestor of i.
 *               Bits for j >= N are zero.
 *   depth       [B, N] int32 out, parent steps from the node to the root.
 *   pos         [B, N] int32 out, P_b + depth (the root sits at position P_b).
 *   status      [B] int32 out: TS_OK, or TS_ERR_BAD_TREE (then anc_mask, depth
 *               and pos of that sequence are zero).
 * Returns TS_ERR_NULL / TS_ERR_UNSUPPORTED (N outside [1, 256], B < 1) / TS_ERR_CUDA.
 */
TS_API ts_status tree_build_ancestry(const int32_t* parent_idx, const int32_t* prefix_len, int B, int N,
                              uint64_t* anc_mask, int32_t* depth, int32_t* pos, int32_t* status,
                              ts_stream stream);

/*
 * Arguments of tree_attn_fwd (all pointers device unless *_host).
 *
 *   q           [B, N, Hq, D] bf16, queries of the tree nodes.
 *   k_cache,
 *   v_cache     [num_blocks, Hkv, block_size, D] bf16, the paged verified-prefix
 *               KV pool.  Prefix token t of sequence b, KV head g, is row
 *               (t mod block_size) of block block_table[b, t div block_size].
 *               A contiguous cache is the special case of one block per
 *               sequence: block_size = P rounded up to a multiple of 16 (rows
 *               past P_b are never read into the result), block_table[b] = {b}.
 *   block_table [B, max_blocks] int32; only the first ceil(P_b / block_size)
 *               entries of row b are used (other entries of the row may be
 *               read, never followed).
 *   prefix_len  [B] int32 device copy of P_b; prefix_len_host the same values
 *               in host memory (used to plan the split of the prefix).
 *               0 <= P_b <= 2^30.
 *   k_tree,
 *   v_tree      [B, N, Hkv, D] bf16, keys/values of the tree nodes themselves.
 *   anc_mask    [B, N, W] uint64 from tree_build_ancestry.
 *   pos         [B, N] int32 from tree_build_ancestry (read only when rotary
 *               embedding is requested; must be 0 = off in this version, the
 *               inputs are taken as already positioned).
 *   out         [B, N, Hq, D] bf16 out.
 *   lse         [B, N, Hq] fp32 out (natural-log softmax normaliser) or NULL.
 *   status      [B] int32, error codes are written here (or NULL: not reported).
 *   scale       softmax scale; 0 selects 1/sqrt(D).
 *   Query head h reads KV head h / G (G = Hq / Hkv, consecutive grouping).
 */
typedef struct ts_attn_params {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* prefix_len_host;
  const void* k_tree;
  const void* v_tree;
  const uint64_t* anc_mask;
  const int32_t* pos;
  void* out;
  float* lse;
  int32_t* status;
  int B, N, Hq, Hkv, D;
  int block_size, num_blocks, max_blocks;
  float scale;
  float rope_theta;
} ts_attn_params;

/*
 * Bytes of device workspace tree_attn_fwd needs for these sizes: 256 bytes
 * for the attention kernel's work-item counter, then the split-prefix
 * partial results.  Host-only: launches nothing, safe without a GPU.
 * Returns 0 for arguments tree_attn_fwd would reject.
 */
TS_API size_t tree_attn_workspace_size(const ts_attn_params* p);

/*
 * tree_attn_plan — how tree_attn_fwd will cut the work for these arguments
 * (host only, launches nothing).  The prefix of every (sequence, KV head,
 * 128-row tile) of T 128-token tiles is cut into ceil(T / *chunk_tiles)
 * splits of near-equal length (split s starts at tile floor(T s / splits));
 * *max_splits is the split count of the longest sequence (the grid's split
 * extent), and *tree_split is 1 when the tree block runs as a split of its
 * own rather than on the last prefix split.  With *max_splits == 1 the
 * attention kernel writes `out` itself; otherwise the splits' partials are
 * merged by a second kernel.  Each output pointer may be NULL.
 * Returns TS_ERR_NULL / TS_ERR_SHAPE / TS_ERR_UNSUPPORTED like tree_attn_fwd.
 */
TS_API ts_status tree_attn_plan(const ts_attn_params* p, int32_t* chunk_tiles, int32_t* max_splits,
                                int32_t* tree_split);

/*
 * tree_attn_plan_order — the order in which the attention kernel takes its
 * work items for these arguments (host only, launches nothing): every
 * (sequence, split) pair once, longest first by prefix_len_host (ties in
 * sequence, then split order).  Entry e of `order` is
 * (b << 24) | (split << 15) | first_tile, first_tile being the split's first
 * prefix tile by prefix_len_host (0x7fff when larger; 0 for a split with no
 * prefix tiles).  *count receives the number of pairs, B * max_splits, or 0
 * when there are more than 256 (the kernel then takes the items sequence by
 * sequence, split by split); at most `cap` entries are written.  `order` may
 * be NULL when cap is 0.
 * Returns TS_ERR_NULL / TS_ERR_SHAPE / TS_ERR_UNSUPPORTED like tree_attn_fwd,
 * and TS_ERR_SHAPE when cap is negative or smaller than *count.
 */
TS_API ts_status tree_attn_plan_order(const ts_attn_params* p, uint32_t* order, int32_t cap, int32_t* count);

/*
 * tree_attn_fwd — the attention layer of the batched verification pass
 * ([P1] Key Mechanisms > Batched Parallel Verification: every node of the
 * tree is scored in one pass, each attending to its own root path; [P2] How
 * It Works: a node attends to the verified prefix, itself and its ancestors).
 *
 * For sequence b, node i, query head h (KV head g = h / G):
 *   keys = prefix tokens 0..P_b-1  ++  tree nodes j with bit j of anc_mask[b,i]
 *   out[b,i,h] = softmax(scale * q . k) . v over those keys, lse likewise.
 *
 * workspace: device buffer of at least tree_attn_workspace_size(p) bytes,
 * 256-byte aligned, ZERO-FILLED before its first use: its first 256 bytes
 * hold the counter from which the attention kernel's CTAs (one per SM) take
 * their work items, and every call, a timed-out one included, leaves them
 * zero again; the rest is scratch for this call only.  Calls sharing one
 * workspace must be stream-ordered.
 * Returns TS_ERR_NULL / TS_ERR_SHAPE / TS_ERR_UNSUPPORTED / TS_ERR_WORKSPACE /
 * TS_ERR_CUDA; a block id outside the pool sets status[b] = TS_ERR_BAD_BLOCK
 * (block 0 is read in its place), a timed-out internal wait sets
 * TS_ERR_TIMEOUT for the sequence of every work item (one 128-row tile of
 * one (sequence, KV head) and one split of its prefix) that the CTA whose
 * wait ran out had taken and not finished.
 */
TS_API ts_status tree_attn_fwd(const ts_attn_params* p, void* workspace, size_t workspace_bytes,
                        ts_stream stream);

/*
 * tree_attn_fwd_stall_test — for testing the failure path only; the pages
 * have no counterpart.  Runs exactly what tree_attn_fwd runs, except that
 * every work item of sequence `stall_seq` stops its key stream before its
 * tile `stall_tile` (128-token tiles, counted from the start of the item's
 * split; the tree block's tiles come last): those loads are never issued, so
 * the wait for them runs out after `wait_limit_us` microseconds, and every
 * other bounded wait of the call uses the same limit.  A CTA whose wait runs
 * out lets its loads and MMAs in flight finish, frees its tensor memory and
 * sets status[b] = TS_ERR_TIMEOUT for the sequence b of every item it had
 * taken and not finished (stall_seq's among them); items with fewer tiles run
 * to the end.  The outputs of those sequences are then unspecified; the other
 * sequences' outputs are those of tree_attn_fwd (with a limit far above
 * their run time), the workspace's counter is back at zero, and the device
 * stays usable.
 * Returns TS_ERR_SHAPE for stall_seq outside [0, B) or stall_tile < 0,
 * TS_ERR_UNSUPPORTED for wait_limit_us outside [100, 10^6], else as
 * tree_attn_fwd.
 */
TS_API ts_status tree_attn_fwd_stall_test(const ts_attn_params* p, void* workspace, size_t workspace_bytes,
                                          int stall_seq, int stall_tile, uint32_t wait_limit_us,
                                          ts_stream stream);

/*
 * tree_attn_fwd_ctas_test — for testing only; the pages have no counterpart.
 * tree_attn_fwd runs one attention CTA per SM, each taking work items until
 * none is left; this call caps the CTAs at `max_ctas` (>= 1), so that small
 * cases also send many items, empty splits among them, through each CTA.
 * With stall_seq >= 0 it also stalls that sequence like
 * tree_attn_fwd_stall_test; with stall_seq == -1 nothing is stalled and
 * stall_tile is ignored.  Every bounded wait uses wait_limit_us.
 * Returns TS_ERR_UNSUPPORTED for max_ctas < 1 or wait_limit_us outside
 * [100, 10^6], TS_ERR_SHAPE for stall_seq outside [-1, B) or (stall_seq >= 0
 * and stall_tile < 0), else as tree_attn_fwd.
 */
TS_API ts_status tree_attn_fwd_ctas_test(const ts_attn_params* p, void* workspace, size_t workspace_bytes,
                                         int max_ctas, int stall_seq, int stall_tile, uint32_t wait_limit_us,
                                         ts_stream stream);

/*
 * Bytes of device workspace tree_verify_greedy needs (a packed argmax key per
 * node and an arrival counter per sequence).  Host-only.
 */
TS_API size_t tree_verify_workspace_size(int B, int N, int V);

/*
 * tree_verify_greedy — greedy target prediction and acceptance.
 *
 * [P3] code listing, verify_candidate_tree: the target's prediction at a node
 * is the argmax of its logits.  [P1] Key Mechanisms > Multi-Token Acceptance &
 * Rollback and [P2] How It Works: the longest valid path from the root is
 * accepted, up to the first rejection.  A node's logits predict its children:
 * node c >= 1 is accepted iff every node x on its chain up to the root
 * satisfies draft_tokens[x] == argmax(target_logits[parent(x)]).  The root is
 * the last verified token and is always accepted.  n* is the deepest accepted
 * node (ties: smallest index).
 *
 *   draft_tokens  [B, N] int32 draft token id of each node (the root's is unused).
 *   target_logits [B, N, V] fp32, finite or -inf (a row of nothing but -inf
 *                 gives index 0); the argmax takes the first index on ties.
 *   parent_idx    [B, N] int32 as for tree_build_ancestry.
 *   accepted      [B, max_depth + 1] int32 out: node ids root .. n*, then -1.
 *   accept_len    [B] int32 out: depth(n*), the number of accepted drafts.
 *   bonus         [B] int32 out: argmax of n*'s logits, the target's next token.
 *   argmax_out    [B, N] int32 out, every node's argmax (required).
 *   status        [B] int32: TS_ERR_BAD_TREE for an invalid tree; TS_ERR_SHAPE
 *                 when depth(n*) > max_depth (accepted row left all -1,
 *                 accept_len and bonus still written).
 *   workspace     at least tree_verify_workspace_size(B, N, V) bytes, 256-byte
 *                 aligned, ZERO-FILLED before its first use; every call leaves
 *                 it zero-filled again, so it can be reused by stream-ordered
 *                 calls without clearing.
 * Returns TS_ERR_NULL / TS_ERR_UNSUPPORTED (N outside [1, 256], V < 1,
 * max_depth < 0) / TS_ERR_WORKSPACE / TS_ERR_CUDA.
 */
TS_API ts_status tree_verify_greedy(const int32_t* draft_tokens, const float* target_logits,
                             const int32_t* parent_idx, int B, int N, int V, int max_depth,
                             int32_t* accepted, int32_t* accept_len, int32_t* bonus,
                             int32_t* argmax_out, int32_t* status, void* workspace,
                             size_t workspace_bytes, ts_stream stream);

/*
 * tree_commit_accepted — append the accepted path's keys/values to the cache.
 *
 * [P1] Key Mechanisms > Speculative KV Cache Reuse (the tree's keys/values are
 * reused), Multi-Token Acceptance & Rollback (keep the accepted path, discard
 * the rejected branches) and Integration with Speculative Decoding (append the
 * accepted prefix and continue from the new state).  The root (the last
 * verified token, attended at position P_b) and the accepted drafts x1..n*
 * become prefix tokens P_b .. P_b + L; rejected branches need no work, their
 * keys/values never entered the cache.
 *
 *   k_tree, v_tree   [B, N, Hkv, D] bf16, the tree's keys/values (as given to
 *                    tree_attn_fwd).
 *   accepted         [B, max_depth + 1] int32 and accept_len [B] int32 from
 *                    tree_verify_greedy.
 *   prefix_len       [B] int32, P_b before the commit; a sequence with P_b
 *                    outside [0, 2^30] commits nothing and keeps it.
 *   k_cache, v_cache [num_blocks, Hkv, block_size, D] bf16, written at rows
 *                    (t mod block_size) of blocks block_table[b, t div
 *                    block_size] for t = P_b .. P_b + L; nothing else changes.
 *                    The caller provides blocks for every position committed.
 *   new_prefix_len   [B] int32 out: P_b + L + 1 (may be the prefix_len array).
 *   status           [B] int32 in/out (or NULL): a sequence whose status is
 *                    not 0 commits nothing and keeps P_b; a destination block
 *                    or node id out of range commits nothing for that
 *                    sequence and sets TS_ERR_BAD_BLOCK.
 * Returns TS_ERR_NULL / TS_ERR_SHAPE / TS_ERR_UNSUPPORTED (D not 64 or 128) /
 * TS_ERR_CUDA.
 */
TS_API ts_status tree_commit_accepted(const void* k_tree, const void* v_tree, const int32_t* accepted,
                                      const int32_t* accept_len, const int32_t* prefix_len, void* k_cache,
                                      void* v_cache, const int32_t* block_table, int B, int N, int Hkv, int D,
                                      int block_size, int num_blocks, int max_blocks, int max_depth,
                                      int32_t* new_prefix_len, int32_t* status, ts_stream stream);

/*
 * tree_verify_stochastic — temperature verification by rejection sampling.
 *
 * [P3] Production Inference Runtimes section: each accepted token is checked
 * against the target model's own distribution by rejection sampling, so the
 * emitted tokens follow the target exactly; [P3] code listing (comment of
 * verify_candidate_tree): greedy or temperature-sampled target predictions;
 * [P1] Key Mechanisms > Multi-Token Acceptance & Rollback.  The pages give no
 * rule for several drafts under one node; this call takes the siblings, drawn
 * from the draft distribution without replacement, in index order:
 *   r = softmax(target_logits[u] / temperature), q' = draft_probs[u];
 *   child c (token x) is accepted iff coins[c] * q'(x) < r(x), and the walk
 *   moves to c;  otherwise r <- max(r - q', 0) renormalised (unchanged if no
 *   mass is left), q'(x) <- 0 and q' is renormalised to the remaining mass.
 * The walk ends at a leaf or when every child of the current node is
 * rejected; the bonus token is then drawn from r by inversion: the smallest v
 * with r(0) + ... + r(v) > coins[0].
 *
 *   draft_tokens  [B, N] int32; the root's entry is unused, the others must lie
 *                 in [0, V).  The children of a node are taken to have been
 *                 drawn without replacement from that node's draft_probs row.
 *   target_logits [B, N, V] fp32, finite.
 *   draft_probs   [B, N, V] fp32 draft probabilities q_u (each row sums to 1);
 *                 only rows of visited nodes with children are read.
 *   parent_idx    [B, N] int32 as for tree_build_ancestry.
 *   coins         [B, N] fp32 uniforms in [0, 1): coins[b, c] decides child c,
 *                 coins[b, 0] draws the bonus token.  The caller owns the
 *                 random numbers.
 *   temperature   > 0 and finite.
 *   accepted      [B, max_depth + 1] int32 out: node ids root .. n*, then -1.
 *   accept_len    [B] int32 out: number of accepted drafts.
 *   bonus         [B] int32 out: the token drawn after n*.
 *   status        [B] int32; only errors are written: TS_ERR_BAD_TREE for an
 *                 invalid tree or a draft token outside [0, V) (row all -1,
 *                 zeros), TS_ERR_SHAPE when the accepted path is longer than
 *                 max_depth (row all -1, accept_len and bonus written),
 *                 TS_ERR_TIMEOUT when an internal copy did not complete.
 * fp32 arithmetic: decisions within fp32 rounding of a threshold may differ
 * from an exact computation (the bonus by one token with mass at an
 * inversion boundary).  Reads only the rows of the nodes the walk visits.
 * No workspace.  The first call on a device sets kernel attributes; make it
 * outside any stream capture.  Returns TS_ERR_NULL / TS_ERR_UNSUPPORTED (N
 * outside [1, 256], V outside [1, 409600] (204800 on GPUs without 16-CTA
 * clusters), B > 65535, max_depth < 0, temperature not positive and finite) /
 * TS_ERR_CUDA.
 */
TS_API ts_status tree_verify_stochastic(const int32_t* draft_tokens, const float* target_logits,
                                        const float* draft_probs, const int32_t* parent_idx, const float* coins,
                                        int B, int N, int V, int max_depth, float temperature, int32_t* accepted,
                                        int32_t* accept_len, int32_t* bonus, int32_t* status, ts_stream stream);

/*
 * tree_build_dynamic — choose the tree to verify from a draft's candidate
 * pool, flatten it, and build its ancestry masks, depths and positions (the
 * outputs of tree_build_ancestry) in one launch.
 *
 * [P2] Common Confusions: the tree shape may be selected dynamically; Where
 * It Appears (EAGLE-2): the tree changes per context and the ancestry mask is
 * built after reranking.  [P1] Key Mechanisms > Tree-Structured Candidate
 * Generation.  The pages give no procedure; this call takes:
 *   value(root) = 0, value(c) = value(parent(c)) + pool_logp[c], accumulated in
 *   fp32 from the root down; the root and the N - 1 candidates of highest value
 *   (ties: smaller pool index) are kept, in pool order.  With log-probabilities
 *   <= 0 the kept set contains every kept node's parent.  Under the model in
 *   which a draft token is accepted with the probability the draft gave it,
 *   the kept tree maximises the expected number of accepted tokens over all
 *   N-node trees cut from the pool.
 *
 *   pool_parent   [B, M] int32: topological (pool_parent[b,0] = -1 is the
 *                 root, the last verified token; 0 <= pool_parent[b,c] < c).
 *   pool_logp     [B, M] fp32: the draft's log-probability of each candidate
 *                 given its parent, <= 0 (-inf allowed); the root's is unused.
 *   pool_token    [B, M] int32: each candidate's token.
 *   prefix_len    [B] int32: P_b, for the positions.
 *   parent_idx    [B, N] int32 out: the kept tree, node k = k-th kept candidate.
 *   draft_tokens  [B, N] int32 out: their tokens.
 *   sel_index     [B, N] int32 out: their pool indices (to gather the draft's
 *                 other per-candidate data).
 *   anc_mask, depth, pos: out, as tree_build_ancestry for the kept tree.
 *   status        [B] int32 out, (re)initialised like tree_build_ancestry:
 *                 0, or TS_ERR_BAD_TREE for a pool that is not topological or
 *                 has a positive or NaN log-probability (that sequence then
 *                 gets a star tree: every node a child of the root).
 * Returns TS_ERR_NULL / TS_ERR_SHAPE (B < 1, N < 1, M < N) /
 * TS_ERR_UNSUPPORTED (N > 256, M > 1024) / TS_ERR_CUDA.
 */
TS_API ts_status tree_build_dynamic(const int32_t* pool_parent, const float* pool_logp, const int32_t* pool_token,
                                    const int32_t* prefix_len, int B, int M, int N, int32_t* parent_idx,
                                    int32_t* draft_tokens, int32_t* sel_index, uint64_t* anc_mask, int32_t* depth,
                                    int32_t* pos, int32_t* status, ts_stream stream);

/*
 * Forests: several draft trees in one flattened sequence.
 *
 * [P3] The Future of Reasoning: the verifier evaluates whole forests of
 * candidate continuations in parallel.  The pages give no rule; the tree rules
 * carry over as follows.  Node 0 is a root (parent -1); any later node may be
 * another root (parent -1) or have a parent with a smaller index.  Every root
 * is a given token attended at position P_b, like a tree's root.  A node's
 * mask, depth and position follow its chain to its own root, so nodes of
 * different trees never see each other; tree_attn_fwd and
 * tree_commit_accepted need nothing new.  Acceptance: every root is accepted;
 * node c is accepted iff every node x on its chain below its root has
 * draft[x] == argmax(logits[parent(x)]); n* is the deepest accepted node of the
 * forest (ties: smallest index); the accepted row runs from n*'s root to n*.
 *
 * tree_build_ancestry_forest and tree_verify_greedy_forest take exactly the
 * arguments of tree_build_ancestry and tree_verify_greedy (same workspace
 * size) and report the same status codes; only the validity rule and the
 * root of a chain differ.
 */
TS_API ts_status tree_build_ancestry_forest(const int32_t* parent_idx, const int32_t* prefix_len, int B, int N,
                                            uint64_t* anc_mask, int32_t* depth, int32_t* pos, int32_t* status,
                                            ts_stream stream);
TS_API ts_status tree_verify_greedy_forest(const int32_t* draft_tokens, const float* target_logits,
                                           const int32_t* parent_idx, int B, int N, int V, int max_depth,
                                           int32_t* accepted, int32_t* accept_len, int32_t* bonus,
                                           int32_t* argmax_out, int32_t* status, void* workspace,
                                           size_t workspace_bytes, ts_stream stream);

/* Size of the library-owned scratch behind tree_verify_greedy_noalloc. */
#define TS_VERIFY_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)

/*
 * tree_verify_greedy_noalloc — tree_verify_greedy for callers that cannot
 * allocate.  The pages have no counterpart to this call; it exists for users
 * of this library that are not allowed to allocate device memory or are not
 * given a workspace: a plugin inside another inference engine that receives
 * only its input and output buffers, or a latency-critical loop in which a
 * cudaMalloc (which may synchronise the whole device) is not acceptable.
 *
 * Arguments, outputs and status codes are those of tree_verify_greedy, minus
 * the workspace.  The scratch is a fixed array of
 * TS_VERIFY_NOALLOC_SCRATCH_BYTES (4 MiB) inside the library; every GPU that
 * loads the library holds it until the process exits.  Sizes whose scratch
 * (tree_verify_workspace_size(B, N, V)) exceeds that limit return
 * TS_ERR_WORKSPACE before anything is launched.  The need is 8 bytes a
 * node and 4 a sequence (each part rounded up to 256 bytes), whatever the
 * vocabulary: 32 KiB for B*N = 4096 nodes, so the limit is B*N of about
 * 520000 nodes.
 *
 * - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 * - The first call on a device looks up the array's device address (with the
 *   device that owns `stream` current) and caches it; make that first call
 *   before any stream capture.
 * - Each call clears the part of the scratch it uses on `stream` (an async
 *   memset) before its kernel.
 * - Every call on a device shares the one array: calls that can overlap on
 *   the GPU (different streams without ordering between them) race and give
 *   wrong results.  Order them on one stream.
 */
TS_API ts_status tree_verify_greedy_noalloc(const int32_t* draft_tokens, const float* target_logits,
                                            const int32_t* parent_idx, int B, int N, int V, int max_depth,
                                            int32_t* accepted, int32_t* accept_len, int32_t* bonus,
                                            int32_t* argmax_out, int32_t* status, ts_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* TREESPEC_H_ */
