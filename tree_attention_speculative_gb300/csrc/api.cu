// C ABI: argument validation, split planning, launches.  See include/treespec.h.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.cuh"

namespace ts {
namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
inline size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

bool supported_group(int G) { return G == 1 || G == 2 || G == 4 || G == 8 || G == 16; }

// Host validation shared by the workspace query and the launch.  Touches no
// device memory and makes no CUDA call.
ts_status check_attn(const ts_attn_params* p) {
  if (!p) return TS_ERR_NULL;
  if (!p->q || !p->k_cache || !p->v_cache || !p->block_table || !p->prefix_len ||
      !p->prefix_len_host || !p->k_tree || !p->v_tree || !p->anc_mask || !p->out)
    return TS_ERR_NULL;
  if (p->B < 1 || p->N < 1 || p->Hq < 1 || p->Hkv < 1 || p->num_blocks < 1 || p->max_blocks < 1 ||
      p->block_size < 1)
    return TS_ERR_SHAPE;
  if (p->N > MAX_NODES) return TS_ERR_UNSUPPORTED;
  if (p->D != 64 && p->D != 128) return TS_ERR_UNSUPPORTED;
  if (p->Hq % p->Hkv != 0) return TS_ERR_SHAPE;
  if (!supported_group(p->Hq / p->Hkv)) return TS_ERR_UNSUPPORTED;
  const int bs = p->block_size;
  if (bs % 16 != 0) return TS_ERR_UNSUPPORTED;
  if (p->rope_theta != 0.f) return TS_ERR_UNSUPPORTED;
  if (!(p->scale >= 0.f) || std::isinf(p->scale)) return TS_ERR_SHAPE;
  for (int b = 0; b < p->B; ++b) {
    const int P = p->prefix_len_host[b];
    if (P < 0) return TS_ERR_SHAPE;
    if (P > (1 << 30)) return TS_ERR_UNSUPPORTED;  // keeps every token index in 32-bit arithmetic
    if (ceil_div(P, bs) > p->max_blocks) return TS_ERR_SHAPE;
  }
  if (!aligned16(p->q) || !aligned16(p->k_cache) || !aligned16(p->v_cache) || !aligned16(p->k_tree) ||
      !aligned16(p->v_tree) || !aligned16(p->out))
    return TS_ERR_SHAPE;
  return TS_OK;
}

// Split plan.  Every (unit, row tile) is one chain of 128-token KV tiles; a
// sequence's prefix is cut into ceil(tiles / chunk_tiles) splits of near-equal
// length (at most `chunk_tiles` tiles each).  The tree block rides
// on the last prefix split of a unit, or (tree_split) on a CTA of its own that
// runs beside the prefix splits.  The attention kernel holds one CTA per SM,
// so the time of a plan is about
//     waves * (chunk + per-CTA overhead) [+ tree tiles]
//       [+ the combine kernel's launch + cost of the partials, when split],
// in units of one tile's work on one SM (about 0.5 us).  The partials are
// written and read back once (bf16 O + fp32 lse per split, about 2D + 4 bytes
// a row) and priced at twice those bytes at the measured HBM rate: at the
// plain price the planner picked 7 splits for the batched-serving workload
// (16 sequences, paged prefixes of 1-16K), which ran 5% slower than 4.  The
// plan with the smallest estimate wins; ties keep the tree on the last prefix
// split.
AttnPlan plan_attn(const ts_attn_params* p) {
  AttnPlan pl{};
  const int G = p->Hq / p->Hkv;
  pl.row_tiles = ceil_div(p->N * G, ROW_TILE);
  const int tree_tiles = ceil_div(p->N, KV_TILE);
  int max_tiles = 1;
  for (int b = 0; b < p->B; ++b) {
    const int t = prefix_tiles(p->prefix_len_host[b]);
    max_tiles = t > max_tiles ? t : max_tiles;
  }
  const double rows = (double)p->B * p->N * p->Hq;
  const double tile_bytes_equiv = 3.6e6;  // HBM bytes moved in one tile-time
  const double cta_overhead = 1.5;        // prologue + epilogue, in tile-times
  // A split plan also runs the combine kernel: its launch, its wait for the
  // attention kernel and its own round trip cost about 2 us whatever its size.
  const double combine_launch = 4.0;
  double best = 1e300;
  int best_chunk = max_tiles, best_ts = 0;
  for (int ts = 0; ts <= 1; ++ts) {
    for (int s = 1; s <= 256; ++s) {
      const int chunk = ceil_div(max_tiles, s);
      if (s > 1 && chunk == ceil_div(max_tiles, s - 1)) continue;
      long long ctas = 0;
      int splits = 1;
      for (int b = 0; b < p->B; ++b) {
        const int ns = num_splits(p->prefix_len_host[b], chunk, ts);
        ctas += (long long)ns * p->Hkv * pl.row_tiles;
        splits = ns > splits ? ns : splits;
      }
      const double waves = (double)((ctas + PLAN_SMS - 1) / PLAN_SMS);
      double cost = waves * (chunk + cta_overhead) + (ts ? 0 : tree_tiles);
      if (splits > 1) cost += combine_launch + 2.0 * splits * rows * 2.0 * (p->D * 2.0 + 4.0) / tile_bytes_equiv;
      if (cost < best) {
        best = cost;
        best_chunk = chunk;
        best_ts = ts;
      }
      if (chunk == 1) break;
    }
  }
  pl.chunk_tiles = best_chunk;
  pl.tree_split = best_ts;
  pl.max_splits = 1;
  for (int b = 0; b < p->B; ++b) {
    const int ns = num_splits(p->prefix_len_host[b], pl.chunk_tiles, pl.tree_split);
    pl.max_splits = ns > pl.max_splits ? ns : pl.max_splits;
  }
  // The order of the work items: every (sequence, split) pair, longest
  // first by the host's prefix lengths, so that the short ones (splits of
  // short prefixes, a tree split) are taken last and fill in beside the
  // long ones instead of starting after them.  Pairs with no work by the
  // host's lengths come last (the device's own lengths decide).
  pl.n_order = 0;
  if ((long long)p->B * pl.max_splits <= ATTN_ORDER_MAX) {
    int len[ATTN_ORDER_MAX], idx[ATTN_ORDER_MAX];
    uint32_t pair[ATTN_ORDER_MAX];
    int n = 0;
    for (int b = 0; b < p->B; ++b) {
      const int tiles = prefix_tiles(p->prefix_len_host[b]);
      const int ps = ceil_div(tiles, pl.chunk_tiles);
      const int ns = num_splits(p->prefix_len_host[b], pl.chunk_tiles, pl.tree_split);
      for (int s = 0; s < pl.max_splits; ++s) {
        int l = s < ps ? split_start(tiles, ps, s + 1) - split_start(tiles, ps, s) : 0;
        if (s == ns - 1) l += tree_tiles;
        const int start = s < ps ? split_start(tiles, ps, s) : 0;
        pair[n] = ((uint32_t)b << ORDER_B_SHIFT) | ((uint32_t)s << ORDER_SPLIT_SHIFT) |
                  (uint32_t)(start < ORDER_START_MASK ? start : ORDER_START_MASK);
        len[n] = l;
        idx[n] = n;
        ++n;
      }
    }
    std::stable_sort(idx, idx + n, [&](int x, int y) { return len[x] > len[y]; });
    for (int e = 0; e < n; ++e) pl.order[e] = pair[idx[e]];
    pl.n_order = n;
  }
  const size_t nrows = (size_t)p->B * p->N * p->Hq;
  pl.part_o_bytes = pl.max_splits > 1 ? round256((size_t)pl.max_splits * nrows * p->D * 2) : 0;
  pl.part_lse_bytes = pl.max_splits > 1 ? round256((size_t)pl.max_splits * nrows * sizeof(float)) : 0;
  // the attention kernel's item counter (256 bytes, zero between calls), then the partials
  pl.workspace_bytes = ATTN_SCHED_BYTES + pl.part_o_bytes + pl.part_lse_bytes;
  return pl;
}

// The kernels' opt-ins, once per device (host-side attributes, so the first
// call should come before any stream capture).  Also reports the largest
// cluster the stochastic verifier may use on this device.
cudaError_t prepare_device(int* stoch_max_cluster = nullptr) {
  static std::mutex mu;
  static bool done[64] = {};
  static int max_cluster[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    e = attn_tc_prepare();
    if (e != cudaSuccess) return e;
    e = stoch_prepare(&max_cluster[dev]);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  if (stoch_max_cluster) *stoch_max_cluster = max_cluster[dev];
  return cudaSuccess;
}

struct VerifyPlan {
  int chunks;
  size_t row_key, seq_ticket, total;
};

VerifyPlan plan_verify(int B, int N, int V) {
  VerifyPlan pl{};
  pl.chunks = ceil_div(V, VERIFY_CHUNK);
  // every byte must start zeroed and is left zeroed by each call
  pl.row_key = 0;
  pl.seq_ticket = round256((size_t)B * N * sizeof(unsigned long long));
  pl.total = pl.seq_ticket + round256((size_t)B * sizeof(unsigned));
  return pl;
}

ts_status verify_greedy_impl(const int32_t* draft_tokens, const float* target_logits, const int32_t* parent_idx,
                             int B, int N, int V, int max_depth, int32_t* accepted, int32_t* accept_len,
                             int32_t* bonus, int32_t* argmax_out, int32_t* status, void* workspace,
                             size_t workspace_bytes, ts_stream stream, int forest) {
  if (!draft_tokens || !target_logits || !parent_idx || !accepted || !accept_len || !bonus ||
      !argmax_out || !status)
    return TS_ERR_NULL;
  if (B < 1 || N < 1 || N > MAX_NODES || V < 1 || max_depth < 0) return TS_ERR_UNSUPPORTED;
  const VerifyPlan pl = plan_verify(B, N, V);
  if (!workspace || workspace_bytes < pl.total || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return TS_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  VerifyArgs a{};
  a.draft = draft_tokens;
  a.logits = target_logits;
  a.parent = parent_idx;
  a.B = B; a.N = N; a.V = V; a.max_depth = max_depth; a.chunks = pl.chunks;
  a.accepted = accepted; a.accept_len = accept_len; a.bonus = bonus; a.argmax = argmax_out;
  a.status = status;
  a.row_key = reinterpret_cast<unsigned long long*>(ws + pl.row_key);
  a.seq_ticket = reinterpret_cast<unsigned*>(ws + pl.seq_ticket);
  a.forest = forest;
  return launch_verify(a, (cudaStream_t)stream) == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

}  // namespace
}  // namespace ts

using namespace ts;

extern "C" {

const char* ts_status_str(ts_status st) {
  switch (st) {
    case TS_OK: return "ok";
    case TS_ERR_NULL: return "null pointer";
    case TS_ERR_SHAPE: return "bad shape, alignment or output size";
    case TS_ERR_BAD_TREE: return "invalid tree (need parent[0] == -1 and 0 <= parent[i] < i)";
    case TS_ERR_UNSUPPORTED: return "unsupported size";
    case TS_ERR_BAD_BLOCK: return "block table entry outside the KV pool";
    case TS_ERR_TIMEOUT: return "internal wait timed out";
    case TS_ERR_CUDA: return "CUDA error";
    case TS_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

ts_status tree_build_ancestry(const int32_t* parent_idx, const int32_t* prefix_len, int B, int N,
                              uint64_t* anc_mask, int32_t* depth, int32_t* pos, int32_t* status,
                              ts_stream stream) {
  if (!parent_idx || !prefix_len || !anc_mask || !depth || !pos || !status) return TS_ERR_NULL;
  if (B < 1 || N < 1 || N > MAX_NODES) return TS_ERR_UNSUPPORTED;
  cudaError_t e = launch_ancestry(parent_idx, prefix_len, B, N, anc_mask, depth, pos, status,
                                  (cudaStream_t)stream);
  return e == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

ts_status tree_build_ancestry_forest(const int32_t* parent_idx, const int32_t* prefix_len, int B, int N,
                                     uint64_t* anc_mask, int32_t* depth, int32_t* pos, int32_t* status,
                                     ts_stream stream) {
  if (!parent_idx || !prefix_len || !anc_mask || !depth || !pos || !status) return TS_ERR_NULL;
  if (B < 1 || N < 1 || N > MAX_NODES) return TS_ERR_UNSUPPORTED;
  cudaError_t e = launch_ancestry(parent_idx, prefix_len, B, N, anc_mask, depth, pos, status,
                                  (cudaStream_t)stream, 1);
  return e == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

size_t tree_attn_workspace_size(const ts_attn_params* p) {
  if (check_attn(p) != TS_OK) return 0;
  return plan_attn(p).workspace_bytes;
}

ts_status tree_attn_plan(const ts_attn_params* p, int32_t* chunk_tiles, int32_t* max_splits,
                         int32_t* tree_split) {
  const ts_status st = check_attn(p);
  if (st != TS_OK) return st;
  const AttnPlan pl = plan_attn(p);
  if (chunk_tiles) *chunk_tiles = pl.chunk_tiles;
  if (max_splits) *max_splits = pl.max_splits;
  if (tree_split) *tree_split = pl.tree_split;
  return TS_OK;
}

ts_status tree_attn_plan_order(const ts_attn_params* p, uint32_t* order, int32_t cap, int32_t* count) {
  const ts_status st = check_attn(p);
  if (st != TS_OK) return st;
  if (!count || (cap > 0 && !order)) return TS_ERR_NULL;
  if (cap < 0) return TS_ERR_SHAPE;
  const AttnPlan pl = plan_attn(p);
  *count = pl.n_order;
  if (cap < pl.n_order) return TS_ERR_SHAPE;
  for (int e = 0; e < pl.n_order; ++e) order[e] = pl.order[e];
  return TS_OK;
}

}  // extern "C"

namespace ts {
namespace {
ts_status attn_fwd_impl(const ts_attn_params* p, void* workspace, size_t workspace_bytes, ts_stream stream,
                        int stall_seq, int stall_tile, unsigned long long wait_limit_ns, int max_ctas) {
  ts_status st = check_attn(p);
  if (st != TS_OK) return st;
  const AttnPlan pl = plan_attn(p);
  if (!workspace || workspace_bytes < pl.workspace_bytes || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return TS_ERR_WORKSPACE;
  AttnArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(p->q);
  a.k_cache = static_cast<const __nv_bfloat16*>(p->k_cache);
  a.v_cache = static_cast<const __nv_bfloat16*>(p->v_cache);
  a.block_table = p->block_table;
  a.prefix_len = p->prefix_len;
  a.k_tree = static_cast<const __nv_bfloat16*>(p->k_tree);
  a.v_tree = static_cast<const __nv_bfloat16*>(p->v_tree);
  a.anc_mask = p->anc_mask;
  a.out = static_cast<__nv_bfloat16*>(p->out);
  a.lse = p->lse;
  a.status = p->status;
  char* ws = static_cast<char*>(workspace);
  a.sched = reinterpret_cast<unsigned*>(ws);
  a.part_o = reinterpret_cast<__nv_bfloat16*>(ws + ATTN_SCHED_BYTES);
  a.part_lse = reinterpret_cast<float*>(ws + ATTN_SCHED_BYTES + pl.part_o_bytes);
  a.B = p->B; a.N = p->N; a.Hq = p->Hq; a.Hkv = p->Hkv; a.G = p->Hq / p->Hkv; a.D = p->D;
  a.W = ceil_div(p->N, 64);
  a.bs = p->block_size; a.num_blocks = p->num_blocks; a.max_blocks = p->max_blocks;
  const float scale = p->scale == 0.f ? 1.f / std::sqrt((float)p->D) : p->scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.chunk_tiles = pl.chunk_tiles;
  a.max_splits = pl.max_splits;
  a.tree_split = pl.tree_split;
  a.row_tiles = pl.row_tiles;
  a.wait_limit_ns = wait_limit_ns;
  a.stall_seq = stall_seq;
  a.stall_tile = stall_tile;
  a.max_ctas = max_ctas;
  a.n_order = pl.n_order;
  a.order_host = pl.order;
  cudaStream_t s = (cudaStream_t)stream;
  if (prepare_device() != cudaSuccess) return TS_ERR_CUDA;
  if (launch_attn_tc(a, s) != cudaSuccess) return TS_ERR_CUDA;
  // with one split per unit the kernel writes `out` itself; otherwise merge the splits
  if (a.max_splits > 1 && launch_combine(a, s) != cudaSuccess) return TS_ERR_CUDA;
  return TS_OK;
}
}  // namespace
}  // namespace ts

extern "C" {

ts_status tree_attn_fwd(const ts_attn_params* p, void* workspace, size_t workspace_bytes,
                        ts_stream stream) {
  return ts::attn_fwd_impl(p, workspace, workspace_bytes, stream, -1, 0, ATTN_WAIT_LIMIT_NS, 0);
}

ts_status tree_attn_fwd_stall_test(const ts_attn_params* p, void* workspace, size_t workspace_bytes,
                                   int stall_seq, int stall_tile, uint32_t wait_limit_us, ts_stream stream) {
  if (p && (stall_seq < 0 || stall_seq >= p->B || stall_tile < 0)) return TS_ERR_SHAPE;
  if (wait_limit_us < 100 || wait_limit_us > 1000000) return TS_ERR_UNSUPPORTED;
  return ts::attn_fwd_impl(p, workspace, workspace_bytes, stream, stall_seq, stall_tile,
                           (unsigned long long)wait_limit_us * 1000ull, 0);
}

ts_status tree_attn_fwd_ctas_test(const ts_attn_params* p, void* workspace, size_t workspace_bytes, int max_ctas,
                                  int stall_seq, int stall_tile, uint32_t wait_limit_us, ts_stream stream) {
  if (max_ctas < 1) return TS_ERR_UNSUPPORTED;
  if (p && (stall_seq < -1 || stall_seq >= p->B || (stall_seq >= 0 && stall_tile < 0))) return TS_ERR_SHAPE;
  if (wait_limit_us < 100 || wait_limit_us > 1000000) return TS_ERR_UNSUPPORTED;
  return ts::attn_fwd_impl(p, workspace, workspace_bytes, stream, stall_seq, stall_seq >= 0 ? stall_tile : 0,
                           (unsigned long long)wait_limit_us * 1000ull, max_ctas);
}

size_t tree_verify_workspace_size(int B, int N, int V) {
  if (B < 1 || N < 1 || N > MAX_NODES || V < 1) return 0;
  return plan_verify(B, N, V).total;
}

ts_status tree_verify_greedy(const int32_t* draft_tokens, const float* target_logits,
                             const int32_t* parent_idx, int B, int N, int V, int max_depth,
                             int32_t* accepted, int32_t* accept_len, int32_t* bonus,
                             int32_t* argmax_out, int32_t* status, void* workspace,
                             size_t workspace_bytes, ts_stream stream) {
  return ts::verify_greedy_impl(draft_tokens, target_logits, parent_idx, B, N, V, max_depth, accepted, accept_len,
                                bonus, argmax_out, status, workspace, workspace_bytes, stream, 0);
}

ts_status tree_verify_greedy_forest(const int32_t* draft_tokens, const float* target_logits,
                                    const int32_t* parent_idx, int B, int N, int V, int max_depth,
                                    int32_t* accepted, int32_t* accept_len, int32_t* bonus,
                                    int32_t* argmax_out, int32_t* status, void* workspace,
                                    size_t workspace_bytes, ts_stream stream) {
  return ts::verify_greedy_impl(draft_tokens, target_logits, parent_idx, B, N, V, max_depth, accepted, accept_len,
                                bonus, argmax_out, status, workspace, workspace_bytes, stream, 1);
}

ts_status tree_commit_accepted(const void* k_tree, const void* v_tree, const int32_t* accepted,
                               const int32_t* accept_len, const int32_t* prefix_len, void* k_cache, void* v_cache,
                               const int32_t* block_table, int B, int N, int Hkv, int D, int block_size,
                               int num_blocks, int max_blocks, int max_depth, int32_t* new_prefix_len,
                               int32_t* status, ts_stream stream) {
  if (!k_tree || !v_tree || !accepted || !accept_len || !prefix_len || !k_cache || !v_cache || !block_table ||
      !new_prefix_len)
    return TS_ERR_NULL;
  if (B < 1 || N < 1 || N > MAX_NODES || Hkv < 1 || block_size < 1 || num_blocks < 1 || max_blocks < 1 ||
      max_depth < 0)
    return TS_ERR_SHAPE;
  if (D != 64 && D != 128) return TS_ERR_UNSUPPORTED;
  if (!aligned16(k_tree) || !aligned16(v_tree) || !aligned16(k_cache) || !aligned16(v_cache)) return TS_ERR_SHAPE;
  CommitArgs a{};
  a.k_tree = static_cast<const __nv_bfloat16*>(k_tree);
  a.v_tree = static_cast<const __nv_bfloat16*>(v_tree);
  a.accepted = accepted;
  a.accept_len = accept_len;
  a.prefix_len = prefix_len;
  a.k_cache = static_cast<__nv_bfloat16*>(k_cache);
  a.v_cache = static_cast<__nv_bfloat16*>(v_cache);
  a.block_table = block_table;
  a.new_prefix_len = new_prefix_len;
  a.status = status;
  a.B = B; a.N = N; a.Hkv = Hkv; a.D = D; a.bs = block_size; a.num_blocks = num_blocks;
  a.max_blocks = max_blocks; a.max_depth = max_depth;
  return launch_commit(a, (cudaStream_t)stream) == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

ts_status tree_verify_stochastic(const int32_t* draft_tokens, const float* target_logits, const float* draft_probs,
                                 const int32_t* parent_idx, const float* coins, int B, int N, int V, int max_depth,
                                 float temperature, int32_t* accepted, int32_t* accept_len, int32_t* bonus,
                                 int32_t* status, ts_stream stream) {
  if (!draft_tokens || !target_logits || !draft_probs || !parent_idx || !coins || !accepted || !accept_len ||
      !bonus || !status)
    return TS_ERR_NULL;
  if (B < 1 || B > 65535 || N < 1 || N > MAX_NODES || V < 1 || V > STOCH_MAX_CLUSTER * STOCH_MAX_SLICE ||
      max_depth < 0)
    return TS_ERR_UNSUPPORTED;
  if (!(temperature > 0.f) || std::isinf(temperature)) return TS_ERR_UNSUPPORTED;
  int max_cluster = STOCH_PORTABLE_CLUSTER;
  if (prepare_device(&max_cluster) != cudaSuccess) return TS_ERR_CUDA;
  // the cluster doubles until a slice holds at most STOCH_TARGET_SLICE elements
  int C = 1;
  while (C < max_cluster && ceil_div(V, C) > STOCH_TARGET_SLICE) C *= 2;
  const int slice = (ceil_div(V, C) + 3) & ~3;
  if (slice > STOCH_MAX_SLICE) return TS_ERR_UNSUPPORTED;
  StochArgs a{};
  a.draft = draft_tokens;
  a.logits = target_logits;
  a.q = draft_probs;
  a.parent = parent_idx;
  a.coins = coins;
  a.B = B; a.N = N; a.V = V; a.max_depth = max_depth;
  a.inv_temp_log2e = 1.4426950408889634f / temperature;
  a.cluster = C;
  a.slice = slice;
  a.bulk = (V % 4 == 0) && aligned16(target_logits) && aligned16(draft_probs);
  a.accepted = accepted; a.accept_len = accept_len; a.bonus = bonus; a.status = status;
  return launch_verify_stoch(a, (cudaStream_t)stream) == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

ts_status tree_build_dynamic(const int32_t* pool_parent, const float* pool_logp, const int32_t* pool_token,
                             const int32_t* prefix_len, int B, int M, int N, int32_t* parent_idx,
                             int32_t* draft_tokens, int32_t* sel_index, uint64_t* anc_mask, int32_t* depth,
                             int32_t* pos, int32_t* status, ts_stream stream) {
  if (!pool_parent || !pool_logp || !pool_token || !prefix_len || !parent_idx || !draft_tokens || !sel_index ||
      !anc_mask || !depth || !pos || !status)
    return TS_ERR_NULL;
  if (B < 1 || N < 1 || M < N) return TS_ERR_SHAPE;
  if (N > MAX_NODES || M > DYN_MAX_POOL) return TS_ERR_UNSUPPORTED;
  DynArgs a{};
  a.pool_parent = pool_parent;
  a.pool_logp = pool_logp;
  a.pool_token = pool_token;
  a.prefix_len = prefix_len;
  a.B = B; a.M = M; a.N = N;
  a.parent_idx = parent_idx; a.draft_tokens = draft_tokens; a.sel_index = sel_index; a.anc_mask = anc_mask;
  a.depth = depth; a.pos = pos; a.status = status;
  return launch_build_dynamic(a, (cudaStream_t)stream) == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

ts_status tree_verify_greedy_noalloc(const int32_t* draft_tokens, const float* target_logits,
                                     const int32_t* parent_idx, int B, int N, int V, int max_depth,
                                     int32_t* accepted, int32_t* accept_len, int32_t* bonus,
                                     int32_t* argmax_out, int32_t* status, ts_stream stream) {
  if (!draft_tokens || !target_logits || !parent_idx || !accepted || !accept_len || !bonus ||
      !argmax_out || !status)
    return TS_ERR_NULL;
  if (B < 1 || N < 1 || N > MAX_NODES || V < 1 || max_depth < 0) return TS_ERR_UNSUPPORTED;
  const VerifyPlan pl = plan_verify(B, N, V);
  if (pl.total > TS_VERIFY_NOALLOC_SCRATCH_BYTES) return TS_ERR_WORKSPACE;
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  const ts_status st = verify_static_scratch(&scratch, &scratch_bytes);
  if (st != TS_OK) return st;
  if (pl.total > scratch_bytes) return TS_ERR_WORKSPACE;
  // The array keeps whatever the previous call left; the argmax keys and
  // arrival counters must start at zero, so clear them on the caller's stream.
  if (cudaMemsetAsync(scratch, 0, pl.total, (cudaStream_t)stream) != cudaSuccess) return TS_ERR_CUDA;
  char* ws = static_cast<char*>(scratch);
  VerifyArgs a{};
  a.draft = draft_tokens;
  a.logits = target_logits;
  a.parent = parent_idx;
  a.B = B; a.N = N; a.V = V; a.max_depth = max_depth; a.chunks = pl.chunks;
  a.accepted = accepted; a.accept_len = accept_len; a.bonus = bonus; a.argmax = argmax_out;
  a.status = status;
  a.row_key = reinterpret_cast<unsigned long long*>(ws + pl.row_key);
  a.seq_ticket = reinterpret_cast<unsigned*>(ws + pl.seq_ticket);
  return launch_verify(a, (cudaStream_t)stream) == cudaSuccess ? TS_OK : TS_ERR_CUDA;
}

}  // extern "C"
