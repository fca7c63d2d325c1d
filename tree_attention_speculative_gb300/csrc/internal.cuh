// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "treespec.h"

namespace ts {

// Programmatic dependent launch.  Every kernel of the library is launched so
// that it may start while the previous kernel in the stream finishes; each one
// runs only its set-up (no global memory) before pdl_wait(), which returns once
// the previous kernel has completed and its writes are visible, and then calls
// pdl_trigger() to let the next kernel begin its own set-up.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Prefix keys are processed in tiles of KV_TILE tokens; packed query rows in
// tiles of ROW_TILE rows (one MMA M extent).
constexpr int KV_TILE = 128;
constexpr int ROW_TILE = 128;
constexpr int MAX_NODES = 256;
constexpr int PLAN_SMS = 152;  // GB300: the planner sizes grids for 152 SMs

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Division by a divisor fixed for a whole launch, for numerators in [0, 2^31),
// by a multiply-high, an add and a shift instead of the ~30-instruction
// integer division: with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// n / d = (umulhi(n, m) + n) >> l (the round-up method of Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994;
// n < 2^31 keeps the sum within 32 bits).
struct FastDiv {
  uint32_t m = 1, l = 0;
  int d = 1;
  static FastDiv make(int d) {
    FastDiv f;
    f.d = d;
    while ((1ull << f.l) < (unsigned long long)d) ++f.l;
    f.m = (uint32_t)((((1ull << 32) * ((1ull << f.l) - (unsigned long long)d)) / (unsigned long long)d) + 1ull);
    return f;
  }
  __host__ __device__ int div(int n) const {
#ifdef __CUDA_ARCH__
    const uint32_t t = __umulhi((uint32_t)n, m);
#else
    const uint32_t t = (uint32_t)(((unsigned long long)(uint32_t)n * m) >> 32);
#endif
    return (int)((t + (uint32_t)n) >> l);
  }
  __host__ __device__ int mod(int n) const { return n - div(n) * d; }
};

// Number of prefix tiles of a sequence, and how many splits its prefix is cut
// into when no split takes more than `chunk_tiles` tiles.  The tree block
// rides on the LAST split of a sequence: with tree_split = 0 that is the last
// prefix split (a sequence with no prefix still has one split for it); with
// tree_split = 1 it is one more split of its own, with no prefix tiles.
__host__ __device__ inline int prefix_tiles(int P) { return ceil_div(P, KV_TILE); }
__host__ __device__ inline int num_splits(int P, int chunk_tiles, int tree_split) {
  const int ps = ceil_div(prefix_tiles(P), chunk_tiles);
  return tree_split ? ps + 1 : (ps == 0 ? 1 : ps);
}
// First prefix tile of split s (0 <= s <= ps) when a sequence's `tiles` prefix
// tiles are cut into ps = ceil(tiles / chunk_tiles) splits of near-equal
// length (they differ by one tile at most, so none exceeds chunk_tiles).  A
// fixed chunk would leave the remainder in one short split; equal splits
// keep the work items of a ragged batch closer in length.  Split s holds
// tiles [split_start(s), split_start(s + 1)).  tiles <= 2^23 (P <= 2^30) and
// s <= ps <= 256 (the planner's limit), so the product fits in 32 bits.
__host__ __device__ inline int split_start(int tiles, int ps, int s) {
  return ps > 0 ? (int)(((unsigned)tiles * (unsigned)s) / (unsigned)ps) : 0;
}

// The prefix length a kernel may use for sequence b: the device value, clamped
// to what the host planned for (grid, workspace) and to the block table's
// width.  Returns true when no clamping was needed.  Kernels report a clamp as
// TS_ERR_SHAPE so a disagreement between the device and host prefix lengths can
// never drive an access outside the planned buffers.
__host__ __device__ inline bool usable_prefix(int P, int chunk_tiles, int max_splits, int tree_split, int bs,
                                              int max_blocks, int* out) {
  long long cap = (long long)chunk_tiles * (max_splits - tree_split) * KV_TILE;
  const long long cap_blocks = (long long)max_blocks * bs;
  if (cap_blocks < cap) cap = cap_blocks;
  long long v = P < 0 ? 0 : P;
  const bool ok = (P >= 0) && (v <= cap);
  if (v > cap) v = cap;
  *out = (int)v;
  return ok;
}

// Everything a launch of the attention kernels needs (device pointers).
struct AttnArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_cache;
  const __nv_bfloat16* v_cache;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const __nv_bfloat16* k_tree;
  const __nv_bfloat16* v_tree;
  const uint64_t* anc_mask;
  __nv_bfloat16* out;
  float* lse;
  int32_t* status;
  unsigned* sched;         // item counter of the persistent attention kernel: zero before and after a call
  __nv_bfloat16* part_o;  // [max_splits, B*N*Hq, D] bf16, normalised partial outputs
  float* part_lse;  // [max_splits, B*N*Hq] fp32, base-2 log-sum-exp of each partial
  int B, N, Hq, Hkv, G, D, W;
  int bs, num_blocks, max_blocks;
  float scale_log2;  // softmax scale * log2(e)
  int chunk_tiles;   // prefix tiles per split
  int max_splits;    // splits of the longest sequence, the tree's own split included
  int tree_split;    // 1: the tree block is a split of its own
  int row_tiles;     // ceil(N*G / ROW_TILE)
  // Every bounded wait of the attention kernel gives up after wait_limit_ns.
  // Testing the failure path: with stall_seq >= 0, every CTA of that sequence
  // stops its K stream before tile stall_tile (its loads are never issued),
  // so the wait for that tile runs out with nothing in flight.
  unsigned long long wait_limit_ns;
  int stall_seq, stall_tile;
  int max_ctas;  // > 0: at most this many CTAs of the persistent kernel (testing); else one per SM
  // The order of the attention kernel's work items (host array, read when
  // the launch is made): every (sequence, split) pair once, longest first by
  // the host's prefix lengths, packed as the ORDER_* constants say.  n_order
  // = 0: no table (items in unit-major order).
  int n_order;
  const uint32_t* order_host;
};
// At most this many (sequence, split) pairs are ordered by a table (so b and
// split each fit in 8 bits); a launch with more keeps the unit-major order.
// An entry packs b (bits 24-31), split (bits 15-23) and the split's first
// prefix tile by the host's prefix length (bits 0-14; all ones if larger).
constexpr int ATTN_ORDER_MAX = 256;
constexpr int ORDER_B_SHIFT = 24;
constexpr int ORDER_SPLIT_SHIFT = 15;
constexpr uint32_t ORDER_SPLIT_MASK = 0x1ffu;
constexpr int ORDER_START_MASK = 0x7fff;
constexpr unsigned long long ATTN_WAIT_LIMIT_NS = 200000000ull;  // 200 ms: far above any legitimate wait
constexpr size_t ATTN_SCHED_BYTES = 256;  // head of the attention workspace: the item counter

struct AttnPlan {
  int chunk_tiles;
  int max_splits;
  int tree_split;
  int row_tiles;
  size_t part_o_bytes;
  size_t part_lse_bytes;
  size_t workspace_bytes;
  int n_order;  // 0 or B * max_splits (see AttnArgs::order_host)
  uint32_t order[ATTN_ORDER_MAX];
};

cudaError_t launch_ancestry(const int32_t* parent, const int32_t* prefix_len, int B, int N,
                            uint64_t* anc, int32_t* depth, int32_t* pos, int32_t* status,
                            cudaStream_t s, int forest = 0);
cudaError_t attn_tc_prepare();
cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_combine(const AttnArgs& a, cudaStream_t s);

struct VerifyArgs {
  const int32_t* draft;
  const float* logits;
  const int32_t* parent;
  int B, N, V, max_depth, chunks;
  int32_t* accepted;
  int32_t* accept_len;
  int32_t* bonus;
  int32_t* argmax;
  int32_t* status;
  unsigned long long* row_key;  // [B*N] packed (value, index) argmax keys, 0 between calls
  unsigned* seq_ticket;         // [B] arrival counters, 0 between calls
  int forest;  // several roots allowed; chains stop at -1
};
constexpr int VERIFY_THREADS = 256;
constexpr int VERIFY_CHUNK = 8192;  // logits per CTA
cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t s);
ts_status verify_static_scratch(void** ptr, size_t* bytes);

struct CommitArgs {
  const __nv_bfloat16* k_tree;
  const __nv_bfloat16* v_tree;
  const int32_t* accepted;
  const int32_t* accept_len;
  const int32_t* prefix_len;
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  const int32_t* block_table;
  int32_t* new_prefix_len;
  int32_t* status;
  int B, N, Hkv, D, bs, num_blocks, max_blocks, max_depth;
};
cudaError_t launch_commit(const CommitArgs& a, cudaStream_t s);

// Stochastic verification: one cluster of `cluster` CTAs per sequence, CTA k
// holding vocabulary slice [k*slice, (k+1)*slice) of the visited node's rows.
struct StochArgs {
  const int32_t* draft;
  const float* logits;
  const float* q;
  const int32_t* parent;
  const float* coins;
  int B, N, V, max_depth;
  float inv_temp_log2e;  // log2(e) / temperature
  int cluster, slice;    // slice: elements per CTA, a multiple of 4
  int bulk;              // rows start 16-byte aligned: slices arrive by bulk copy
  int32_t* accepted;
  int32_t* accept_len;
  int32_t* bonus;
  int32_t* status;
};
constexpr int STOCH_THREADS = 256;
constexpr int STOCH_MAX_CLUSTER = 16;                  // where the GPU allows non-portable clusters
constexpr int STOCH_PORTABLE_CLUSTER = 8;
constexpr int STOCH_TARGET_SLICE = 8192;               // the cluster grows until a slice is this small
constexpr int STOCH_MAX_SLICE = 25600;                 // 2 x 100 KB of shared memory per CTA
cudaError_t stoch_prepare(int* max_cluster);

// Dynamic tree construction: one CTA per sequence over a candidate pool.
struct DynArgs {
  const int32_t* pool_parent;
  const float* pool_logp;
  const int32_t* pool_token;
  const int32_t* prefix_len;
  int B, M, N;
  int32_t* parent_idx;
  int32_t* draft_tokens;
  int32_t* sel_index;
  uint64_t* anc_mask;
  int32_t* depth;
  int32_t* pos;
  int32_t* status;
};
constexpr int DYN_MAX_POOL = 1024;
cudaError_t launch_build_dynamic(const DynArgs& a, cudaStream_t s);
cudaError_t launch_verify_stoch(const StochArgs& a, cudaStream_t s);

}  // namespace ts
