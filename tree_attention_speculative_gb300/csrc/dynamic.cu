// Dynamic draft-tree construction: rerank a candidate pool, flatten the kept
// tree and build its ancestry masks, depths and positions in one kernel.
//
// [P2] Common Confusions (the tree shape may be selected dynamically) and
// Where It Appears (EAGLE-2: the tree changes per context, and the ancestry
// mask is built after reranking); [P1] Key Mechanisms > Tree-Structured
// Candidate Generation; [P2] Tradeoffs (tree construction, flattening and
// position bookkeeping).
//
// value(root) = 0, value(c) = value(parent(c)) + logp(c) in fp32 from the
// root down; the root and the N - 1 candidates of highest value (ties to the
// smaller pool index) are kept, in pool order.  Log-probabilities are <= 0, so
// a parent's value is at least its child's and its index is smaller: the kept
// set always contains the parent of every kept node.
//
// One CTA per sequence, one thread per pool candidate (the pool's parents
// and values live in shared memory).  Values are computed level by level
// (one barrier per level), so each candidate adds its log-probability to its
// parent's finished value exactly as the definition orders it.  The N-th best
// value is found bit by bit, each bit one counting barrier
// (__syncthreads_count); ties at it go to the smaller pool index; warp ballots
// give the kept candidates their tree indices; then each of the first N
// threads walks one kept node's new parent chain for its mask row.
#include "internal.cuh"

namespace ts {
namespace {

constexpr int DYN_THREADS = DYN_MAX_POOL;  // one thread per pool candidate
constexpr int DYN_WARPS = DYN_THREADS / 32;

// Order-preserving map of a float to an unsigned key, inverted so that an
// ascending order puts the largest value first.
__device__ __forceinline__ uint32_t desc_key(float v) {
  if (v == 0.f) v = 0.f;  // one zero
  const uint32_t u = __float_as_uint(v);
  const uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ~asc;
}

struct DynShared {
  int parent[DYN_MAX_POOL];
  float value[DYN_MAX_POOL];
  int newidx[DYN_MAX_POOL];  // tree index of a kept candidate, -1 otherwise
  int tparent[MAX_NODES];    // the kept tree's parent array
  int wsum[DYN_WARPS];
  int maxd;
};

// Exclusive prefix count of `flag` over the threads in thread order, and the total.
__device__ __forceinline__ int block_excl_count(bool flag, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  if (lane == 0) wsum[warp] = __popc(bal);
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll 8
  for (int w = 0; w < DYN_WARPS; ++w) {
    const int x = wsum[w];
    before += w < warp ? x : 0;
    all += x;
  }
  __syncthreads();
  *total = all;
  return before + __popc(bal & ((1u << lane) - 1u));
}

__global__ void __launch_bounds__(DYN_THREADS) k_build_dynamic(DynArgs a) {
  __shared__ DynShared sh;
  const int b = blockIdx.x, c = threadIdx.x;
  const int M = a.M, N = a.N, W = (N + 63) / 64;
  const bool in = c < M;
  pdl_wait();
  pdl_trigger();

  const int p = in ? a.pool_parent[(size_t)b * M + c] : 0;
  const float lp = in ? a.pool_logp[(size_t)b * M + c] : 0.f;
  const int P = a.prefix_len[b];
  if (in) sh.parent[c] = p;
  if (c == 0) sh.maxd = 0;
  const bool bad = in && ((c == 0) ? (p != -1) : (p < 0 || p >= c || !(lp <= 0.f)));
  if (__syncthreads_or(bad)) {
    // report the invalid pool and leave a harmless star tree behind
    for (int k = c; k < N; k += DYN_THREADS) {
      a.parent_idx[(size_t)b * N + k] = k == 0 ? -1 : 0;
      a.draft_tokens[(size_t)b * N + k] = 0;
      a.sel_index[(size_t)b * N + k] = 0;
      a.depth[(size_t)b * N + k] = k == 0 ? 0 : 1;
      a.pos[(size_t)b * N + k] = P + (k == 0 ? 0 : 1);
      for (int w = 0; w < W; ++w) {
        unsigned long long m = 0;
        if (w == 0) m |= 1ull;
        if (k / 64 == w) m |= 1ull << (k % 64);
        a.anc_mask[((size_t)b * N + k) * W + w] = m;
      }
    }
    if (c == 0) a.status[b] = TS_ERR_BAD_TREE;
    return;
  }

  // depth (walk to the root), then values level by level from the root down
  int d = 0;
  if (in)
    for (int x = c; x != 0; x = sh.parent[x]) ++d;
  const int wd = __reduce_max_sync(0xffffffffu, d);
  if ((c & 31) == 0) atomicMax(&sh.maxd, wd);
  if (c == 0) sh.value[0] = 0.f;
  __syncthreads();
  const int maxd = sh.maxd;
  for (int l = 1; l <= maxd; ++l) {
    if (in && d == l) sh.value[c] = __fadd_rn(sh.value[p], lp);
    __syncthreads();
  }
  const uint32_t key = in ? desc_key(sh.value[c]) : 0xffffffffu;

  // The N-th smallest key K, bit by bit from the top: K is the least t with
  // #{key <= t} >= N; each step is one counting barrier.
  uint32_t K = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t probe = K + ((1u << bit) - 1u);
    if (__syncthreads_count(in && key <= probe) < N) K += 1u << bit;
  }
  // kept: key < K, or key == K among the first (N - #{key < K}) in pool order
  const int below = __syncthreads_count(in && key < K);
  int ties_total;
  const int tie_rank = block_excl_count(in && key == K, sh.wsum, &ties_total);
  const bool keep = in && (key < K || (key == K && tie_rank < N - below));
  int kept_total;
  const int k = block_excl_count(keep, sh.wsum, &kept_total);
  if (in) sh.newidx[c] = keep ? k : -1;
  __syncthreads();
  if (keep) {
    const int tp = c == 0 ? -1 : sh.newidx[p];
    sh.tparent[k] = tp;
    a.parent_idx[(size_t)b * N + k] = tp;
    a.sel_index[(size_t)b * N + k] = c;
    a.draft_tokens[(size_t)b * N + k] = a.pool_token[(size_t)b * M + c];
  }
  __syncthreads();

  // ancestry rows, depths and positions of the kept tree
  if (c < N) {
    unsigned long long m0 = 0, m1 = 0, m2 = 0, m3 = 0;
    int dd = 0;
    for (int x = c; x != -1; x = sh.tparent[x]) {
      const unsigned long long bitm = 1ull << (x & 63);
      switch (x >> 6) {
        case 0: m0 |= bitm; break;
        case 1: m1 |= bitm; break;
        case 2: m2 |= bitm; break;
        default: m3 |= bitm; break;
      }
      if (x != c) ++dd;
    }
    uint64_t* row = a.anc_mask + ((size_t)b * N + c) * W;
    row[0] = m0;
    if (W > 1) row[1] = m1;
    if (W > 2) row[2] = m2;
    if (W > 3) row[3] = m3;
    a.depth[(size_t)b * N + c] = dd;
    a.pos[(size_t)b * N + c] = P + dd;
  }
  if (c == 0) a.status[b] = TS_OK;
}

}  // namespace

cudaError_t launch_build_dynamic(const DynArgs& a, cudaStream_t s) {
  return launch_pdl(k_build_dynamic, dim3(a.B), dim3(DYN_THREADS), 0, s, a);
}

}  // namespace ts
