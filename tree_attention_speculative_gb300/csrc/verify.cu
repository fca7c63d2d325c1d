// Greedy verification: vocab argmax of every node's logits fused with the
// parent-chain acceptance walk.
//
// [P3] code listing, verify_candidate_tree (the target's greedy prediction is
// the argmax of a node's logits); [P1] Key Mechanisms > Multi-Token Acceptance
// & Rollback and [P2] How It Works (accept the longest valid root path, up to
// the first rejection).  The listing's own flattened-index scan is not
// tree-aware and is not followed: a node's logits predict its children, and a
// node is accepted only if every edge on its chain to the root matches.
//
// Layout of the work: the logits of row (b, i) are cut into chunks of
// VERIFY_CHUNK floats, one CTA per (row, chunk).  Each CTA streams its chunk
// with 16-byte loads (all of a thread's loads are issued before any is used),
// keeps a running (max, first index) per thread, and reduces it with warp
// shuffles and one shared-memory step.  The CTA's result is folded into the
// row's 64-bit key with one atomicMax: the high word is the value mapped to
// an order-preserving unsigned, the low word 0xFFFFFFFF - index, so the
// larger value and, on ties, the smaller index win, and every real key is
// above 0.  The last CTA to finish a sequence (an atomicInc ticket that
// wraps back to 0) decodes the row keys into argmax, sets them back to 0 and
// runs the acceptance walk, one thread per node.  No CTA ever waits for
// another, so nothing here can hang; the keys and tickets return to zero by
// themselves.
#include <cfloat>
#include <climits>
#include <mutex>

#include "internal.cuh"
#include "sm100.cuh"

namespace ts {

__device__ __forceinline__ void take_better(float& v, int& i, float v2, int i2) {
  // larger value wins; equal values keep the smaller index (first occurrence)
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

// Order-preserving map of a finite float to an unsigned (larger float, larger
// unsigned); -inf maps to 0x007FFFFF, so the packed key of any value is > 0.
// -0.0 is first turned into +0.0: the two compare equal, so between chunks,
// as inside one, a tie at zero must go to the smaller index.
__device__ __forceinline__ unsigned long long argmax_key(float v, int i) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)ord << 32) | (0xFFFFFFFFu - (uint32_t)i);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    take_better(v, i, v2, i2);
  }
}

// Reduce (v, i) over the CTA; the result is valid in thread 0.
__device__ __forceinline__ void block_argmax(float& v, int& i) {
  __shared__ float sv[VERIFY_THREADS / 32];
  __shared__ int si[VERIFY_THREADS / 32];
  warp_argmax(v, i);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    sv[w] = v;
    si[w] = i;
  }
  __syncthreads();
  if (w == 0) {
    v = (l < VERIFY_THREADS / 32) ? sv[l] : -INFINITY;
    i = (l < VERIFY_THREADS / 32) ? si[l] : INT_MAX;
    warp_argmax(v, i);
  }
}

// Eight CTAs per SM (32 registers a thread), so a grid of up to 8 * SMs CTAs
// is resident at once.
__global__ void __launch_bounds__(VERIFY_THREADS, 8)
k_verify(VerifyArgs a) {
  const int row = blockIdx.x / a.chunks;
  const int chunk = blockIdx.x - row * a.chunks;
  const int b = row / a.N;
  const float* x = a.logits + (size_t)row * a.V;
  const int lo = chunk * VERIFY_CHUNK;
  const int hi = min(a.V, lo + VERIFY_CHUNK);
  // Prefetch this chunk into L2 while the previous kernel finishes (a
  // prefetch reads no data, so it may precede the wait; see sm100.cuh).
  if (threadIdx.x == 0 && ((reinterpret_cast<uintptr_t>(x + lo) & 15) == 0) && hi - lo >= 4)
    sm100::bulk_prefetch_l2(x + lo, (uint32_t)((hi - lo) * 4) & ~15u);
  // the sequence's draft tokens and parents, which its walk reads (one
  // 128-byte line per thread, by the sequence's first CTA)
  if (row == b * a.N && chunk == 0 && (int)threadIdx.x * 32 < a.N) {
    sm100::prefetch_l2(a.draft + (size_t)b * a.N + threadIdx.x * 32);
    sm100::prefetch_l2(a.parent + (size_t)b * a.N + threadIdx.x * 32);
  }
  pdl_wait();
  pdl_trigger();

  // Each thread starts at (-inf, its first index), so a row of nothing but
  // -inf still yields its first index; a thread with no element keeps
  // INT_MAX, which loses every tie.
  float bv = -INFINITY;
  int bi = INT_MAX;
  const bool vec = ((reinterpret_cast<uintptr_t>(x + lo) & 15) == 0) && (((hi - lo) & 3) == 0);
  if (vec) {
    constexpr int PER = VERIFY_CHUNK / (4 * VERIFY_THREADS);  // float4 per thread in a full chunk
    const float4* x4 = reinterpret_cast<const float4*>(x + lo);
    const int n4 = (hi - lo) >> 2;
    if ((int)threadIdx.x < n4) bi = lo + 4 * threadIdx.x;
    float4 r[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int e = threadIdx.x + k * VERIFY_THREADS;
      r[k] = (e < n4) ? __ldcs(x4 + e) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int base = lo + 4 * (threadIdx.x + k * VERIFY_THREADS);
      // indices grow with k and within the float4: strict '>' keeps the first maximum
      if (r[k].x > bv) { bv = r[k].x; bi = base; }
      if (r[k].y > bv) { bv = r[k].y; bi = base + 1; }
      if (r[k].z > bv) { bv = r[k].z; bi = base + 2; }
      if (r[k].w > bv) { bv = r[k].w; bi = base + 3; }
    }
  } else {
    if (lo + (int)threadIdx.x < hi) bi = lo + threadIdx.x;
    for (int e = lo + threadIdx.x; e < hi; e += VERIFY_THREADS) {
      const float v = x[e];
      if (v > bv) { bv = v; bi = e; }
    }
  }
  block_argmax(bv, bi);

  __shared__ int s_flag;
  if (threadIdx.x == 0) {
    atomicMax(&a.row_key[row], argmax_key(bv, bi));
    __threadfence();  // the key before the ticket
    const unsigned last = (unsigned)(a.N * a.chunks - 1);
    const bool is_last = atomicInc(&a.seq_ticket[b], last) == last;
    if (is_last) __threadfence();  // every other CTA's key before this CTA's reads (the barrier passes it on)
    s_flag = is_last;
  }
  __syncthreads();
  if (!s_flag) return;

  // ---- acceptance walk for sequence b (this CTA saw every row of b finish) ----
  __shared__ int s_par[MAX_NODES], s_draft[MAX_NODES], s_pred[MAX_NODES];
  __shared__ int s_key[VERIFY_THREADS / 32];
  const int N = a.N;
  const int t = threadIdx.x;
  bool ok = true;
  if (t < N) {
    const int p = a.parent[(size_t)b * N + t];
    ok = (t == 0) ? (p == -1) : ((p >= 0 && p < t) || (a.forest && p == -1));
    s_par[t] = p;
    s_draft[t] = a.draft[(size_t)b * N + t];
    unsigned long long* key = a.row_key + (size_t)b * N + t;
    const int am = (int)(0xFFFFFFFFu - (uint32_t)(__ldcg(key) & 0xFFFFFFFFull));
    *key = 0ull;  // ready for the next call
    s_pred[t] = am;
    a.argmax[(size_t)b * N + t] = am;
  }
  const int valid = __syncthreads_and(ok);
  int32_t* acc_row = a.accepted + (size_t)b * (a.max_depth + 1);
  if (!valid) {
    for (int k = t; k <= a.max_depth; k += VERIFY_THREADS) acc_row[k] = -1;
    if (t == 0) {
      a.accept_len[b] = 0;
      a.bonus[b] = 0;
      a.status[b] = TS_ERR_BAD_TREE;
    }
    return;
  }
  // key = (depth << 16) | (0xFFFF - node) for accepted nodes: the maximum key
  // is the deepest accepted node, smallest index on ties.  The root (every
  // root of a forest) is always accepted, so the maximum is never the -1 of a
  // rejected node.  A chain ends at its root, the node whose parent is -1.
  int key = -1;
  if (t < N) {
    bool acc = true;
    int d = 0, y = t;
    while (s_par[y] != -1) {
      const int p = s_par[y];
      acc = acc && (s_draft[y] == s_pred[p]);
      y = p;
      ++d;
    }
    if (acc) key = (d << 16) | (0xFFFF - t);
  }
  key = __reduce_max_sync(0xffffffffu, key);
  if ((t & 31) == 0) s_key[t >> 5] = key;
  __syncthreads();
  if (t < 32) {
    int k2 = (t < VERIFY_THREADS / 32) ? s_key[t] : -1;
    k2 = __reduce_max_sync(0xffffffffu, k2);
    if (t == 0) s_key[0] = k2;
  }
  __syncthreads();
  const int best = s_key[0];
  const int L = best >> 16;
  const int nstar = 0xFFFF - (best & 0xFFFF);
  const bool fits = L <= a.max_depth;
  for (int k = t; k <= a.max_depth; k += VERIFY_THREADS)
    if (!fits || k > L) acc_row[k] = -1;
  if (t == 0) {
    if (fits) {
      int y = nstar;
      for (int k = L; k >= 0; --k) {
        acc_row[k] = y;
        y = s_par[y];
      }
    } else {
      a.status[b] = TS_ERR_SHAPE;
    }
    a.accept_len[b] = L;
    a.bonus[b] = s_pred[nstar];
  }
}

cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t s) {
  const int grid = a.B * a.N * a.chunks;
  return launch_pdl(k_verify, dim3(grid), dim3(VERIFY_THREADS), 0, s, a);
}

// ---------------------------------------------------------------------------
// Library-owned scratch for tree_verify_greedy_noalloc.
//
// Some callers cannot hand the library a workspace: plugins inside another
// engine that only receive their input and output buffers, or code on a
// latency-critical path where a cudaMalloc (which may synchronise the device)
// is not allowed.  For them the verify kernel can run on this fixed array,
// which every GPU that loads the library holds until the process exits.
// Host code must not use the array's name as a pointer (on the host it names
// a stand-in, not device memory): its device address is looked up once per
// device with cudaGetSymbolAddress, with that device current.
static __device__ __align__(256) unsigned char g_verify_scratch[TS_VERIFY_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
void* g_verify_scratch_addr[kMaxDevices] = {};
std::mutex g_verify_scratch_mu;
}  // namespace

// Device address and size of the scratch array on the current device; the
// first call on a device performs the lookup.
ts_status verify_static_scratch(void** ptr, size_t* bytes) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TS_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TS_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_verify_scratch_mu);
  if (!g_verify_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || !p) return TS_ERR_CUDA;
    g_verify_scratch_addr[dev] = p;
  }
  *ptr = g_verify_scratch_addr[dev];
  *bytes = sizeof(g_verify_scratch);
  return TS_OK;
}

}  // namespace ts
