// Stochastic (temperature) verification of a scored draft tree by recursive
// rejection sampling.
//
// [P3] Production Inference Runtimes section: each accepted token is checked
// against the target's own distribution by rejection sampling, so the output
// follows the target exactly.  [P1] Key Mechanisms > Multi-Token Acceptance &
// Rollback: the accepted branch is kept up to the first rejection.  For
// several drafts under one node (siblings drawn from the draft distribution
// without replacement) the siblings are tried in index order:
//   accept child c (token x)  iff  coins[c] * q'(x) < r(x);
//   on rejection  r  <- normalise(max(r - q', 0)),  q'(x) <- 0, q' renormalised;
// starting from r = softmax(l_u / T), q' = q_u.  When no child is accepted
// (or u is a leaf) the bonus token is drawn from r by inversion with coins[0].
//
// Design.  The walk only ever needs the rows of the nodes it visits, so it is
// run lazily, one sequence per thread-block cluster of C CTAs.  CTA k of the
// cluster owns vocabulary slice [k*S, (k+1)*S) and holds, in shared memory, its
// slice of the visited node's target logits and draft probabilities (brought
// in by one bulk copy each).  Per visited node:
//   1. local max and sum of exp((l - max)/T), one cluster exchange -> the
//      global normaliser and a rescale factor per CTA;
//   2. every CTA gathers r(x), q'(x) of the node's children tokens from their
//      owners over distributed shared memory, so each acceptance test is local;
//   3. each rejection costs one slice pass (sum of the residual) and one
//      exchange, then an in-place update of the slice;
//   4. the bonus draw locates the owning CTA from the per-CTA masses and that
//      CTA scans its slice.
// Every CTA takes every decision itself from exchanged values read in the same
// order with the same fp32 operations, so the CTAs of a cluster never diverge.
// Reuse of a buffer or an exchange slot is ordered by the cluster barriers:
// records alternate between two slots, and a CTA overwrites its slices only
// after every CTA has signalled that its gathers for the node are done.
#include <float.h>

#include "internal.cuh"
#include "sm100.cuh"

namespace ts {
namespace {

using namespace sm100;

constexpr int ST_WARPS = STOCH_THREADS / 32;
constexpr uint64_t WAIT_NS = 200ull * 1000 * 1000;  // a bulk copy that takes this long is an error

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cl_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cl_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_peer_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ int ld_peer_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// One bulk copy global -> this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// What each CTA publishes at an exchange.
struct Rec {
  float a, b;
  int err, pad;
};

struct Shared {
  int parent[MAX_NODES];
  int draft[MAX_NODES];
  int kid_start[MAX_NODES + 1];
  int kid_cnt[MAX_NODES];
  int kids[MAX_NODES];
  int path[MAX_NODES];
  float cr[MAX_NODES];  // residual mass r(x) * S of the current node's children tokens
  float cq[MAX_NODES];  // draft probability q(x) of the same tokens (0 once excluded)
  Rec rec[2];           // exchange slots, alternating
  Rec all[STOCH_MAX_CLUSTER];
  float fac[STOCH_MAX_CLUSTER];  // per-CTA rescale of the slice values
  float tot[STOCH_MAX_CLUSTER];  // per-CTA mass of the current residual
  float red[ST_WARPS + 1];
  int claim;
  uint64_t bar;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <bool MAX>
__device__ float block_reduce(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = MAX ? warp_max(v) : warp_sum(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float w = lane < ST_WARPS ? red[lane] : (MAX ? -FLT_MAX : 0.f);
    w = MAX ? warp_max(w) : warp_sum(w);
    if (lane == 0) red[ST_WARPS] = w;
  }
  __syncthreads();
  return red[ST_WARPS];
}

// The residual update of one element: max(f * rho - k * q, 0), written with
// explicit roundings so that every CTA that evaluates it for the same inputs
// gets the same bits.
__device__ __forceinline__ float residual(float rho_scaled, float k, float q) {
  return fmaxf(__fmaf_rn(-k, q, rho_scaled), 0.f);
}

// Exchange: publish (a, b, err) and read every CTA's record, in rank order, into sh.all.
__device__ void exchange(Shared& sh, int& xcnt, bool& pending, int C, float a, float b, int err) {
  if (pending) {
    cl_wait();
    pending = false;
  }
  Rec* slot = &sh.rec[xcnt & 1];
  if (threadIdx.x == 0) *slot = Rec{a, b, err, 0};
  cl_arrive();
  cl_wait();
  if ((int)threadIdx.x < C) {
    const uint32_t base = peer_addr(slot, threadIdx.x);
    sh.all[threadIdx.x] = Rec{ld_peer_f32(base), ld_peer_f32(base + 4), ld_peer_s32(base + 8), 0};
  }
  __syncthreads();
  ++xcnt;
}

__global__ void __launch_bounds__(STOCH_THREADS, 1) k_verify_stoch(StochArgs a) {
  extern __shared__ __align__(128) float dyn[];
  __shared__ Shared sh;
  float* bufL = dyn;             // slice of the node's target logits, then of the residual
  float* bufQ = dyn + a.slice;   // slice of the node's draft probabilities
  const int C = a.cluster;
  const int rank = (int)cluster_rank();
  const int b = blockIdx.y;
  const int tid = threadIdx.x;
  const int N = a.N, V = a.V;
  const int v0 = rank * a.slice;
  const int len = max(0, min(a.slice, V - v0));

  if (tid == 0) {
    mbar_init(&sh.bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  // Bring in one node's slices (logits always, draft probabilities if it has children).
  uint32_t phase = 0;
  auto issue = [&](int u, bool with_q) {
    const size_t row = ((size_t)b * N + u) * (size_t)V + v0;
    if (a.bulk) {
      if (tid == 0) {
        // order this CTA's earlier generic-proxy accesses of the slices before the copy's writes
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const uint32_t bytes = (uint32_t)len * 4u;
        mbar_arrive_expect_tx(&sh.bar, with_q ? 2u * bytes : bytes);
        if (bytes) {
          bulk_load(bufL, a.logits + row, bytes, &sh.bar);
          if (with_q) bulk_load(bufQ, a.q + row, bytes, &sh.bar);
        }
      }
    } else {
      for (int i = tid; i < len; i += STOCH_THREADS) {
        bufL[i] = a.logits[row + i];
        if (with_q) bufQ[i] = a.q[row + i];
      }
    }
  };
  auto land = [&]() -> bool {  // wait for the slices issued last; false on time-out
    if (!a.bulk) {
      __syncthreads();
      return true;
    }
    const bool ok = mbar_wait(&sh.bar, phase, WAIT_NS);
    phase ^= 1u;
    return __syncthreads_and(ok) != 0;
  };

  issue(0, N > 1);

  // tree and draft tokens; every CTA checks them and reaches the same verdict
  bool bad = false;
  for (int i = tid; i < N; i += STOCH_THREADS) {
    const int p = a.parent[(size_t)b * N + i];
    const int d = a.draft[(size_t)b * N + i];
    sh.parent[i] = p;
    sh.draft[i] = d;
    sh.kid_cnt[i] = 0;
    bad |= (i == 0) ? (p != -1) : (p < 0 || p >= i || d < 0 || d >= V);
  }
  if (__syncthreads_or(bad)) {
    const bool landed = land();
    (void)landed;
    if (rank == 0 && tid == 0) {
      for (int d = 0; d <= a.max_depth; ++d) a.accepted[(size_t)b * (a.max_depth + 1) + d] = -1;
      a.accept_len[b] = 0;
      a.bonus[b] = 0;
      a.status[b] = TS_ERR_BAD_TREE;
    }
    return;  // no distributed shared memory was touched
  }
  // children lists in index order
  for (int c = 1 + tid; c < N; c += STOCH_THREADS) atomicAdd(&sh.kid_cnt[sh.parent[c]], 1);
  __syncthreads();
  if (tid == 0) {
    int s = 0;
    for (int u = 0; u < N; ++u) {
      sh.kid_start[u] = s;
      s += sh.kid_cnt[u];
    }
    sh.kid_start[N] = s;
    sh.path[0] = 0;
  }
  __syncthreads();
  for (int c = 1 + tid; c < N; c += STOCH_THREADS) {
    const int p = sh.parent[c];
    int r = 0;
    for (int j = 1; j < c; ++j) r += (sh.parent[j] == p);
    sh.kids[sh.kid_start[p] + r] = c;
  }
  __syncthreads();

  const float kT = a.inv_temp_log2e;
  int xcnt = 0;
  bool pending = false;  // a "done reading peers' slices" arrive not yet waited on
  int err = 0;
  int depth = 0;
  int u = 0;
  bool first = true;

  while (true) {
    const int nk = sh.kid_cnt[u];
    if (!first) {
      if (pending) {
        cl_wait();
        pending = false;
      }
      issue(u, nk > 0);
    }
    first = false;
    if (!land()) err = 1;

    // 1. normaliser of softmax(l / T) over the vocabulary
    float m = -FLT_MAX;
    for (int i = tid; i < len; i += STOCH_THREADS) m = fmaxf(m, bufL[i]);
    const float m_me = block_reduce<true>(m, sh.red);
    float s = 0.f;
    for (int i = tid; i < len; i += STOCH_THREADS) {
      const float e = exp2f((bufL[i] - m_me) * kT);
      bufL[i] = e;
      s += e;
    }
    const float s_me = block_reduce<false>(s, sh.red);
    exchange(sh, xcnt, pending, C, len > 0 ? m_me : -FLT_MAX, s_me, err);
    int err_any = 0;
    float gm = -FLT_MAX;
    for (int r = 0; r < C; ++r) {
      err_any |= sh.all[r].err;
      gm = fmaxf(gm, sh.all[r].a);
    }
    if (err_any) {
      err = 1;
      break;
    }
    float S = 0.f;
    float fac_me = 1.f;
    if (tid < C) {
      const float f = exp2f((sh.all[tid].a - gm) * kT);
      sh.fac[tid] = f;
      sh.tot[tid] = __fmul_rn(f, sh.all[tid].b);
    }
    __syncthreads();
    for (int r = 0; r < C; ++r) S = __fadd_rn(S, sh.tot[r]);
    fac_me = sh.fac[rank];

    // 2. gather the children tokens' values from their owners
    const int k0 = sh.kid_start[u];
    for (int j = tid; j < nk; j += STOCH_THREADS) {
      const int x = sh.draft[sh.kids[k0 + j]];
      const int o = x / a.slice;
      const int off = x - o * a.slice;
      sh.cr[j] = __fmul_rn(sh.fac[o], ld_peer_f32(peer_addr(bufL + off, o)));
      sh.cq[j] = ld_peer_f32(peer_addr(bufQ + off, o));
    }
    cl_arrive();  // this CTA is done reading its peers' slices for node u
    pending = true;
    __syncthreads();

    // 3. try the children in index order
    float Qm = 1.f;  // draft mass left after excluding rejected tokens
    int next = -1;
    for (int j = 0; j < nk; ++j) {
      const int c = sh.kids[k0 + j];
      const int x = sh.draft[c];
      const float coin = a.coins[(size_t)b * N + c];
      const float rx = sh.cr[j], qx = sh.cq[j];
      const bool acc = Qm > 0.f ? (__fmul_rn(__fmul_rn(coin, qx), S) < __fmul_rn(rx, Qm)) : (rx > 0.f);
      if (acc) {
        next = c;
        break;
      }
      if (Qm > 0.f) {
        // residual: r <- max(r - q', 0), in the slice's own scale: rho <- max(f*rho - (S/Qm)*q, 0)
        const float kq = __fdiv_rn(S, Qm);
        float t = 0.f;
        for (int i = tid; i < len; i += STOCH_THREADS) t += residual(__fmul_rn(fac_me, bufL[i]), kq, bufQ[i]);
        const float t_me = block_reduce<false>(t, sh.red);
        exchange(sh, xcnt, pending, C, t_me, 0.f, 0);
        float S2 = 0.f;
        for (int r = 0; r < C; ++r) S2 = __fadd_rn(S2, sh.all[r].a);
        if (S2 > 0.f) {
          for (int i = tid; i < len; i += STOCH_THREADS) bufL[i] = residual(__fmul_rn(fac_me, bufL[i]), kq, bufQ[i]);
          for (int jj = j + 1 + tid; jj < nk; jj += STOCH_THREADS) sh.cr[jj] = residual(sh.cr[jj], kq, sh.cq[jj]);
          if (tid < C) {
            sh.fac[tid] = 1.f;
            sh.tot[tid] = sh.all[tid].a;
          }
          fac_me = 1.f;
          S = S2;
        }
        __syncthreads();  // every thread is done with bufQ before x's entry is cleared
      }
      // take x out of the draft distribution
      Qm = __fsub_rn(Qm, qx);
      const int o = x / a.slice;
      if (o == rank && tid == 0) bufQ[x - o * a.slice] = 0.f;
      for (int jj = j + 1 + tid; jj < nk; jj += STOCH_THREADS)
        if (sh.draft[sh.kids[k0 + jj]] == x) sh.cq[jj] = 0.f;
      __syncthreads();
    }
    if (next >= 0) {
      ++depth;
      if (tid == 0) sh.path[depth] = next;
      u = next;
      continue;  // the next iteration waits on the arrive above before reusing the slices
    }

    // 4. bonus token: smallest v with cumulative residual mass > coins[0] * S
    const float t_all = __fmul_rn(a.coins[(size_t)b * N], S);
    int owner = -1;
    float base = 0.f, cum = 0.f;
    for (int r = 0; r < C; ++r) {
      const float nc = __fadd_rn(cum, sh.tot[r]);
      if (owner < 0 && nc > t_all) {
        owner = r;
        base = cum;
      }
      cum = nc;
    }
    bool last_positive = false;
    if (owner < 0) {  // rounding left the target beyond the total: take the last token with mass
      for (int r = C - 1; r >= 0; --r)
        if (sh.tot[r] > 0.f) {
          owner = r;
          break;
        }
      last_positive = true;
    }
    if (owner == rank) {
      const float tt = __fsub_rn(t_all, base);
      const int per = (len + STOCH_THREADS - 1) / STOCH_THREADS;
      const int lo = min(len, tid * per), hi = min(len, lo + per);
      float mine = 0.f;
      for (int i = lo; i < hi; ++i) mine = __fadd_rn(mine, __fmul_rn(fac_me, bufL[i]));
      // exclusive scan of the per-thread sums
      const int lane = tid & 31, warp = tid >> 5;
      float inc = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (lane == 31) sh.red[warp] = inc;
      if (tid == 0) sh.claim = INT_MAX;
      __syncthreads();
      if (warp == 0) {
        float w = lane < ST_WARPS ? sh.red[lane] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, w, o);
          if (lane >= o) w += y;
        }
        if (lane < ST_WARPS) sh.red[lane] = w - sh.red[lane];  // exclusive prefix of the warps
      }
      __syncthreads();
      const float excl = sh.red[warp] + (inc - mine);
      // A thread whose range ends beyond the target claims the first token in
      // it where the running mass passes the target; the smallest claim wins,
      // so a rounding gap between two ranges only moves the draw to the
      // neighbouring token with mass.
      int found = -1;
      if (!last_positive && lo < hi) {
        const float d = __fsub_rn(tt, excl);
        if (d < mine) {
          float acc = 0.f;
          for (int i = lo; i < hi; ++i) {
            const float w = __fmul_rn(fac_me, bufL[i]);
            acc = __fadd_rn(acc, w);
            if (acc > d && w > 0.f) {
              found = i;
              break;
            }
          }
        }
      }
      if (found >= 0) atomicMin(&sh.claim, found);
      __syncthreads();
      if (sh.claim == INT_MAX) {  // take the last token of the slice with mass
        int lastpos = -1;
        for (int i = lo; i < hi; ++i)
          if (bufL[i] > 0.f) lastpos = i;
        __syncthreads();
        if (tid == 0) sh.claim = -1;
        __syncthreads();
        if (lastpos >= 0) atomicMax(&sh.claim, lastpos);
        __syncthreads();
      }
      if (tid == 0) a.bonus[b] = v0 + max(sh.claim, 0);
    }
    break;
  }

  // write the path (CTA 0), then make sure no peer still reads this CTA's
  // shared memory before it exits
  if (rank == 0 && tid == 0) {
    const size_t row = (size_t)b * (a.max_depth + 1);
    const bool fits = depth <= a.max_depth;
    for (int d = 0; d <= a.max_depth; ++d) a.accepted[row + d] = (fits && !err && d <= depth) ? sh.path[d] : -1;
    a.accept_len[b] = err ? 0 : depth;
    if (err) {
      a.bonus[b] = 0;
      a.status[b] = TS_ERR_TIMEOUT;
    } else if (!fits) {
      a.status[b] = TS_ERR_SHAPE;
    }
  }
  if (err && a.bulk) {
    // a copy that timed out may still be in flight into this CTA's slices
    const bool landed = mbar_wait(&sh.bar, phase ^ 1u, WAIT_NS);
    (void)landed;
  }
  if (pending) cl_wait();
  cl_arrive();
  cl_wait();
}

}  // namespace

cudaError_t stoch_prepare() {
  const size_t smem = (size_t)2 * STOCH_MAX_SLICE * sizeof(float);
  return cudaFuncSetAttribute(k_verify_stoch, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_verify_stoch(const StochArgs& a, cudaStream_t s) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.cluster, a.B);
  cfg.blockDim = dim3(STOCH_THREADS);
  cfg.dynamicSmemBytes = (size_t)2 * a.slice * sizeof(float);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = a.cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_verify_stoch, a);
}

}  // namespace ts
