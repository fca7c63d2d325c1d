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
// run lazily, one sequence per thread-block cluster of C CTAs (C up to 16 where
// the GPU allows non-portable clusters, else 8).  CTA k of the cluster owns
// vocabulary slice [k*S, (k+1)*S) and holds, in shared memory, its slice of the
// visited node's target logits and draft probabilities (one bulk copy each).
// Per visited node:
//   1. the slice's (max, sum of exp((l - max)/T)) in one pass; one cluster
//      exchange gives the global normaliser and a rescale factor per CTA;
//   2. every CTA reads the node's children tokens' logits and draft
//      probabilities from global memory itself (while the slices land) and
//      rescales them as their owner would, so each acceptance test is local;
//   3. each rejection costs one slice pass (sum of the residual), one
//      exchange and an in-place update of the slice;
//   4. the bonus draw locates the owning CTA from the per-CTA masses, and that
//      CTA scans its slice, each warp a contiguous run read lane by lane.
// Every CTA takes every decision itself from exchanged values read in the same
// order with the same fp32 operations, so the CTAs of a cluster never diverge.
// An exchange is one 16-byte record per CTA pushed into every peer's shared
// memory (st.async, completing on the receiver's mbarrier): no cluster-wide
// barrier on the walk, and no CTA ever reads another's slices.
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
// One bulk copy global -> this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

struct Shared {
  int parent[MAX_NODES];
  int draft[MAX_NODES];
  int has_kids[MAX_NODES];
  int kid_list[MAX_NODES];  // the current node's children, in index order
  int path[MAX_NODES];
  float cl[MAX_NODES];  // target logit of each child's token at the current node
  float cr[MAX_NODES];  // its residual mass r(x) * S
  float cq[MAX_NODES];  // its draft probability q(x) (0 once excluded)
  float coin[MAX_NODES];
  float4 xrec[2][STOCH_MAX_CLUSTER];  // exchange records, one slot per sending CTA, two exchanges in flight
  float4 all[STOCH_MAX_CLUSTER];      // the last exchange's records, copied out of the slot
  float fac[STOCH_MAX_CLUSTER];       // per-CTA rescale of the slice values
  float tot[STOCH_MAX_CLUSTER];       // per-CTA mass of the current residual
  float red[2 * ST_WARPS];
  float wm[ST_WARPS], ws[ST_WARPS];   // each warp's (max, sum) from the normaliser pass
  float wmass[ST_WARPS];              // each warp's residual mass once the slice holds residuals
  float wpend[ST_WARPS];              // the same for a residual being computed
  float S;
  int nk;
  int xerr;  // some CTA of the cluster reported an error at the last exchange
  int claim;
  uint64_t bar;      // the slices' bulk copies
  uint64_t xbar[2];  // arrival of every CTA's record for an exchange slot
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// exp((l - m) / T) as 2^((l - m) * log2(e) / T), with explicit roundings: every
// CTA that evaluates it for the same (l, m) gets the same bits.
__device__ __forceinline__ float unnorm_p(float l, float m, float kT) { return ex2(__fmul_rn(__fsub_rn(l, m), kT)); }

// The residual of one element: max(rho - k * q, 0), rho already in the common
// scale; explicit roundings for the same reason.
__device__ __forceinline__ float residual(float rho, float k, float q) { return fmaxf(__fmaf_rn(-k, q, rho), 0.f); }

// Merge two (max, sum of 2^((x - max) kT)) pairs.
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2, float kT) {
  const float mn = fmaxf(m, m2);
  s = __fmul_rn(s, unnorm_p(m, mn, kT)) + __fmul_rn(s2, unnorm_p(m2, mn, kT));
  m = mn;
}

// Store 16 bytes into a peer CTA's shared memory; completes on the peer's mbarrier.
__device__ __forceinline__ void st_async16(uint32_t dst, float4 v, uint32_t peer_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(dst),
               "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)),
               "r"(__float_as_uint(v.w)), "r"(peer_bar)
               : "memory");
}

// The current value of slice element x: while the slice still holds raw
// logits, the unnormalised target probability rescaled to the common scale;
// after the first residual update, the residual itself (scale 1).
struct SliceVal {
  float m, kT, f;
  bool raw;
  __device__ __forceinline__ float operator()(float x) const { return __fmul_rn(f, raw ? unnorm_p(x, m, kT) : x); }
};

__global__ void __launch_bounds__(STOCH_THREADS, 2) k_verify_stoch(StochArgs a) {
  extern __shared__ __align__(128) float dyn[];
  __shared__ Shared sh;
  float* bufL = dyn;            // slice of the node's target logits, then of the residual
  float* bufQ = dyn + a.slice;  // slice of the node's draft probabilities
  const int C = a.cluster;
  const int rank = (int)cluster_rank();
  const int b = blockIdx.y;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int N = a.N, V = a.V;
  const int v0 = rank * a.slice;
  const int len = max(0, min(a.slice, V - v0));
  // The slice as float4 (padded to a multiple of 4 with tokens of no mass);
  // warp w walks the contiguous run [wlo, whi) of it, lane by lane.
  const int len4 = (len + 3) >> 2;
  const int run4 = (len4 + ST_WARPS - 1) / ST_WARPS;
  const int wlo = min(len4, warp * run4), whi = min(len4, wlo + run4);
  float4* L4 = reinterpret_cast<float4*>(bufL);
  const float4* Q4 = reinterpret_cast<const float4*>(bufQ);
  const float kT = a.inv_temp_log2e;

  if (tid == 0) {
    mbar_init(&sh.bar, 1);
    mbar_init(&sh.xbar[0], 1);
    mbar_init(&sh.xbar[1], 1);
    fence_barrier_init();
  }
  __syncthreads();
  cl_arrive();  // this CTA's exchange barriers exist; waited on before the first record is sent
  pdl_wait();
  pdl_trigger();

  int err = 0;
  // Exchange: publish (a, b, err) to every CTA of the cluster and collect
  // everyone's record, in rank order, into sh.all.  Records go straight into
  // the peers' slots (st.async), completing on the peers' slot barrier, so no
  // cluster-wide barrier is needed.  Slot s is rewritten by a peer only after
  // that peer has this CTA's record of the next exchange, which is sent after
  // this CTA copied slot s out.
  int xcnt = 0;
  auto exchange = [&](float va, float vb, int e) {
    const int s = xcnt & 1;
    if (xcnt == 0) cl_wait();
    if (tid == 0) mbar_arrive_expect_tx(&sh.xbar[s], (uint32_t)C * 16u);
    if (tid < C) {
      const float4 rec = make_float4(va, vb, __int_as_float(e), 0.f);
      st_async16(peer_addr(&sh.xrec[s][rank], tid), rec, peer_addr(&sh.xbar[s], tid));
    }
    const bool ok = mbar_wait(&sh.xbar[s], (uint32_t)(xcnt >> 1) & 1u, WAIT_NS);
    if (tid < C) sh.all[tid] = sh.xrec[s][tid];
    if (!__syncthreads_and(ok)) err = 1;
    ++xcnt;
  };

  // Bring in one node's slices (logits always, draft probabilities if it has
  // children).  Lane 0 of warp 1 issues the bulk copies, so warp 0 is free to
  // fetch the children's values meanwhile.
  uint32_t phase = 0;
  auto issue = [&](int u, bool with_q) {
    const size_t row = ((size_t)b * N + u) * (size_t)V + v0;
    if (a.bulk) {
      if (tid == 32) {
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
      for (int i = tid; i < 4 * len4; i += STOCH_THREADS) {
        bufL[i] = i < len ? a.logits[row + i] : -FLT_MAX;
        if (with_q) bufQ[i] = i < len ? a.q[row + i] : 0.f;
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

  // tree and draft tokens; every CTA checks them and reaches the same conclusion
  bool bad = false;
  for (int i = tid; i < N; i += STOCH_THREADS) {
    const int p = a.parent[(size_t)b * N + i];
    const int d = a.draft[(size_t)b * N + i];
    sh.parent[i] = p;
    sh.draft[i] = d;
    sh.has_kids[i] = 0;
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
    cl_wait();
    return;  // no distributed shared memory was touched
  }
  for (int c = 1 + tid; c < N; c += STOCH_THREADS) sh.has_kids[sh.parent[c]] = 1;
  if (tid == 0) sh.path[0] = 0;

  int depth = 0;
  int u = 0;
  bool first = true;

  while (true) {
    __syncthreads();  // the previous node's reads of the slices and child arrays are done
    const size_t urow = ((size_t)b * N + u) * (size_t)V;
    // No CTA reads another's slices, so the next node's copy may start at once.
    if (!first) issue(u, sh.has_kids[u] != 0);
    first = false;
    // u's children in index order (warp ballots over the parent array)
    if (warp == 0) {
      int cnt = 0;
      for (int base = (u + 1) & ~31; base < N; base += 32) {
        const int c = base + lane;
        const bool kid = c > u && c < N && sh.parent[c] == u;
        const unsigned bal = __ballot_sync(0xffffffffu, kid);
        if (kid) sh.kid_list[cnt + __popc(bal & ((1u << lane) - 1u))] = c;
        cnt += __popc(bal);
      }
      if (lane == 0) sh.nk = cnt;
    }
    __syncthreads();
    const int k0 = 0;
    const int nk = sh.nk;
    // the children tokens' own values and coins, straight from global memory while the slices land
    for (int j = tid; j < nk; j += STOCH_THREADS) {
      const int c = sh.kid_list[k0 + j];
      const int x = sh.draft[c];
      sh.cl[j] = a.logits[urow + x];
      sh.cq[j] = a.q[urow + x];
      sh.coin[j] = a.coins[(size_t)b * N + c];
    }
    if (!land()) err = 1;

    // 1. normaliser of softmax(l / T): (max, sum of 2^((l - max) kT)) in one
    //    pass, eight float4 per thread at a time held in registers
    float m = -FLT_MAX, s = 0.f;
    for (int i0 = wlo + lane; i0 < whi; i0 += 8 * 32) {
      float4 l[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int i = i0 + 32 * k;
        l[k] = i < whi ? L4[i] : make_float4(-FLT_MAX, -FLT_MAX, -FLT_MAX, -FLT_MAX);
      }
      float mx = m;
#pragma unroll
      for (int k = 0; k < 8; ++k) mx = fmaxf(mx, fmaxf(fmaxf(l[k].x, l[k].y), fmaxf(l[k].z, l[k].w)));
      float part[4] = {__fmul_rn(s, unnorm_p(m, mx, kT)), 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        part[0] += unnorm_p(l[k].x, mx, kT);
        part[1] += unnorm_p(l[k].y, mx, kT);
        part[2] += unnorm_p(l[k].z, mx, kT);
        part[3] += unnorm_p(l[k].w, mx, kT);
      }
      s = (part[0] + part[1]) + (part[2] + part[3]);
      m = mx;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      merge_ms(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o), kT);
    if (lane == 0) {
      sh.wm[warp] = m;
      sh.ws[warp] = s;
    }
    __syncthreads();
    // every warp merges the warps' pairs in the same order
    m = lane < ST_WARPS ? sh.wm[lane] : -FLT_MAX;
    s = lane < ST_WARPS ? sh.ws[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      merge_ms(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o), kT);
    const float m_me = m;
    exchange(len > 0 ? m_me : -FLT_MAX, s, err);
    // warp 0 folds the records: global max, per-CTA factor and mass, total
    if (warp == 0) {
      const float4 rec = lane < C ? sh.all[lane] : make_float4(-FLT_MAX, 0.f, 0.f, 0.f);
      const int e_any = __any_sync(0xffffffffu, lane < C && __float_as_int(rec.z) != 0);
      float gm = rec.x;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
      const float f = unnorm_p(rec.x, gm, kT);
      const float t = __fmul_rn(f, rec.y);
      if (lane < C) {
        sh.fac[lane] = f;
        sh.tot[lane] = t;
      }
      __syncwarp();
      float tv[STOCH_MAX_CLUSTER];
#pragma unroll
      for (int r = 0; r < STOCH_MAX_CLUSTER; ++r) tv[r] = __shfl_sync(0xffffffffu, t, r);
      float S0 = 0.f;  // sequential, in rank order, as the bonus draw adds them up
#pragma unroll
      for (int r = 0; r < STOCH_MAX_CLUSTER; ++r)
        if (r < C) S0 = __fadd_rn(S0, tv[r]);
      if (lane == 0) {
        sh.S = S0;
        sh.xerr = e_any;
      }
      // 2. the children tokens' target mass in the common scale (what their owner computes)
      for (int j = lane; j < nk; j += 32) {
        const int o = sh.draft[sh.kid_list[k0 + j]] / a.slice;
        sh.cr[j] = __fmul_rn(sh.fac[o], unnorm_p(sh.cl[j], sh.all[o].x, kT));
      }
    }
    __syncthreads();
    if (sh.xerr) {
      err = 1;
      break;
    }
    float S = sh.S;
    SliceVal val{m_me, kT, sh.fac[rank], true};

    // 3. try the children in index order
    float Qm = 1.f;  // draft mass left after excluding rejected tokens
    int next = -1;
    for (int j = 0; j < nk; ++j) {
      const int c = sh.kid_list[k0 + j];
      const int x = sh.draft[c];
      const float rx = sh.cr[j], qx = sh.cq[j];
      const bool acc = Qm > 0.f ? (__fmul_rn(__fmul_rn(sh.coin[j], qx), S) < __fmul_rn(rx, Qm)) : (rx > 0.f);
      if (acc) {
        next = c;
        break;
      }
      if (Qm > 0.f) {
        // residual: r <- max(r - q', 0), in the common scale: rho <- max(rho - (S/Qm) q, 0)
        const float kq = __fdiv_rn(S, Qm);
        float t = 0.f;
        for (int i = wlo + lane; i < whi; i += 32) {
          const float4 l = L4[i], q = Q4[i];
          t += (residual(val(l.x), kq, q.x) + residual(val(l.y), kq, q.y)) +
               (residual(val(l.z), kq, q.z) + residual(val(l.w), kq, q.w));
        }
        t = warp_sum(t);
        if (lane == 0) sh.wpend[warp] = t;
        __syncthreads();
        const float t_me = warp_sum(lane < ST_WARPS ? sh.wpend[lane] : 0.f);
        exchange(t_me, 0.f, 0);
        float S2 = 0.f;
        for (int r = 0; r < C; ++r) S2 = __fadd_rn(S2, sh.all[r].x);
        if (err) break;
        if (S2 > 0.f) {
          for (int i = wlo + lane; i < whi; i += 32) {
            const float4 l = L4[i], q = Q4[i];
            L4[i] = make_float4(residual(val(l.x), kq, q.x), residual(val(l.y), kq, q.y),
                                residual(val(l.z), kq, q.z), residual(val(l.w), kq, q.w));
          }
          for (int jj = j + 1 + tid; jj < nk; jj += STOCH_THREADS) sh.cr[jj] = residual(sh.cr[jj], kq, sh.cq[jj]);
          if (tid < C) {
            sh.fac[tid] = 1.f;
            sh.tot[tid] = sh.all[tid].x;
          }
          if (tid < ST_WARPS) sh.wmass[tid] = sh.wpend[tid];
          val.raw = false;
          val.f = 1.f;
          S = S2;
        }
        __syncthreads();  // every thread is done with bufQ before x's entry is cleared
      }
      // take x out of the draft distribution
      Qm = __fsub_rn(Qm, qx);
      const int o = x / a.slice;
      if (o == rank && tid == 0) bufQ[x - o * a.slice] = 0.f;
      for (int jj = j + 1 + tid; jj < nk; jj += STOCH_THREADS)
        if (sh.draft[sh.kid_list[k0 + jj]] == x) sh.cq[jj] = 0.f;
      __syncthreads();
    }
    if (err) break;
    if (next >= 0) {
      ++depth;
      if (tid == 0) sh.path[depth] = next;
      u = next;
      continue;
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
      // each warp's mass is known from the last pass over the slice
      auto wmass = [&](int w) -> float {
        return val.raw ? __fmul_rn(val.f, __fmul_rn(sh.ws[w], unnorm_p(sh.wm[w], m_me, kT))) : sh.wmass[w];
      };
      // the warp whose run holds the target: the first whose running total passes it
      const float t_me = __fsub_rn(t_all, base);
      int tw = -1;
      float excl = 0.f;
      for (int w = 0; w < ST_WARPS && tw < 0; ++w) {
        const float nx = __fadd_rn(excl, wmass(w));
        if (nx > t_me) tw = w;
        else excl = nx;
      }
      if (tid == 0) sh.claim = INT_MAX;
      __syncthreads();
      // That warp finds the lane whose group of the run holds the target (each
      // lane sums a contiguous group of float4, reading it in an order rotated
      // by the lane so that the lanes hit different banks); then the warp walks
      // that group one token per lane to the first token with mass where the
      // running sum passes the target.  If rounding leaves the target beyond
      // the last group, the run's last token with mass is taken.
      if (!last_positive && warp == tw && wlo < whi) {
        const float d = __fsub_rn(t_me, excl);
        const int g4 = (whi - wlo + 31) >> 5;  // float4 per lane group
        const int glo = min(whi, wlo + lane * g4), ghi = min(whi, glo + g4);
        const int rot = lane % g4;
        float gs = 0.f;
        for (int k = 0; k < g4; ++k) {
          int idx = k + rot;
          if (idx >= g4) idx -= g4;
          const int i = glo + idx;
          if (i < ghi) {
            const float4 l = L4[i];
            gs += (val(l.x) + val(l.y)) + (val(l.z) + val(l.w));
          }
        }
        float inc = gs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, gs > 0.f && inc > d);
        const unsigned any = __ballot_sync(0xffffffffu, gs > 0.f);
        // the group that passes the target, else the run's last group with mass
        const int L = hit ? __ffs(hit) - 1 : (any ? 31 - __clz(any) : -1);
        if (L >= 0) {
          float run = __shfl_sync(0xffffffffu, inc - gs, L);
          const int e_lo = 4 * __shfl_sync(0xffffffffu, glo, L), e_hi = 4 * __shfl_sync(0xffffffffu, ghi, L);
          int pick = -1, lastpos = -1;
          for (int e0 = e_lo; e0 < e_hi && pick < 0; e0 += 32) {
            const int e = e0 + lane;
            const float w = e < e_hi ? val(bufL[e]) : 0.f;
            float ew = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const float y = __shfl_up_sync(0xffffffffu, ew, o);
              if (lane >= o) ew += y;
            }
            const unsigned pos = __ballot_sync(0xffffffffu, w > 0.f);
            const unsigned pass = __ballot_sync(0xffffffffu, w > 0.f && __fadd_rn(run, ew) > d);
            if (pass) pick = e0 + __ffs(pass) - 1;
            if (pos) lastpos = e0 + 31 - __clz(pos);
            run = __fadd_rn(run, __shfl_sync(0xffffffffu, ew, 31));
          }
          if (lane == 0 && (pick >= 0 || lastpos >= 0)) sh.claim = pick >= 0 ? pick : lastpos;
        }
      }
      __syncthreads();
      if (sh.claim == INT_MAX) {  // take the last token of the slice with mass
        int lastpos = -1;
        for (int i = tid; i < 4 * len4; i += STOCH_THREADS)
          if (val(bufL[i]) > 0.f) lastpos = i;
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

  // write the path (CTA 0); then no CTA exits while a peer may still send it a record
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
  if (xcnt == 0) cl_wait();
  cl_arrive();
  cl_wait();
}

}  // namespace

// Opt-ins, once per device: the slices' shared memory and, where the GPU
// allows it, clusters of 16 CTAs (otherwise clusters stay at 8).
cudaError_t stoch_prepare(int* max_cluster) {
  const size_t smem = (size_t)2 * STOCH_MAX_SLICE * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(k_verify_stoch, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  *max_cluster = STOCH_PORTABLE_CLUSTER;
  if (cudaFuncSetAttribute(k_verify_stoch, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    (void)cudaGetLastError();
    return cudaSuccess;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(STOCH_MAX_CLUSTER, 1);
  cfg.blockDim = dim3(STOCH_THREADS);
  cfg.dynamicSmemBytes = (size_t)2 * 8192 * sizeof(float);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = STOCH_MAX_CLUSTER;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_verify_stoch, &cfg) == cudaSuccess && n > 0)
    *max_cluster = STOCH_MAX_CLUSTER;
  else
    (void)cudaGetLastError();
  return cudaSuccess;
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
