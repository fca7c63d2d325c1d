// Ancestry bitmasks, depths and positions of a flattened draft tree.
//
// [P1] Key Mechanisms > Modified Causal Attention Mask; [P2] How It Works and
// Tradeoffs ("position bookkeeping"); [P3] code listing,
// build_tree_attention_mask (walk parent pointers to the root).
//
// A forest (several roots, [P3] The Future of Reasoning) differs only in the
// validity rule: any node may have parent -1; every chain then stops at its
// own root.
//
// One CTA per sequence, one thread per node.  Parents are staged in shared
// memory; each thread validates its own parent pointer, the CTA agrees on the
// tree's validity with one barrier-and, then each node walks its chain to the
// root (at most depth <= i steps, since parents precede children), setting one
// bit per visited node.  Latency bound: a few hundred nanoseconds of work.
#include "internal.cuh"

namespace ts {

__global__ void __launch_bounds__(MAX_NODES)
k_ancestry(const int32_t* __restrict__ parent, const int32_t* __restrict__ prefix_len, int N, int W,
           uint64_t* __restrict__ anc, int32_t* __restrict__ depth, int32_t* __restrict__ pos,
           int32_t* __restrict__ status, int forest) {
  __shared__ int sp[MAX_NODES];
  const int b = blockIdx.x;
  const int i = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  const int P = prefix_len[b];  // loaded beside the parents, not after the walk
  int p = -1;
  bool ok = true;
  if (i < N) {
    p = parent[(size_t)b * N + i];
    // a forest may start a new tree (parent -1) at any node; node 0 is always a root
    ok = (i == 0) ? (p == -1) : ((p >= 0 && p < i) || (forest && p == -1));
    sp[i] = p;
  }
  const int valid = __syncthreads_and(ok);
  if (i < N) {
    uint64_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
    int d = 0;
    if (valid) {
      int c = i;
      while (true) {
        const uint64_t bit = 1ull << (c & 63);
        switch (c >> 6) {
          case 0: w0 |= bit; break;
          case 1: w1 |= bit; break;
          case 2: w2 |= bit; break;
          default: w3 |= bit; break;
        }
        c = sp[c];
        if (c < 0) break;
        ++d;
      }
    }
    uint64_t* row = anc + ((size_t)b * N + i) * W;
    row[0] = w0;
    if (W > 1) row[1] = w1;
    if (W > 2) row[2] = w2;
    if (W > 3) row[3] = w3;
    depth[(size_t)b * N + i] = d;
    pos[(size_t)b * N + i] = valid ? P + d : 0;
  }
  if (i == 0) status[b] = valid ? TS_OK : TS_ERR_BAD_TREE;
}

cudaError_t launch_ancestry(const int32_t* parent, const int32_t* prefix_len, int B, int N,
                            uint64_t* anc, int32_t* depth, int32_t* pos, int32_t* status,
                            cudaStream_t s, int forest) {
  const int threads = ceil_div(N, 32) * 32;
  return launch_pdl(k_ancestry, dim3(B), dim3(threads), 0, s, parent, prefix_len, N, ceil_div(N, 64), anc, depth,
                    pos, status, forest);
}

}  // namespace ts
