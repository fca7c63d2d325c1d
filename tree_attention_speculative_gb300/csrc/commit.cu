// Commit the accepted path's keys/values to the paged KV cache.
//
// [P1] Key Mechanisms > Speculative KV Cache Reuse (the tree's keys/values are
// reused, not recomputed), Multi-Token Acceptance & Rollback (the accepted
// path is kept, rejected branches discarded) and Integration with Speculative
// Decoding (the accepted prefix is appended and generation continues).
//
// The root (the last verified token, attended at position P_b) and the
// accepted drafts x1..n* become prefix tokens P_b .. P_b + L.  Rejected
// branches need no work: their keys/values never entered the cache.
//
// One CTA per sequence.  Every thread first checks the destinations it will
// write (block table entry inside the pool, node id inside the tree); if any
// is bad the sequence commits nothing and reports TS_ERR_BAD_BLOCK, so a
// sequence is never left half-committed.  Then the rows move with 16-byte
// loads and stores.  The new prefix length is written after a barrier, so it
// may alias the prefix-length input.
#include "internal.cuh"

namespace ts {

__global__ void __launch_bounds__(256)
k_commit(CommitArgs a) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const int P = a.prefix_len[b];
  const int st = a.status ? a.status[b] : TS_OK;
  const int L = a.accept_len[b];
  const int vec = a.D / 8;  // uint4 per key row
  // P bounded so that every position P + d stays far inside int range
  const bool commit = (st == TS_OK) && L >= 0 && L <= a.max_depth && P >= 0 && P <= (1 << 30);
  const int n = commit ? (L + 1) * a.Hkv * vec : 0;

  // validate every destination before writing any
  bool ok = true;
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int d = e / (a.Hkv * vec);
    const int node = a.accepted[(size_t)b * (a.max_depth + 1) + d];
    const int t = P + d;
    const int bi = t / a.bs;
    const int blk = (bi >= 0 && bi < a.max_blocks) ? a.block_table[(size_t)b * a.max_blocks + bi] : -1;
    ok = ok && node >= 0 && node < a.N && blk >= 0 && blk < a.num_blocks;
  }
  const int all_ok = __syncthreads_and(ok);
  if (commit && all_ok) {
    for (int e = threadIdx.x; e < n; e += blockDim.x) {
      const int d = e / (a.Hkv * vec);
      const int rem = e - d * (a.Hkv * vec);
      const int g = rem / vec;
      const int c = rem - g * vec;
      const int node = a.accepted[(size_t)b * (a.max_depth + 1) + d];
      const int t = P + d;
      const int blk = a.block_table[(size_t)b * a.max_blocks + t / a.bs];
      const size_t src = (((size_t)b * a.N + node) * a.Hkv + g) * a.D + c * 8;
      const size_t dst = (((size_t)blk * a.Hkv + g) * a.bs + (t % a.bs)) * a.D + c * 8;
      reinterpret_cast<uint4*>(a.k_cache + dst)[0] = reinterpret_cast<const uint4*>(a.k_tree + src)[0];
      reinterpret_cast<uint4*>(a.v_cache + dst)[0] = reinterpret_cast<const uint4*>(a.v_tree + src)[0];
    }
  }
  __syncthreads();  // every thread has read prefix_len[b] before it may be overwritten
  if (threadIdx.x == 0) {
    a.new_prefix_len[b] = (commit && all_ok) ? P + L + 1 : P;
    if (commit && !all_ok && a.status) a.status[b] = TS_ERR_BAD_BLOCK;
  }
}

cudaError_t launch_commit(const CommitArgs& a, cudaStream_t s) {
  return launch_pdl(k_commit, dim3(a.B), dim3(256), 0, s, a);
}

}  // namespace ts
