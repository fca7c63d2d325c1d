// Split combine: merge the per-split partial results of the prefix sweep.
//
// The verification pass of [P1] Key Mechanisms > Batched Parallel Verification
// is one softmax over all keys a node sees.  The prefix is cut into splits so
// that enough CTAs share the work; each split s leaves a normalised partial
// O_s and its base-2 log-sum-exp L_s.  The exact softmax over the union is
//     out = sum_s 2^(L_s - M) O_s / sum_s 2^(L_s - M),  M = max_s L_s,
//     lse = ln 2 * (M + log2 sum_s 2^(L_s - M)).
// One warp per output row (b, node, head); each lane owns D/32 consecutive
// channels, so partial reads and the bf16 store are coalesced.
#include "internal.cuh"

namespace ts {

template <int D>
__global__ void __launch_bounds__(256)
k_combine(AttnArgs a) {
  constexpr int PER = D / 32;
  const int rows = a.B * a.N * a.Hq;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  if (row >= rows) return;
  const int b = row / (a.N * a.Hq);
  int P;
  usable_prefix(a.prefix_len[b], a.chunk_tiles, a.max_splits, a.bs, a.max_blocks, &P);
  const int ns = num_splits(P, a.chunk_tiles);
  const size_t stride_lse = (size_t)rows;
  const size_t stride_o = (size_t)rows * D;

  // every split's lse in flight at once: lane s holds split s (then s+32, ...)
  float m = -INFINITY;
  for (int s = lane; s < ns; s += 32) m = fmaxf(m, a.part_lse[s * stride_lse + row]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;
  float den = 0.f;
  // partial rows: up to 8 independent loads in flight per lane
  for (int s0 = 0; s0 < ns; s0 += 8) {
    float w[8];
    float v[8][PER];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int s = s0 + i;
      w[i] = 0.f;
      if (s < ns) {
        w[i] = a.part_lse[s * stride_lse + row];
        const float* o = a.part_o + s * stride_o + (size_t)row * D + lane * PER;
        if constexpr (PER == 4) {
          const float4 x = *reinterpret_cast<const float4*>(o);
          v[i][0] = x.x; v[i][1] = x.y; v[i][2] = x.z; v[i][3] = x.w;
        } else {
          const float2 x = *reinterpret_cast<const float2*>(o);
          v[i][0] = x.x; v[i][1] = x.y;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (s0 + i < ns) {
        const float wi = exp2f(w[i] - m);
        den += wi;
#pragma unroll
        for (int k = 0; k < PER; ++k) acc[k] = fmaf(wi, v[i][k], acc[k]);
      }
    }
  }
  const float inv = 1.f / den;
  __nv_bfloat16* dst = a.out + (size_t)row * D + lane * PER;
#pragma unroll
  for (int k = 0; k < PER; k += 2)
    *reinterpret_cast<__nv_bfloat162*>(dst + k) = __floats2bfloat162_rn(acc[k] * inv, acc[k + 1] * inv);
  if (a.lse && lane == 0) a.lse[row] = (m + log2f(den)) * 0.69314718055994531f;
}

cudaError_t launch_combine(const AttnArgs& a, cudaStream_t s) {
  const int rows = a.B * a.N * a.Hq;
  const int grid = ceil_div(rows, 8);
  return a.D == 128 ? launch_pdl(k_combine<128>, dim3(grid), dim3(256), 0, s, a)
                   : launch_pdl(k_combine<64>, dim3(grid), dim3(256), 0, s, a);
}

}  // namespace ts
