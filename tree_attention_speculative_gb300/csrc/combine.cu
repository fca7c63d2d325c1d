// Split combine: merge the per-split partial results of the prefix sweep.
//
// The verification pass of [P1] Key Mechanisms > Batched Parallel Verification
// is one softmax over all keys a node sees.  The prefix is cut into splits so
// that enough CTAs share the work; each split s leaves a normalised partial
// O_s (bf16, the output's type) and its base-2 log-sum-exp L_s (fp32).  The exact softmax over the union is
//     out = sum_s 2^(L_s - M) O_s / sum_s 2^(L_s - M),  M = max_s L_s,
//     lse = ln 2 * (M + log2 sum_s 2^(L_s - M)).
// D/8 lanes per output row (b, node, head): each lane owns 8 consecutive
// channels, so every partial read and the output store is one 16-byte access
// per lane and a warp merges 32/(D/8) rows at once.  The splits are taken in
// groups of GRP (8, or 16 when a sequence may have more than 8 splits, so
// that up to 16 take one round trip): a group's lse and O loads are all in
// flight at once (the first group's are issued together with the
// prefix-length load, for every split the workspace holds, and the ones past
// this sequence's split count are dropped), and a running maximum rescales
// the sums between groups.  128-thread blocks; the 8-wide kernel (71
// registers) fits beside an attention CTA on one SM.
#include "internal.cuh"

namespace ts {

constexpr int COMBINE_THREADS = 128;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& x, float (&f)[8]) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
    f[2 * k] = t.x;
    f[2 * k + 1] = t.y;
  }
}

template <int D, int GRP>
__global__ void __launch_bounds__(COMBINE_THREADS)
k_combine(AttnArgs a) {
  constexpr int LPR = D / 8;                        // lanes per row
  constexpr int ROWS_PER_BLOCK = COMBINE_THREADS / LPR;
  const int rows = a.B * a.N * a.Hq;
  const int row = blockIdx.x * ROWS_PER_BLOCK + (int)threadIdx.x / LPR;
  const int sub = (int)threadIdx.x % LPR;          // channels 8*sub .. 8*sub+7
  pdl_wait();
  pdl_trigger();
  if (row >= rows) return;
  const int b = row / (a.N * a.Hq);
  const size_t stride_lse = (size_t)rows;
  const size_t stride_o = (size_t)rows * D;

  float w[GRP];
  uint4 raw[GRP];
  auto load_group = [&](int s0, int limit) {
#pragma unroll
    for (int i = 0; i < GRP; ++i) {
      const int s = s0 + i;
      w[i] = -INFINITY;
      raw[i] = make_uint4(0, 0, 0, 0);
      if (s < limit) {
        w[i] = a.part_lse[s * stride_lse + row];
        raw[i] = *reinterpret_cast<const uint4*>(a.part_o + s * stride_o + (size_t)row * D + sub * 8);
      }
    }
  };
  const int p_dev = a.prefix_len[b];
  load_group(0, a.max_splits);
  int P;
  usable_prefix(p_dev, a.chunk_tiles, a.max_splits, a.tree_split, a.bs, a.max_blocks, &P);
  const int ns = num_splits(P, a.chunk_tiles, a.tree_split);

  float m = -INFINITY, den = 0.f;
  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0.f;
  for (int s0 = 0; s0 < ns; s0 += GRP) {
    if (s0 > 0) load_group(s0, ns);
    float gm = -INFINITY;
#pragma unroll
    for (int i = 0; i < GRP; ++i)
      if (s0 + i < ns) gm = fmaxf(gm, w[i]);
    const float m_new = fmaxf(m, gm);
    const float f = (m == -INFINITY) ? 0.f : exp2f(m - m_new);
    den *= f;
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] *= f;
    m = m_new;
#pragma unroll
    for (int i = 0; i < GRP; ++i) {
      if (s0 + i < ns) {
        const float wi = exp2f(w[i] - m);
        den += wi;
        float v[8];
        bf16x8_to_f32(raw[i], v);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = fmaf(wi, v[k], acc[k]);
      }
    }
  }
  const float inv = 1.f / den;
  uint4 o;
  uint32_t* ow = &o.x;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __nv_bfloat162 t = __floats2bfloat162_rn(acc[2 * k] * inv, acc[2 * k + 1] * inv);
    ow[k] = *reinterpret_cast<const uint32_t*>(&t);
  }
  *reinterpret_cast<uint4*>(a.out + (size_t)row * D + sub * 8) = o;
  if (a.lse && sub == 0) a.lse[row] = (m + log2f(den)) * 0.69314718055994531f;
}

cudaError_t launch_combine(const AttnArgs& a, cudaStream_t s) {
  const int rows = a.B * a.N * a.Hq;
  const int per_block = COMBINE_THREADS / (a.D / 8);
  const int grid = ceil_div(rows, per_block);
  const bool wide = a.max_splits > 8;
  if (a.D == 128)
    return wide ? launch_pdl(k_combine<128, 16>, dim3(grid), dim3(COMBINE_THREADS), 0, s, a)
                : launch_pdl(k_combine<128, 8>, dim3(grid), dim3(COMBINE_THREADS), 0, s, a);
  return wide ? launch_pdl(k_combine<64, 16>, dim3(grid), dim3(COMBINE_THREADS), 0, s, a)
              : launch_pdl(k_combine<64, 8>, dim3(grid), dim3(COMBINE_THREADS), 0, s, a);
}

}  // namespace ts
