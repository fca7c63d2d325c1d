// Split combine: merge the per-split partial results of the prefix sweep.
//
// The verification pass of [P1] Key Mechanisms > Batched Parallel Verification
// is one softmax over all keys a node sees.  The prefix is cut into splits so
// that enough CTAs share the work; each split s leaves a normalised partial
// O_s (bf16, the output's type) and its base-2 log-sum-exp L_s (fp32).  The exact softmax over the union is
//     out = sum_s 2^(L_s - M) O_s / sum_s 2^(L_s - M),  M = max_s L_s,
//     lse = ln 2 * (M + log2 sum_s 2^(L_s - M)).
// D/CH lanes per output row (b, node, head): each lane owns CH consecutive
// channels (8, or 16 for plans of at most 4 splits), so every partial read
// and the output store is one or two 16-byte accesses per lane.  The splits are taken in
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

template <int D, int GRP, int CH>
__global__ void __launch_bounds__(COMBINE_THREADS)
k_combine(AttnArgs a) {
  constexpr int V = CH / 8;                         // 16-byte pieces a lane loads per split
  constexpr int LPR = D / CH;                       // lanes per row
  constexpr int ROWS_PER_BLOCK = COMBINE_THREADS / LPR;
  const int rows = a.B * a.N * a.Hq;
  const int row = blockIdx.x * ROWS_PER_BLOCK + (int)threadIdx.x / LPR;
  const int sub = (int)threadIdx.x % LPR;          // channels CH*sub .. CH*sub+CH-1
  pdl_wait();
  pdl_trigger();
  if (row >= rows) return;
  const int b = row / (a.N * a.Hq);
  const size_t stride_lse = (size_t)rows;
  const size_t stride_o = (size_t)rows * D;

  float w[GRP];
  uint4 raw[GRP][V];
  auto load_group = [&](int s0, int limit) {
#pragma unroll
    for (int i = 0; i < GRP; ++i) {
      const int s = s0 + i;
      w[i] = -INFINITY;
#pragma unroll
      for (int v = 0; v < V; ++v) raw[i][v] = make_uint4(0, 0, 0, 0);
      if (s < limit) {
        w[i] = a.part_lse[s * stride_lse + row];
#pragma unroll
        for (int v = 0; v < V; ++v)
          raw[i][v] = reinterpret_cast<const uint4*>(a.part_o + s * stride_o + (size_t)row * D + sub * CH)[v];
      }
    }
  };
  const int p_dev = a.prefix_len[b];
  load_group(0, a.max_splits);
  int P;
  usable_prefix(p_dev, a.chunk_tiles, a.max_splits, a.tree_split, a.bs, a.max_blocks, &P);
  const int ns = num_splits(P, a.chunk_tiles, a.tree_split);

  float m = -INFINITY, den = 0.f;
  float acc[CH];
#pragma unroll
  for (int k = 0; k < CH; ++k) acc[k] = 0.f;
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
    for (int k = 0; k < CH; ++k) acc[k] *= f;
    m = m_new;
#pragma unroll
    for (int i = 0; i < GRP; ++i) {
      if (s0 + i < ns) {
        const float wi = exp2f(w[i] - m);
        den += wi;
#pragma unroll
        for (int q = 0; q < V; ++q) {
          float v[8];
          bf16x8_to_f32(raw[i][q], v);
#pragma unroll
          for (int k = 0; k < 8; ++k) acc[8 * q + k] = fmaf(wi, v[k], acc[8 * q + k]);
        }
      }
    }
  }
  const float inv = 1.f / den;
#pragma unroll
  for (int q = 0; q < V; ++q) {
    uint4 o;
    uint32_t* ow = &o.x;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __nv_bfloat162 t = __floats2bfloat162_rn(acc[8 * q + 2 * k] * inv, acc[8 * q + 2 * k + 1] * inv);
      ow[k] = *reinterpret_cast<const uint32_t*>(&t);
    }
    reinterpret_cast<uint4*>(a.out + (size_t)row * D + sub * CH)[q] = o;
  }
  if (a.lse && sub == 0) a.lse[row] = (m + log2f(den)) * 0.69314718055994531f;
}

cudaError_t launch_combine(const AttnArgs& a, cudaStream_t s) {
  const int rows = a.B * a.N * a.Hq;
  // Up to 4 splits: 16 channels a lane and groups of 4, so that a grid of
  // twice as many rows a CTA is resident in one wave (the 8-channel kernel's
  // 71 registers leave room for 7 CTAs an SM: the 16 sequences of 1-16K
  // tokens took two waves).
  if (a.max_splits <= 4) {
    const int per_block = COMBINE_THREADS / (a.D / 16);
    const int grid = ceil_div(rows, per_block);
    return a.D == 128 ? launch_pdl(k_combine<128, 4, 16>, dim3(grid), dim3(COMBINE_THREADS), 0, s, a)
                      : launch_pdl(k_combine<64, 4, 16>, dim3(grid), dim3(COMBINE_THREADS), 0, s, a);
  }
  const int per_block = COMBINE_THREADS / (a.D / 8);
  const int grid = ceil_div(rows, per_block);
  const bool wide = a.max_splits > 8;
  if (a.D == 128)
    return wide ? launch_pdl(k_combine<128, 16, 8>, dim3(grid), dim3(COMBINE_THREADS), 0, s, a)
                : launch_pdl(k_combine<128, 8, 8>, dim3(grid), dim3(COMBINE_THREADS), 0, s, a);
  return wide ? launch_pdl(k_combine<64, 16, 8>, dim3(grid), dim3(COMBINE_THREADS), 0, s, a)
              : launch_pdl(k_combine<64, 8, 8>, dim3(grid), dim3(COMBINE_THREADS), 0, s, a);
}

}  // namespace ts
