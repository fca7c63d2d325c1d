// Tree attention, CUDA-core formulation: the parity anchor for the tiled
// tensor-core kernel.  Same work split, same partial format, no tensor cores.
//
// [P1] Key Mechanisms > Batched Parallel Verification and Modified Causal
// Attention Mask; [P2] How It Works.  For unit (b, kv head g) the G query heads
// of all N nodes are packed as rows r = node * G + head_in_group.  Grid:
// (split, row tile of 128 rows, unit).  Split s walks prefix tiles
// [s*chunk, min((s+1)*chunk, tiles_b)); the last split of a unit also walks
// the tree keys, gated by the ancestry bitmask.  One thread owns one row and
// keeps its online-softmax state (running max, running sum, fp32 accumulator).
#include "internal.cuh"

namespace ts {

namespace {

constexpr int THREADS = ROW_TILE;  // one thread per packed row
constexpr float NEG_INF = -INFINITY;

template <int D>
struct Smem {
  float q[D][ROW_TILE];                  // q transposed: thread r reads q[d][r], conflict-free
  __nv_bfloat16 k[KV_TILE][D];
  __nv_bfloat16 v[KV_TILE][D];
  float s[KV_TILE][ROW_TILE];            // scores of the current tile
};

// Copy one key row of D bf16 (D*2 bytes) with 16-byte loads, or zero it.
template <int D>
__device__ __forceinline__ void copy_row(__nv_bfloat16* dst, const __nv_bfloat16* src, int lane8) {
  // lane8 in [0, D/8): one uint4 per call
  uint4 v = make_uint4(0, 0, 0, 0);
  if (src) v = *reinterpret_cast<const uint4*>(src + lane8 * 8);
  *reinterpret_cast<uint4*>(dst + lane8 * 8) = v;
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(THREADS)
k_attn_simt(AttnArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem<D>& sm = *reinterpret_cast<Smem<D>*>(smem_raw);

  const int split = blockIdx.x, rt = blockIdx.y, unit = blockIdx.z;
  const int b = unit / a.Hkv, g = unit - b * a.Hkv;
  int P;
  if (!usable_prefix(a.prefix_len[b], a.chunk_tiles, a.max_splits, a.bs, a.max_blocks, &P) && a.status &&
      threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
    a.status[b] = TS_ERR_SHAPE;
  const int tiles = prefix_tiles(P);
  const int ns = num_splits(P, a.chunk_tiles);
  if (split >= ns) return;
  const int t_begin = split * a.chunk_tiles;
  const int t_end = min(tiles, t_begin + a.chunk_tiles);
  const bool has_tree = (split == ns - 1);

  const int r = rt * ROW_TILE + threadIdx.x;
  const int R = a.N * a.G;
  const bool active = r < R;
  const int node = active ? r / a.G : 0;
  const int h = g * a.G + (active ? r - node * a.G : 0);

  // stage this thread's query row (fp32, transposed)
  {
    const __nv_bfloat16* qr = a.q + (((size_t)b * a.N + node) * a.Hq + h) * D;
    for (int d = 0; d < D; d += 2) {
      float2 f = make_float2(0.f, 0.f);
      if (active) f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(qr + d));
      sm.q[d][threadIdx.x] = f.x;
      sm.q[d + 1][threadIdx.x] = f.y;
    }
  }
  uint64_t mask[4] = {0, 0, 0, 0};
  if (active)
    for (int w = 0; w < a.W; ++w) mask[w] = a.anc_mask[((size_t)b * a.N + node) * a.W + w];

  float m = NEG_INF, l = 0.f;
  float acc[D];
#pragma unroll
  for (int d = 0; d < D; ++d) acc[d] = 0.f;

  const int tree_tiles = has_tree ? ceil_div(a.N, KV_TILE) : 0;
  const int n_iter = (t_end - t_begin) + tree_tiles;
  for (int it = 0; it < n_iter; ++it) {
    const bool is_tree = it >= (t_end - t_begin);
    const int tile = is_tree ? it - (t_end - t_begin) : t_begin + it;
    const int key0 = tile * KV_TILE;
    const int valid = is_tree ? min(KV_TILE, a.N - key0) : min(KV_TILE, P - key0);
    __syncthreads();  // previous tile fully consumed
    // cooperative load: KV_TILE rows x D/8 uint4 for K and V
    for (int e = threadIdx.x; e < KV_TILE * (D / 8); e += THREADS) {
      const int j = e / (D / 8), c = e - j * (D / 8);
      const __nv_bfloat16* ks = nullptr;
      const __nv_bfloat16* vs = nullptr;
      if (j < valid) {
        if (is_tree) {
          const size_t off = (((size_t)b * a.N + key0 + j) * a.Hkv + g) * D;
          ks = a.k_tree + off;
          vs = a.v_tree + off;
        } else {
          const int t = key0 + j;
          const int blk = a.block_table[(size_t)b * a.max_blocks + t / a.bs];
          if (blk >= 0 && blk < a.num_blocks) {
            const size_t off = (((size_t)blk * a.Hkv + g) * a.bs + (t % a.bs)) * D;
            ks = a.k_cache + off;
            vs = a.v_cache + off;
          } else if (a.status && c == 0) {
            a.status[b] = TS_ERR_BAD_BLOCK;
          }
        }
      }
      copy_row<D>(&sm.k[j][0], ks, c);
      copy_row<D>(&sm.v[j][0], vs, c);
    }
    __syncthreads();
    // scores for this tile
    float tmax = NEG_INF;
    for (int j = 0; j < KV_TILE; ++j) {
      bool vis = j < valid;
      if (is_tree && vis) {
        const int nj = key0 + j;
        vis = (mask[nj >> 6] >> (nj & 63)) & 1ull;
      }
      float sc = NEG_INF;
      if (vis) {
        float dot = 0.f;
#pragma unroll 8
        for (int d = 0; d < D; d += 2) {
          const float2 kf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.k[j][d]));
          dot = fmaf(sm.q[d][threadIdx.x], kf.x, dot);
          dot = fmaf(sm.q[d + 1][threadIdx.x], kf.y, dot);
        }
        sc = dot * a.scale_log2;
      }
      sm.s[j][threadIdx.x] = sc;
      tmax = fmaxf(tmax, sc);
    }
    const float m_new = fmaxf(m, tmax);
    if (m_new == NEG_INF) continue;  // nothing visible yet (cannot happen for real rows)
    const float corr = exp2f(m - m_new);
    l *= corr;
#pragma unroll
    for (int d = 0; d < D; ++d) acc[d] *= corr;
    for (int j = 0; j < KV_TILE; ++j) {
      const float p = exp2f(sm.s[j][threadIdx.x] - m_new);
      if (p == 0.f) continue;
      l += p;
#pragma unroll
      for (int d = 0; d < D; d += 2) {
        const float2 vf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&sm.v[j][d]));
        acc[d] = fmaf(p, vf.x, acc[d]);
        acc[d + 1] = fmaf(p, vf.y, acc[d + 1]);
      }
    }
    m = m_new;
  }
  if (!active) return;
  const size_t orow = ((size_t)b * a.N + node) * a.Hq + h;
  const size_t rows = (size_t)a.B * a.N * a.Hq;
  float* po = a.part_o + (size_t)split * rows * D + orow * D;
  const float inv = 1.f / l;
#pragma unroll
  for (int d = 0; d < D; d += 4)
    *reinterpret_cast<float4*>(po + d) = make_float4(acc[d] * inv, acc[d + 1] * inv, acc[d + 2] * inv, acc[d + 3] * inv);
  a.part_lse[(size_t)split * rows + orow] = m + log2f(l);
}

cudaError_t launch_attn(const AttnArgs& a, cudaStream_t s) {
  // the shared-memory opt-in is set once per process (not a stream operation,
  // so it is kept out of any later stream capture)
  static bool attr_set = false;
  if (!attr_set) {
    cudaFuncSetAttribute(k_attn_simt<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem<128>));
    cudaFuncSetAttribute(k_attn_simt<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem<64>));
    attr_set = true;
  }
  dim3 grid(a.max_splits, a.row_tiles, a.B * a.Hkv);
  if (a.D == 128)
    k_attn_simt<128><<<grid, THREADS, sizeof(Smem<128>), s>>>(a);
  else
    k_attn_simt<64><<<grid, THREADS, sizeof(Smem<64>), s>>>(a);
  return cudaGetLastError();
}

}  // namespace ts
