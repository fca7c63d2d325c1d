// Tree attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes — [P1] Key Mechanisms > Batched Parallel Verification and
// Modified Causal Attention Mask; [P2] How It Works: every tree node's query
// attends to the whole verified prefix of its sequence and to the tree nodes
// on its own root path (its ancestors and itself), in one pass.
//
// How.  For a unit (sequence b, KV head g) the G query heads of all N nodes
// share every key, so they are packed as the M rows of the MMA:
// row r = node * G + head_in_group.  A work item is one tile of 128 rows and
// one split of the unit's prefix (a run of 128-token KV tiles); the last split
// also runs the tree block: the N tree keys, gated per row by the ancestry
// bitmask.  All of these share one online softmax.
//
// The kernel is persistent: one CTA per SM.  CTA c starts with item c; the
// others go to whichever CTA asks first (a counter in the workspace, taken
// by atomic add: items of unequal length, and empty splits past a short
// prefix, then balance out by themselves).  The K producer takes the items
// (skipping empty splits at once) and passes them to the other roles
// through a small queue in shared memory; the rings, the S buffers and the
// barrier phases continue from one item into the next, so the producers load
// the next item's first tiles and the QK issuer loads its Q tile while the
// softmax is still finishing the current one.  The counter is back at zero
// when the kernel ends: every CTA asks until it is told there is nothing
// left, and the last of all those requests resets it.  With one CTA per item
// instead, the set-up before the first tile (~3 us) and the epilogue
// (~2.5 us) were measured at 10 % of a 65-tile item and nearly 40 % of a
// 10-tile item.
//
//   warp 0     TMEM allocation; TMA loads of the K tiles
//   warp 3     TMA loads of the V tiles (paged blocks: one box per block); K
//              and V each stream through their own ring.  At CTA start it
//              also prefetches the tensor maps, the first Q tile and the first
//              block-table entry into L2, ahead of the launch wait.
//   warp 1     QK issuer (one thread): loads each item's Q tile once the
//              previous item's QKs have completed (q_empty), then
//              S(j) = Q K(j)^T, both operands in swizzled shared memory, into
//              S buffer j%3 once PV(j-3) (the last reader of that buffer) has
//              completed (s_free[j%3]).
//   warp 2     PV issuer (one thread): O += P(j) V(j), P read from TMEM, V
//              from shared memory, as soon as the softmax has written P(j).
//   warps 4-7  softmax: thread t owns TMEM lane t = row t.  Loads S from TMEM,
//              masks, tracks the running max/sum, writes P (bf16) back over S,
//              rescales O when the max moves by more than 2^20 (exact: the final
//              normalisation uses the same running max).  At the end of an
//              item each thread normalises its row of O to bf16 and stores it:
//              the output itself, or this split's partial.  After the CTA's
//              last item the K ring is idle, so the rows go there instead, in
//              the 128-byte-swizzled layout of a TMA box, and one thread
//              stores the boxes.
//   With QK and PV on two issuers the next tile's QK^T and this tile's PV
//   run while the softmax works.  Each control warp shares its sub-partition
//   with a softmax warp, and the scheduler keeps issuing from a ready compute
//   warp: beside a busy warp a control warp was measured to run several times
//   slower (8 TMA boxes in ~2500 cycles against ~420 alone), so the producer
//   loops are kept to a few instructions a tile.  Issuing the loads from the
//   softmax warps instead was measured slower still (each TMA issue blocks the
//   issuing warp until the SM's TMA unit, ~50 cycles a 4 KB box, takes it).
//
// Shared-memory K/V tiles of the prefix are laid out [8-row group][D half]
// [8 rows x 128 B] (each 1 KB piece one 128-byte-swizzle atom), so one TMA box
// brings every D column of a paged block; tree tiles are [D half][128 rows].
// TMEM (512 columns): O at [0, D), three S buffers at [128, 256), [256, 384)
// and [384, 512): QK can run two tiles ahead of the softmax, so the softmax
// does not wait for the PV that frees the buffer it needs next.  The tree
// block rides on the last prefix split of a unit or, when the host plans it
// so, on a split of its own that runs beside the prefix splits.
// Every mbarrier wait is bounded; a timeout sets a shared abort flag and every
// role winds down.  Before the CTA frees its TMEM and exits, an aborted CTA
// drains what it still has in flight: the producers wait (bounded) for the
// loads they issued to land, and each MMA issuer commits to a barrier of its
// own and waits for its MMAs to finish.  It then reports TS_ERR_TIMEOUT for
// the sequence of every item it had not finished.
#include "fastexp.cuh"
#include "internal.cuh"
#include "sm100.cuh"
#include "tensor_map.cuh"

namespace ts {
namespace {

using namespace sm100;

constexpr int NUM_THREADS = 256;
constexpr int SOFTMAX_THREADS = 128;
// Warp roles.  On each SM sub-partition one control warp shares the issue
// slots with one softmax warp (warp w runs on sub-partition w % 4).
constexpr int PRODUCER_WARP = 0;
constexpr int QK_WARP = 1;
constexpr int PV_WARP = 2;
constexpr int V_PRODUCER_WARP = 3;
constexpr int SOFTMAX_WARP0 = 4;  // warps 4-7; warp w reads TMEM lanes 32 * (w % 4) ..
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_O = 0;
constexpr uint32_t TMEM_S0 = 128;
constexpr int NSB = 3;  // S buffers in TMEM
constexpr int ITEM_Q = 16;  // entries of the item queue (a role can lag the K producer by at most ~7 items)
// O is rescaled only when a row's max rises by more than 2^20 (log2 units).
// Until then p = 2^(s - m_run) <= 2^20: bf16 P (range to 3e38) and the fp32 O
// and l accumulators (relative precision independent of scale) stay exact up
// to rounding, and the final normalisation uses the same running max.  Fewer
// rescales matter where hot keys move the max often (each rescale waits for
// the previous PV).
constexpr float RESCALE_THRESHOLD = 20.0f;
constexpr float NEG_INF = -INFINITY;

template <int D>
struct Cfg {
  static constexpr int HALVES = D / 64;                        // 128-byte swizzle atoms along D
  static constexpr int TILE_BYTES = KV_TILE * D * 2;           // one K or V tile
  static constexpr int HALF_BYTES = KV_TILE * 128;             // one 64-column half of a tile
  static constexpr int Q_BYTES = ROW_TILE * D * 2;
  // Ring depths (K and V), as many tiles as fit beside the Q tile.  Moving a
  // V slot to K (4 + 2 for D = 128) was measured slower: PV then waited for V.
  static constexpr int NSTK = (D == 128) ? 3 : 6;
  static constexpr int NSTV = (D == 128) ? 3 : 6;
};

template <int D>
struct __align__(1024) Smem {
  using C = Cfg<D>;
  uint8_t q[C::Q_BYTES];
  uint8_t k[C::NSTK][C::TILE_BYTES];
  uint8_t v[C::NSTV][C::TILE_BYTES];
  uint64_t q_full;
  uint64_t q_empty;  // the Q tile is no longer read: every QK of its item completed
  uint64_t k_full[C::NSTK];
  uint64_t v_full[C::NSTV];
  uint64_t k_empty[C::NSTK];  // K slot free: its QK completed
  uint64_t v_empty[C::NSTV];  // V slot free: its PV completed
  uint64_t s_full[NSB];
  uint64_t p_full[NSB];
  uint64_t s_free[NSB];  // S buffer b no longer read: PV of its last tile completed
  uint64_t o_ready;
  uint64_t drain[2];  // an aborted CTA's QK and PV issuers wait here for their MMAs
  uint32_t tmem_base;
  int abort_flag;
  int pv_done;  // PVs completed so far, published by the PV issuer (release/acquire)
  // The CTA's items, in the order it takes them: entry k (k % ITEM_Q) holds
  // (item, prefix length) of its k-th item, or item -1 after the last.
  // Written by the K producer, which takes the items; items_pub entries are
  // published, items_done items finished (stored) by the softmax.
  int2 item_q[ITEM_Q];
  int items_pub;
  int items_done;
};

struct TcArgs {
  AttnArgs a;
  int box_rows;   // rows per paged TMA box: gcd(block_size, 128), so a box never crosses a block
  int direct;     // 1: a single split per unit -> write bf16 out (+ lse) directly
  int n_items;    // row_tiles * max_splits * B * Hkv work items
  int nodes_per_tile;  // ROW_TILE / G
  int out32;           // the output (or the partials) start on a 32-byte boundary
  // the launch's divisors, for divisions on the device's critical paths
  FastDiv fd_rt, fd_ms, fd_hkv, fd_chunk, fd_bs, fd_g;
  int n_order;  // 0, or B * max_splits entries in order[]
  uint32_t order[ATTN_ORDER_MAX];  // (sequence, split, first tile), packed as ORDER_* says, in taking order
};

// A work item: row tile rt of unit (b, g), split `split`.  The row tiles of
// a unit are numbered side by side, so that CTAs taking items one after the
// other read the same K/V tiles at about the same time (from L2).  With an
// order table, items go (sequence, split) pair by pair in the table's order
// (longest first), the KV heads of a pair next to each other; without one,
// unit-major, then split.  Numbered split-major instead, the last splits of
// the longest prefixes were taken last and ran on alone (103 against 93 us
// on 16 paged prefixes of 1-16K tokens).
// start_hint: the split's first prefix tile by the host's prefix length
// (the device's may differ; its block-table entries are loaded before the
// device's is known, and checked against it when used).
struct ItemPos {
  int rt, split, b, g, start_hint;
};
__device__ __forceinline__ ItemPos item_pos(int it, const TcArgs& t) {
  ItemPos p;
  const int rs = t.fd_rt.div(it);
  p.rt = it - rs * t.a.row_tiles;
  if (t.n_order) {
    const int e = t.fd_hkv.div(rs);
    p.g = rs - e * t.a.Hkv;
    const uint32_t v = t.order[e];
    p.b = (int)(v >> ORDER_B_SHIFT);
    p.split = (int)((v >> ORDER_SPLIT_SHIFT) & ORDER_SPLIT_MASK);
    const int h = (int)(v & ORDER_START_MASK);
    p.start_hint = h == ORDER_START_MASK ? p.split * t.a.chunk_tiles : h;
  } else {
    const int unit = t.fd_ms.div(rs);
    p.split = rs - unit * t.a.max_splits;
    p.b = t.fd_hkv.div(unit);
    p.g = unit - p.b * t.a.Hkv;
    p.start_hint = p.split * t.a.chunk_tiles;
  }
  return p;
}

// Its extent, once the sequence's prefix length is known.
struct Item {
  ItemPos pos;
  int P;         // usable prefix length
  int t_begin;   // first prefix tile of the split
  int n_prefix;  // prefix tiles of this split
  int n_tiles;   // + tree tiles on the sequence's last split
  bool work;     // false: the split lies past this sequence's prefix
  bool p_ok;     // false: the device prefix length had to be clamped
};
__device__ __forceinline__ Item make_item(int it, int p_dev, const TcArgs& t) {
  const AttnArgs& a = t.a;
  Item I;
  I.pos = item_pos(it, t);
  I.p_ok = usable_prefix(p_dev, a.chunk_tiles, a.max_splits, a.tree_split, a.bs, a.max_blocks, &I.P);
  const int tiles = prefix_tiles(I.P);
  // num_splits(I.P, chunk_tiles, tree_split), without its division
  const int ps = t.fd_chunk.div(tiles + a.chunk_tiles - 1);
  const int ns = a.tree_split ? ps + 1 : (ps == 0 ? 1 : ps);
  const int s = I.pos.split;
  I.work = s < ns;
  I.t_begin = s < ps ? split_start(tiles, ps, s) : tiles;
  I.n_prefix = s < ps ? split_start(tiles, ps, s + 1) - I.t_begin : 0;
  I.n_tiles = I.n_prefix + ((s == ns - 1) ? ceil_div(a.N, KV_TILE) : 0);
  return I;
}

// Abort state of a CTA: its flag and the wait limit.
struct Ctl {
  volatile int* flag;
  uint64_t limit;
};

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Ctl& c) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*c.flag) return false;
    if (globaltimer_ns() - t0 > c.limit) {
      *c.flag = 1;
      return false;
    }
  }
}

// Bounded wait until the published PV count reaches `target`.
__device__ __forceinline__ bool wait_count(const int* counter, int target, const Ctl& c) {
  const uint32_t addr = smem_u32(counter);
  auto load = [&]() {
    int v;
    asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
  };
  if (load() >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (load() >= target) return true;
    if (*c.flag) return false;
    if (globaltimer_ns() - t0 > c.limit) {
      *c.flag = 1;
      return false;
    }
  }
}

// A plain global load the compiler may not move: issued where it is written.
__device__ __forceinline__ int ld_global_early(const int* p) {
  int v;
  asm volatile("ld.global.b32 %0, [%1];" : "=r"(v) : "l"(reinterpret_cast<uint64_t>(p)) : "memory");
  return v;
}

// One 32-byte store of 8 words (a whole DRAM sector), to a 32-byte aligned address.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(reinterpret_cast<uint64_t>(p)),
               "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
k_attn_tc(const __grid_constant__ TcArgs args, const __grid_constant__ CUtensorMap tm_q,
          const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_vc,
          const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_vt,
          const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_po) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  Smem<D>& sm = *reinterpret_cast<Smem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const AttnArgs& a = args.a;
  volatile int* abort_flag = &sm.abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Ctl ctl{abort_flag, a.wait_limit_ns};
  const int n_items = args.n_items;
  const int stride = gridDim.x;
  const int first = blockIdx.x;  // < n_items: the grid has at most one CTA per item
  // Geometry of this warp's paged loads (producer warps): rows per box,
  // boxes per tile, tiles per group of 32 block-table entries.
  const int g_box = args.box_rows;
  const int g_boxes = KV_TILE / g_box;  // 1 .. 8
  const int g_tpg = 32 / g_boxes;
  // First of all, by a warp that has no part in the set-up: fetch the tensor
  // maps (kernel parameters) and prefetch into L2 the first item's Q tile and
  // the block-table entry of its first tile, so that their address
  // translation and DRAM latency overlap the set-up and the wait (prefetches
  // read no data; see sm100.cuh).
  const ItemPos pos0 = item_pos(first, args);
  if (warp == V_PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kc);
    tma_prefetch_desc(&tm_vc);
    tma_prefetch_desc(&tm_kt);
    tma_prefetch_desc(&tm_vt);
    for (int hh = 0; hh < C::HALVES; ++hh) tma_prefetch_4d(&tm_q, 64 * hh, pos0.g * a.G, pos0.rt * args.nodes_per_tile, pos0.b);
    if (a.max_blocks > 0) {
      // the 16-byte piece holding the entry, through the bulk-copy unit
      const int idx = args.fd_bs.div(pos0.start_hint * KV_TILE);
      const int* row0 = a.block_table + (size_t)pos0.b * a.max_blocks;
      const uintptr_t e = reinterpret_cast<uintptr_t>(row0 + (idx < a.max_blocks ? idx : a.max_blocks - 1));
      bulk_prefetch_l2(reinterpret_cast<const void*>(e & ~uintptr_t(15)), 16);
    }
  }
  // the first item's first block-table entries, one per lane of a producer
  // warp (index clamped to the table's row; entries past the prefix are
  // discarded when used)
  const bool producer = (warp == PRODUCER_WARP || warp == V_PRODUCER_WARP) && a.max_blocks > 0;
  const int* blk_first_addr = a.block_table;
  if (producer) {
    const int t0 = (pos0.start_hint + lane / g_boxes) * KV_TILE + (lane % g_boxes) * g_box;
    const int idx = args.fd_bs.div(t0);
    blk_first_addr = a.block_table + (size_t)pos0.b * a.max_blocks + (idx < a.max_blocks ? idx : a.max_blocks - 1);
  }

  if (threadIdx.x == 0) {
    sm.abort_flag = 0;
    sm.pv_done = 0;
    sm.items_pub = 0;
    sm.items_done = 0;
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    for (int i = 0; i < C::NSTK; ++i) {
      mbar_init(&sm.k_full[i], 1);
      mbar_init(&sm.k_empty[i], 1);
    }
    for (int i = 0; i < C::NSTV; ++i) {
      mbar_init(&sm.v_full[i], 1);
      mbar_init(&sm.v_empty[i], 1);
    }
    for (int i = 0; i < NSB; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.p_full[i], SOFTMAX_THREADS);
      mbar_init(&sm.s_free[i], 1);
    }
    mbar_init(&sm.o_ready, 1);
    mbar_init(&sm.drain[0], 1);
    mbar_init(&sm.drain[1], 1);
    fence_barrier_init();
  }
  if (warp == PRODUCER_WARP) tmem_alloc(&sm.tmem_base, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  // everything above read no global memory (prefetches return no data) and
  // overlaps the previous kernel's tail; wait for it before reading any
  // input.  The next kernel is
  // released only at this CTA's teardown (released at the start, its CTAs
  // were measured to delay this kernel's first loads by about 2 us).
  pdl_wait();
  // The producers fetch the first item's prefix length and first
  // block-table entries together (volatile loads, issued where written), so
  // the two latencies overlap.
  //
  // With one CTA per item (the grid as large as the item count) nothing is
  // taken from the counter and nothing goes through the queue: every role
  // reads the prefix length itself and works on item blockIdx.x alone (the
  // queue's hand-over was measured to add ~1 us to such a CTA's start).
  const bool single = (int)gridDim.x == n_items;
  const bool grabber = warp == PRODUCER_WARP && !single;
  const int p_first = (grabber || single) ? ld_global_early(a.prefix_len + pos0.b) : 0;
  const int blk_first = producer ? ld_global_early(blk_first_addr) : 0;
  const bool single_work = single && make_item(first, p_first, args).work;

  // Entry k of the item queue (every role but the K producer; with one CTA
  // per item, every role): false if the wait gave up.
  auto queue_entry = [&](int k, int2& e) -> bool {
    if (single) {
      e = (k == 0 && single_work) ? make_int2(first, p_first) : make_int2(-1, 0);
      return true;
    }
    if (!wait_count(&sm.items_pub, k + 1, ctl)) return false;
    const volatile int* q = reinterpret_cast<volatile int*>(&sm.item_q[k % ITEM_Q]);
    e.x = q[0];
    e.y = q[1];
    return true;
  };
  // Taking an item (lane 0 of the K producer): -1 once none is left.  The
  // request that comes last of all (every CTA makes exactly one that finds
  // nothing) puts the counter back to zero for the next call.
  auto take_item = [&]() -> int {
    const unsigned v = atomicAdd(a.sched, 1u);
    if (v == (unsigned)(n_items - 1)) atomicExch(a.sched, 0u);
    return stride + (int)v < n_items ? stride + (int)v : -1;
  };
  // K producer state the teardown of an aborted CTA needs: the item it took
  // but has not published yet (-1: none), and whether the counter said
  // nothing was left.
  int held = -1;
  bool exhausted = single;  // nothing to take from the counter

  // ------------------------------------------------------------ K or V producer
  // One warp streams the K tiles, another the V tiles: a single warp issues a
  // TMA request only every ~120 cycles, so one warp alone could not keep up
  // with 16 paged boxes per tile.  Each ring slot is refilled as soon as its
  // own consumer (QK for K, PV for V) has released it, whichever item the
  // tile belongs to.  Returns how many tiles it issued (all of them unless a
  // wait gave up or a stall was asked for).
  auto kv_producer = [&](bool is_v) -> int {
    const CUtensorMap* tm_pool = is_v ? &tm_vc : &tm_kc;
    const CUtensorMap* tm_node = is_v ? &tm_vt : &tm_kt;
    uint64_t* full = is_v ? sm.v_full : sm.k_full;
    uint64_t* empty = is_v ? sm.v_empty : sm.k_empty;
    const int nst = is_v ? C::NSTV : C::NSTK;
    const uint32_t box_bytes = g_box * D * 2;
    // This warp's loop is on the tile period's critical path and shares its
    // sub-partition with a softmax warp: it was measured to take ~900 cycles
    // a tile for ~150 dependent integer instructions (runtime divisions, a
    // 32-lane wait and vote).  So every per-tile quantity is kept
    // incrementally (boxes per tile and tiles per table group are powers of
    // two), only lane 0 waits, and a block id is checked when it is used,
    // not when it is loaded.
    const int lg_boxes = __ffs(g_boxes) - 1;
    const int koff = (lane & (g_boxes - 1)) * g_box;  // this lane's box: keys [koff, +box) of a tile
    int slot = 0, phase = 0;  // ring slot and its phase
    int jg = 0;               // tiles issued, over every item
    // K producer: the item in hand and its prefix length
    int cand = first, cand_p = p_first;
    if (grabber) held = first;
    for (int k = 0;; ++k) {
      int it, p_dev;
      if (grabber) {
        // skip empty splits (a short prefix), taking the next item each time
        for (;;) {
          if (cand < 0 || make_item(cand, cand_p, args).work) break;
          int nx = -1;
          if (lane == 0) nx = take_item();
          cand = __shfl_sync(0xffffffffu, nx, 0);
          held = cand;
          exhausted = cand < 0;
          cand_p = cand >= 0 ? ld_global_early(a.prefix_len + item_pos(cand, args).b) : 0;
        }
        // entry k reuses entry k - ITEM_Q's slot: that item must be finished
        bool ok = k < ITEM_Q;
        if (!ok && lane == 0) ok = wait_count(&sm.items_done, k - ITEM_Q + 1, ctl);
        if (!__shfl_sync(0xffffffffu, ok, 0)) return jg;
        if (lane == 0) {
          sm.item_q[k % ITEM_Q] = make_int2(cand, cand_p);
          asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sm.items_pub)), "r"(k + 1) : "memory");
        }
        held = -1;
        if (cand < 0) return jg;
        it = cand;
        p_dev = cand_p;
        // take the next item now: its prefix length loads while this one streams
        int nx = -1;
        if (lane == 0) nx = take_item();
        cand = __shfl_sync(0xffffffffu, nx, 0);
        held = cand;
        exhausted = cand < 0;
        cand_p = cand >= 0 ? ld_global_early(a.prefix_len + item_pos(cand, args).b) : 0;
      } else {
        int2 e;
        bool ok = true;
        if (lane == 0) ok = queue_entry(k, e);
        if (!__shfl_sync(0xffffffffu, ok, 0)) return jg;
        it = __shfl_sync(0xffffffffu, e.x, 0);
        p_dev = __shfl_sync(0xffffffffu, e.y, 0);
        if (it < 0) return jg;
      }
      const Item I = make_item(it, p_dev, args);
      const int b = I.pos.b, g = I.pos.g, t_begin = I.t_begin, n_prefix = I.n_prefix, P = I.P;
      const int* table_row = a.block_table + (size_t)b * a.max_blocks;
      // Block-table entries are software-pipelined: lane L holds the entry of
      // box (L % boxes) of tile (L / boxes) of a group of 32/boxes tiles; the
      // next group is loaded (one coalesced read) when the current one starts,
      // so the table's load latency hides behind several tiles of TMA issue.
      // (the entries loaded at the start were for the host's prefix length;
      // if the device's moves the split's start, they are loaded again here)
      const bool use_first = it == first && t_begin == I.pos.start_hint;
      auto load_group = [&](int grp) -> int {
        const int tile = grp * g_tpg + (lane >> lg_boxes);
        const int t0 = (t_begin + tile) * KV_TILE + koff;
        if (tile >= n_prefix || t0 >= P) return 0;
        return (grp == 0 && use_first) ? blk_first : table_row[args.fd_bs.div(t0)];
      };
      int grp_cur = load_group(0);
      int grp_nxt = (n_prefix > g_tpg) ? load_group(1) : 0;
      const int stop = (!is_v && b == a.stall_seq) ? a.stall_tile : I.n_tiles;
      // key of this lane's box in the current tile, and its row in its block
      // (advanced by a tile, 128 mod block_size rows, each step; constant when
      // blocks divide a tile)
      int key = t_begin * KV_TILE + koff;
      int row = args.fd_bs.mod(key);
      const int row_step = args.fd_bs.mod(KV_TILE);
      int jt = 0;  // tile within the table group
      for (int j = 0; j < I.n_tiles; ++j, ++jg) {
        uint8_t* dst = is_v ? sm.v[slot] : sm.k[slot];
        if (jg >= nst) {
          bool ok = true;
          if (lane == 0) ok = wait_bar(&empty[slot], phase ^ 1, ctl);
          if (!__shfl_sync(0xffffffffu, ok, 0)) return jg;
        }
        if (j == stop) return jg;
        if (j < n_prefix) {
          if (jt == 0 && j > 0) {
            grp_cur = grp_nxt;
            const int g2 = (j >> (5 - lg_boxes)) + 1;
            grp_nxt = (g2 * g_tpg < n_prefix) ? load_group(g2) : 0;
          }
          // lane i < boxes handles the box of tokens [key, key + box_rows)
          int blk = __shfl_sync(0xffffffffu, grp_cur, (jt << lg_boxes) + lane);
          const bool issue = lane < g_boxes && key < P;
          if (issue && (blk < 0 || blk >= a.num_blocks)) {
            if (a.status) a.status[b] = TS_ERR_BAD_BLOCK;
            blk = 0;  // read a valid block instead; the sequence is reported as failed
          }
          const unsigned mask = __ballot_sync(0xffffffffu, issue);
          if (lane == 0) mbar_arrive_expect_tx(&full[slot], __popc(mask) * box_bytes);
          __syncwarp();
          // one box = every D column of box_rows tokens of one paged block
          if (issue) tma_load_5d(dst + lane * box_bytes, tm_pool, &full[slot], 0, 0, 0, row >> 3, blk * a.Hkv + g);
          key += KV_TILE;
          row += row_step;
          if (row >= a.bs) row -= a.bs;
          jt = (jt + 1) & (g_tpg - 1);
        } else if (lane == 0) {
          const int n0 = (j - n_prefix) * KV_TILE;  // first tree node of this tile; nodes >= N read as zeros
          mbar_arrive_expect_tx(&full[slot], C::TILE_BYTES);
          for (int h = 0; h < C::HALVES; ++h) tma_load_4d(dst + h * C::HALF_BYTES, tm_node, &full[slot], 64 * h, g, n0, b);
        }
        __syncwarp();
        if (++slot == nst) {
          slot = 0;
          phase ^= 1;
        }
      }
    }
  };
  int issued = 0;                  // tiles this warp's producer issued (K or V), for the drain of an aborted CTA
  int q_issued = 0, q_landed = 0;  // Q loads the QK issuer started / saw land, for the same drain

  if (warp == PRODUCER_WARP || warp == V_PRODUCER_WARP) {
    issued = kv_producer(warp == V_PRODUCER_WARP);  // one call site: one copy of the loop
  } else if (warp == QK_WARP) {
    if (lane == 0) {
      // ---------------------------------------------------------- QK issuer
      constexpr uint32_t ID_QK = idesc_bf16_f32(ROW_TILE, KV_TILE, 0, 0);
      const uint32_t q_addr = smem_u32(sm.q);
      const int nodes_per_tile = args.nodes_per_tile;
      int jg = 0;  // tiles, over every item
      bool ok = true;
      auto load_q = [&](const ItemPos& q) {
        mbar_arrive_expect_tx(&sm.q_full, C::Q_BYTES);
        for (int h = 0; h < C::HALVES; ++h)
          tma_load_4d(sm.q + h * (ROW_TILE * 128), &tm_q, &sm.q_full, 64 * h, q.g * a.G, q.rt * nodes_per_tile, q.b);
        ++q_issued;
      };
      // The CTA's first item is `first` unless that split is empty: its Q
      // tile needs no prefix length, so it is loaded at once (with one CTA
      // per item, only if the split has work).
      if (!single || single_work) load_q(pos0);
      for (int k = 0; ok; ++k) {
        int2 e;
        if (!(ok = queue_entry(k, e))) break;
        if (e.x < 0) break;
        const Item I = make_item(e.x, e.y, args);
        if (k > 0 || e.x != first) {
          if (k == 0) {
            // the tile loaded at once is not needed: let it land, free the buffer
            if (!(ok = wait_bar(&sm.q_full, 0, ctl))) break;
            ++q_landed;
            mma_commit(&sm.q_empty);
          }
          // this item's Q tile, once every QK of the previous one has completed
          if (!(ok = wait_bar(&sm.q_empty, (q_issued - 1) & 1, ctl))) break;
          load_q(I.pos);
        }
        if (!(ok = wait_bar(&sm.q_full, (q_issued - 1) & 1, ctl))) break;
        ++q_landed;
        bool next_q_seen = false;
        for (int j = 0; j < I.n_tiles; ++j, ++jg) {
          const int slot = jg % C::NSTK;
          if (!next_q_seen) {
            // once the next item is known (the K producer names it after its
            // last K tile of this one), its Q tile goes into L2
            int pub;
            asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(pub) : "r"(smem_u32(&sm.items_pub)) : "memory");
            if (pub > k + 1) {
              next_q_seen = true;
              const int nx = sm.item_q[(k + 1) % ITEM_Q].x;
              if (nx >= 0) {
                const ItemPos pn = item_pos(nx, args);
                for (int h = 0; h < C::HALVES; ++h)
                  tma_prefetch_4d(&tm_q, 64 * h, pn.g * a.G, pn.rt * nodes_per_tile, pn.b);
              }
            }
          }
          // K(j) has landed; S buffer jg%3 is free once the PV three tiles
          // back has completed (a per-buffer barrier: it can never run two
          // completions ahead)
          ok = wait_bar(&sm.k_full[slot], (jg / C::NSTK) & 1, ctl) &&
               (jg < NSB || wait_bar(&sm.s_free[jg % NSB], ((jg / NSB) - 1) & 1, ctl));
          if (!ok) break;
          tc_fence_after();
          const uint32_t k_addr = smem_u32(sm.k[slot]);
          const uint32_t d_tmem = tmem + TMEM_S0 + (jg % NSB) * 128;
          // prefix tiles: D halves 1 KB apart, 8-row groups HALVES KB apart;
          // tree tiles: D halves 16 KB apart, 8-row groups 1 KB apart
          const bool tree = j >= I.n_prefix;
          const uint32_t k_half = tree ? C::HALF_BYTES : 1024;
          const uint32_t k_sbo = tree ? 1024 : C::HALVES * 1024;
#pragma unroll
          for (int k2 = 0; k2 < D / 16; ++k2) {
            const uint32_t off = (k2 >> 2) * (ROW_TILE * 128) + (k2 & 3) * 32;
            const uint32_t koff = (k2 >> 2) * k_half + (k2 & 3) * 32;
            mma_ss(d_tmem, smem_desc_sw128(q_addr + off, 16, 1024), smem_desc_sw128(k_addr + koff, 16, k_sbo), ID_QK,
                   k2 > 0);
          }
          mma_commit(&sm.s_full[jg % NSB]);
          mma_commit(&sm.k_empty[slot]);  // K(j) no longer read
        }
        if (ok) mma_commit(&sm.q_empty);  // Q no longer read once these QKs complete
      }
      // A Q tile loaded for nothing (the first split was empty and no other
      // item came) must land before the CTA may exit.
      if (ok && q_issued > q_landed && wait_bar(&sm.q_full, (q_issued - 1) & 1, ctl)) ++q_landed;
    }
  } else if (warp == PV_WARP) {
    if (lane == 0) {
      // ---------------------------------------------------------- PV issuer
      constexpr uint32_t ID_PV = idesc_bf16_f32(ROW_TILE, D, 0, 1);
      int jg = 0;  // tiles, over every item
      bool ok = true;
      for (int k = 0; ok; ++k) {
        int2 e;
        if (!(ok = queue_entry(k, e))) break;
        if (e.x < 0) break;
        const Item I = make_item(e.x, e.y, args);
        for (int j = 0; j < I.n_tiles; ++j, ++jg) {
          const int slot = jg % C::NSTV;
          if (!(ok = wait_bar(&sm.p_full[jg % NSB], (jg / NSB) & 1, ctl))) break;
          if (!(ok = wait_bar(&sm.v_full[slot], (jg / C::NSTV) & 1, ctl))) break;
          tc_fence_after();
          const uint32_t v_addr = smem_u32(sm.v[slot]);
          const uint32_t p_tmem = tmem + TMEM_S0 + (jg % NSB) * 128;
          const bool tree = j >= I.n_prefix;
          const uint32_t v_lbo = tree ? C::HALF_BYTES : 1024;    // between D halves
          const uint32_t v_sbo = tree ? 1024 : C::HALVES * 1024;  // between 8-key groups
#pragma unroll
          for (int k2 = 0; k2 < KV_TILE / 16; ++k2)
            mma_ts(tmem + TMEM_O, p_tmem + k2 * 8, smem_desc_sw128(v_addr + k2 * 2 * v_sbo, v_lbo, v_sbo), ID_PV,
                   j > 0 || k2 > 0);
          mma_commit(&sm.o_ready);
          mma_commit(&sm.s_free[jg % NSB]);
          mma_commit(&sm.v_empty[slot]);  // V(j) no longer read
          // wait for this PV here (every phase in order) and publish the
          // count, so the softmax looks at O only when it has to rescale it
          // or, at the end of an item, read it
          if (!(ok = wait_bar(&sm.o_ready, jg & 1, ctl))) break;
          tc_fence_after();
          asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sm.pv_done)), "r"(jg + 1) : "memory");
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x - SOFTMAX_WARP0 * 32;  // TMEM lane == packed row within the tile
    const int R = a.N * a.G;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const size_t rows_all = (size_t)a.B * a.N * a.Hq;
    int jg = 0;  // tiles, over every item
    bool ok = true;
    // the CTA's last item ends in the idle K ring, stored by TMA boxes after
    // the loop (every softmax thread reaches that barrier, whatever happens)
    bool staged = false;
    ItemPos last_pos{0, 0, 0, 0};
    uint8_t* stage = &sm.k[0][0];
    int2 e;
    ok = queue_entry(0, e);
    for (int k = 0; ok && e.x >= 0; ++k) {
      const Item I = make_item(e.x, e.y, args);
      const int b = I.pos.b, g = I.pos.g, rt = I.pos.rt, split = I.pos.split;
      const int t_begin = I.t_begin, n_prefix = I.n_prefix, P = I.P;
      if (!I.p_ok && r == 0 && rt == 0 && split == 0 && a.status) a.status[b] = TS_ERR_SHAPE;
      const int grow = rt * ROW_TILE + r;
      const bool active = grow < R;
      const int node = active ? args.fd_g.div(grow) : 0;
      const int h = g * a.G + (active ? grow - node * a.G : 0);
      // ancestry words of this row; words past W stay zero.  Padding rows (past
      // N*G) see every key so that their softmax stays finite; never written out.
      // Unrolled with fixed indices, so the words stay in registers and the
      // loads are waited for only at the tree tile: a loop over a.W put them in
      // local memory, and with it the end of one item to the first tile of the
      // next took 0.70 us on the 64-sequence, 8K-prefix layer (0.45 now).
      uint64_t anc[4] = {0ull, 0ull, 0ull, 0ull};
      if (active) {
        const uint64_t* arow = a.anc_mask + ((size_t)b * a.N + node) * a.W;
#pragma unroll
        for (int w = 0; w < 4; ++w)
          if (w < a.W) anc[w] = arow[w];
      } else {
        anc[0] = anc[1] = anc[2] = anc[3] = ~0ull;
      }
      float m_run = NEG_INF, l_run = 0.f;
      for (int j = 0; j < I.n_tiles; ++j, ++jg) {
        if (!__all_sync(0xffffffffu, wait_bar(&sm.s_full[jg % NSB], (jg / NSB) & 1, ctl))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t s_tmem = tmem + lane_base + TMEM_S0 + (jg % NSB) * 128;
        float s[KV_TILE];
        {
          // all four TMEM loads in flight before one wait
          uint32_t u[KV_TILE / 32][32];
#pragma unroll
          for (int c = 0; c < KV_TILE / 32; ++c) tmem_ld32(s_tmem + c * 32, u[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < KV_TILE / 32; ++c) {
            reg_fence32(u[c]);
#pragma unroll
            for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(u[c][e]);
          }
        }
        // masking: ragged prefix tail, or the tree block's ancestry bits
        bool tail_zero_v = false;
        int valid = KV_TILE;
        if (j < n_prefix) {
          const int key0 = (t_begin + j) * KV_TILE;
          valid = min(KV_TILE, P - key0);
          if (valid < KV_TILE) {
            tail_zero_v = true;
#pragma unroll
            for (int c = 0; c < KV_TILE; ++c)
              if (c >= valid) s[c] = NEG_INF;
          }
        } else {
          const int tt = j - n_prefix;  // tree tile: nodes [128*tt, 128*tt + 128)
          const uint64_t lo = tt == 0 ? anc[0] : (tt == 1 ? anc[2] : 0ull);
          const uint64_t hi = tt == 0 ? anc[1] : (tt == 1 ? anc[3] : 0ull);
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (!((lo >> c) & 1ull)) s[c] = NEG_INF;
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (!((hi >> c) & 1ull)) s[64 + c] = NEG_INF;
        }
        // row max with 8 independent chains, then a 3-level tree
        float mk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mk[e] = s[e];
#pragma unroll
        for (int c = 8; c < KV_TILE; c += 8)
#pragma unroll
          for (int e = 0; e < 8; ++e) mk[e] = fmaxf(mk[e], s[c + e]);
        float mx = fmaxf(fmaxf(fmaxf(mk[0], mk[1]), fmaxf(mk[2], mk[3])), fmaxf(fmaxf(mk[4], mk[5]), fmaxf(mk[6], mk[7])));
        mx *= a.scale_log2;
        const float m_new = fmaxf(m_run, mx);
        const bool rescale = (j > 0) && (m_new > m_run + RESCALE_THRESHOLD);
        float m_use = m_run;
        if (j == 0 || rescale) m_use = m_new;
        // nothing visible so far: every p is 0 (and O is rescaled away later)
        const float m_exp = (m_use == NEG_INF) ? 0.f : m_use;
        // p = 2^(s*scale*log2e - m), packed to bf16 pairs and written over S
        // x = s * scale * log2(e) - m and the running sums on packed pairs
        // (one f32x2 instruction per two scores), p = 2^x on the ex2 unit
        const uint64_t scale2 = fx::pack2(a.scale_log2, a.scale_log2);
        const uint64_t negm2 = fx::pack2(-m_exp, -m_exp);
        uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};  // 4 independent packed partial sums
        uint32_t pk[KV_TILE / 2];
#pragma unroll
        for (int e = 0; e < KV_TILE / 2; ++e) {
          float x0, x1;
          fx::unpack2(fx::fma2(fx::pack2(s[2 * e], s[2 * e + 1]), scale2, negm2), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          sum2[e & 3] = fx::add2(sum2[e & 3], fx::pack2(p0, p1));
          pk[e] = pack_bf16x2(p0, p1);
        }
        float rowsum;
        {
          float r0, r1;
          fx::unpack2(fx::add2(fx::add2(sum2[0], sum2[1]), fx::add2(sum2[2], sum2[3])), r0, r1);
          rowsum = r0 + r1;
        }
        {
          uint32_t part[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) part[e] = pk[e];
          tmem_st32(s_tmem, part);
#pragma unroll
          for (int e = 0; e < 32; ++e) part[e] = pk[32 + e];
          tmem_st32(s_tmem + 32, part);
        }
        if (tail_zero_v) {
          // rows >= valid of this V tile hold whatever the pool had past the
          // prefix (or stale data): zero them so 0 * V can never be NaN
          const int slot = jg % C::NSTV;
          if (!__all_sync(0xffffffffu, wait_bar(&sm.v_full[slot], (jg / C::NSTV) & 1, ctl))) {
            ok = false;
            break;
          }
          if (r >= valid) {
            for (int hh = 0; hh < C::HALVES; ++hh) {
              uint4* row = reinterpret_cast<uint4*>(sm.v[slot] + ((r >> 3) * C::HALVES + hh) * 1024 + (r & 7) * 128);
#pragma unroll
              for (int e = 0; e < 8; ++e) row[e] = make_uint4(0, 0, 0, 0);
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        if (j > 0 && __any_sync(0xffffffffu, rescale)) {
          // O must hold every earlier PV complete before it is rescaled.  TMEM loads
          // and stores are warp-collective: the whole warp rescales its rows
          // together, with factor 1 for rows whose max did not move enough.
          if (!__all_sync(0xffffffffu, wait_count(&sm.pv_done, jg, ctl))) {
            ok = false;
            break;
          }
          tc_fence_after();
          {
            const float f = !rescale ? 1.f : ((m_run == NEG_INF) ? 0.f : ex2(m_run - m_new));
            l_run *= f;
#pragma unroll
            for (int c = 0; c < D; c += 64) {
              uint32_t u0[32], u1[32];
              tmem_ld32(tmem + lane_base + TMEM_O + c, u0);
              if (c + 32 < D) tmem_ld32(tmem + lane_base + TMEM_O + c + 32, u1);
              tmem_ld_wait();
              reg_fence32(u0);
              reg_fence32(u1);
#pragma unroll
              for (int e = 0; e < 32; ++e) u0[e] = __float_as_uint(__uint_as_float(u0[e]) * f);
#pragma unroll
              for (int e = 0; e < 32; ++e) u1[e] = __float_as_uint(__uint_as_float(u1[e]) * f);
              tmem_st32(tmem + lane_base + TMEM_O + c, u0);
              if (c + 32 < D) tmem_st32(tmem + lane_base + TMEM_O + c + 32, u1);
            }
          }
        }
        m_run = m_use;
        l_run += rowsum;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.p_full[jg % NSB]);
      }
      if (!ok) break;
      // end of the item: wait for its last PV, normalise, store; and see
      // whether another item follows
      int2 e_next;
      const bool epi = __all_sync(0xffffffffu, wait_count(&sm.pv_done, jg, ctl) && queue_entry(k + 1, e_next));
      if (!epi) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv = 1.f / l_run;
      const float lse2 = m_run + __log2f(l_run);
      const size_t orow = ((size_t)b * a.N + node) * a.Hq + h;
      // The CTA's last item goes to the idle K ring (every QK has completed
      // before the last PV could start) as bf16 TMA boxes of 64 columns (one
      // per D half), each 128 rows of 128 bytes: columns c .. c+31 are
      // chunks (c % 64) / 8 .. +3 of box c / 64, chunk k of row r at
      // k ^ (r % 8) (the 128-byte swizzle, conflict-free for these writes).
      // Any other item writes its rows straight to global memory (the rings
      // carry the next items' tiles), 16 bytes a store.
      const bool to_stage = e_next.x < 0;
      __nv_bfloat16* dst = args.direct ? a.out + orow * D : a.part_o + ((size_t)split * rows_all + orow) * D;
      // The loop is kept rolled: unrolled, it changed how the softmax loop
      // above was compiled, which then ran 10% slower on long prefixes.
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_base + TMEM_O + c, u);
        tmem_ld_wait();
        uint8_t* srow = stage + (c / 64) * (ROW_TILE * 128) + r * 128;
        uint32_t w[16];  // the 32 columns as bf16 pairs
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = pack_bf16x2(__uint_as_float(u[2 * e]) * inv, __uint_as_float(u[2 * e + 1]) * inv);
        if (to_stage) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(srow + ((((c % 64) / 8 + q) ^ (r & 7)) << 4)) =
                make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        } else if (active) {
          // a row's 64 bytes here: two 32-byte stores where the output is
          // 32-byte aligned (each a whole DRAM sector), else four of 16
          if (args.out32) {
            st_global_v8(dst + c, w);
            st_global_v8(dst + c + 16, w + 8);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              reinterpret_cast<uint4*>(dst + c)[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          }
        }
      }
      if (active) {
        if (args.direct) {
          if (a.lse) a.lse[orow] = lse2 * 0.69314718055994531f;
        } else {
          a.part_lse[(size_t)split * rows_all + orow] = lse2;
        }
      }
      if (to_stage) {
        fence_proxy_async();
        staged = true;
        last_pos = I.pos;
      } else {
        // O has been read: the next item's first PV may overwrite it (it
        // waits for that item's first P, which follows in program order)
        tc_fence_before();
        __syncwarp();
        if (r == 0) asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sm.items_done)), "r"(k + 1) : "memory");
      }
      e = e_next;
    }
    // every softmax thread reaches this barrier, whatever happened above
    const bool all_staged = named_barrier_and(1, SOFTMAX_THREADS, staged);
    if (all_staged && r == 0) {
      // rows of nodes >= N fall outside the tensor and are not written
      const int node0 = last_pos.rt * args.nodes_per_tile;
      for (int hh = 0; hh < C::HALVES; ++hh) {
        if (args.direct)
          tma_store_4d(&tm_o, stage + hh * (ROW_TILE * 128), 64 * hh, last_pos.g * a.G, node0, last_pos.b);
        else
          tma_store_5d(&tm_po, stage + hh * (ROW_TILE * 128), 64 * hh, last_pos.g * a.G, node0, last_pos.b,
                       last_pos.split);
      }
      bulk_commit_group();
      bulk_wait_read_all();
      asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sm.items_done)), "r"(0x7fffffff) : "memory");
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // A wait gave up.  Nothing may still write this CTA's shared memory or
    // TMEM once it exits: wait (bounded, regardless of the flag) for the last
    // loads each producer issued (only the newest tiles of a ring, as many
    // as it has slots, can be outstanding), for a Q tile still on its way,
    // and for every MMA each issuer started.
    if ((warp == PRODUCER_WARP || warp == V_PRODUCER_WARP) && lane == 0) {
      uint64_t* full = warp == PRODUCER_WARP ? sm.k_full : sm.v_full;
      const int nst = warp == PRODUCER_WARP ? C::NSTK : C::NSTV;
      for (int j = max(0, issued - nst); j < issued; ++j) mbar_wait(&full[j % nst], (j / nst) & 1, a.wait_limit_ns);
    } else if ((warp == QK_WARP || warp == PV_WARP) && lane == 0) {
      if (q_issued > q_landed) mbar_wait(&sm.q_full, (q_issued - 1) & 1, a.wait_limit_ns);
      uint64_t* d = &sm.drain[warp - QK_WARP];
      mma_commit(d);
      mbar_wait(d, 0, a.wait_limit_ns);
    }
    tc_fence_before();
    __syncthreads();
    // Every item this CTA took and did not finish reports the timeout for
    // its sequence: those published and not finished, the one the K producer
    // holds, and (so that the counter still ends at zero) every item it
    // takes from now on.
    if (threadIdx.x == 0) {
      auto report = [&](int it) {
        if (it < 0 || !a.status) return;
        const Item I = make_item(it, a.prefix_len[item_pos(it, args).b], args);
        if (I.work) a.status[I.pos.b] = TS_ERR_TIMEOUT;
      };
      const int pub = single ? (single_work ? 1 : 0) : sm.items_pub, done = sm.items_done;
      for (int k = done; k < pub && k < done + ITEM_Q; ++k) report(single ? first : sm.item_q[k % ITEM_Q].x);
      report(held);
      while (!exhausted) {
        const int it = take_item();
        exhausted = it < 0;
        report(it);
      }
    }
  }
  pdl_trigger();
  if (warp == PRODUCER_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int D>
constexpr size_t smem_bytes() {
  return sizeof(Smem<D>) + 1024;  // + alignment slack for the 1024-byte swizzle atoms
}

// Streaming multiprocessors of the current device (queried once per device).
int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev < 0 || dev >= 64) return -1;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    cache[dev] = n;
  }
  return cache[dev];
}

template <int D>
cudaError_t launch_tc(const AttnArgs& a, cudaStream_t s) {
  TcArgs t{};
  t.a = a;
  t.box_rows = KV_TILE;  // gcd(block_size, 128): block sizes are multiples of 16
  while (a.bs % t.box_rows != 0) t.box_rows >>= 1;
  t.direct = a.max_splits == 1;
  t.n_items = a.row_tiles * a.max_splits * a.B * a.Hkv;
  t.nodes_per_tile = ROW_TILE / a.G;
  t.out32 = (reinterpret_cast<uintptr_t>(t.direct ? (const void*)a.out : (const void*)a.part_o) & 31) == 0;
  t.fd_rt = FastDiv::make(a.row_tiles);
  t.fd_ms = FastDiv::make(a.max_splits);
  t.fd_hkv = FastDiv::make(a.Hkv);
  t.fd_chunk = FastDiv::make(a.chunk_tiles);
  t.fd_bs = FastDiv::make(a.bs);
  t.fd_g = FastDiv::make(a.G);
  t.n_order = (a.n_order == a.B * a.max_splits && a.n_order <= ATTN_ORDER_MAX && a.order_host) ? a.n_order : 0;
  for (int e = 0; e < t.n_order; ++e) t.order[e] = a.order_host[e];
  CUtensorMap m_q, m_kc, m_vc, m_kt, m_vt;
  // q [B, N, Hq, D]: dims (D, Hq, N, B); box (64, G, 128/G, 1) = 128 packed rows
  {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)a.Hq, (uint64_t)a.N, (uint64_t)a.B};
    const uint64_t str[3] = {(uint64_t)D * 2, (uint64_t)a.Hq * D * 2, (uint64_t)a.N * a.Hq * D * 2};
    const uint32_t box[4] = {64, (uint32_t)a.G, (uint32_t)(ROW_TILE / a.G), 1};
    if (!encode_bf16_sw128(&m_q, a.q, 4, dims, str, box)) return cudaErrorInvalidValue;
  }
  // KV pool [num_blocks, Hkv, bs, D] viewed as (64 columns, 8 rows, D/64 halves,
  // bs/8 row groups, num_blocks*Hkv slabs): a box (64, 8, D/64, box_rows/8, 1)
  // lands in shared memory as [row group][half][8 rows x 128 B]
  {
    const uint64_t dims[5] = {64, 8, (uint64_t)(D / 64), (uint64_t)(a.bs / 8), (uint64_t)a.num_blocks * a.Hkv};
    const uint64_t str[4] = {(uint64_t)D * 2, 128, (uint64_t)8 * D * 2, (uint64_t)a.bs * D * 2};
    const uint32_t box[5] = {64, 8, (uint32_t)(D / 64), (uint32_t)(t.box_rows / 8), 1};
    if (!encode_bf16_sw128(&m_kc, a.k_cache, 5, dims, str, box)) return cudaErrorInvalidValue;
    if (!encode_bf16_sw128(&m_vc, a.v_cache, 5, dims, str, box)) return cudaErrorInvalidValue;
  }
  // tree K/V [B, N, Hkv, D]: dims (D, Hkv, N, B); box (64, 1, 128, 1); nodes >= N read as zeros
  {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)a.Hkv, (uint64_t)a.N, (uint64_t)a.B};
    const uint64_t str[3] = {(uint64_t)D * 2, (uint64_t)a.Hkv * D * 2, (uint64_t)a.N * a.Hkv * D * 2};
    const uint32_t box[4] = {64, 1, (uint32_t)KV_TILE, 1};
    if (!encode_bf16_sw128(&m_kt, a.k_tree, 4, dims, str, box)) return cudaErrorInvalidValue;
    if (!encode_bf16_sw128(&m_vt, a.v_tree, 4, dims, str, box)) return cudaErrorInvalidValue;
  }
  // output boxes of 64 columns: bf16 out [B, N, Hq, D] like q (direct), or the
  // bf16 partial of each split [max_splits, B, N, Hq, D]
  CUtensorMap m_o, m_po;
  std::memset(&m_o, 0, sizeof(m_o));
  std::memset(&m_po, 0, sizeof(m_po));
  if (t.direct) {
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)a.Hq, (uint64_t)a.N, (uint64_t)a.B};
    const uint64_t str[3] = {(uint64_t)D * 2, (uint64_t)a.Hq * D * 2, (uint64_t)a.N * a.Hq * D * 2};
    const uint32_t box[4] = {64, (uint32_t)a.G, (uint32_t)(ROW_TILE / a.G), 1};
    if (!encode_bf16_sw128(&m_o, a.out, 4, dims, str, box)) return cudaErrorInvalidValue;
  } else {
    const uint64_t dims[5] = {(uint64_t)D, (uint64_t)a.Hq, (uint64_t)a.N, (uint64_t)a.B, (uint64_t)a.max_splits};
    const uint64_t str[4] = {(uint64_t)D * 2, (uint64_t)a.Hq * D * 2, (uint64_t)a.N * a.Hq * D * 2,
                             (uint64_t)a.B * a.N * a.Hq * D * 2};
    const uint32_t box[5] = {64, (uint32_t)a.G, (uint32_t)(ROW_TILE / a.G), 1, 1};
    if (!encode_bf16_sw128(&m_po, a.part_o, 5, dims, str, box)) return cudaErrorInvalidValue;
  }
  // One CTA per SM (each holds ~225 KB of shared memory), or one per item
  // when there are fewer.  With the items taken longest first, this also
  // beat one CTA per item (left to the hardware's own scheduling) on
  // HBM-bound plans: on 16 paged prefixes of 1-16K tokens, 86.7-87.0
  // against 89.7 us (a CTA goes on to its next item in ~2.7 us, where a new
  // CTA took ~7.4 us to its first tile).
  int ctas = sm_count();
  if (ctas <= 0) return cudaErrorInvalidDevice;
  if (a.max_ctas > 0 && a.max_ctas < ctas) ctas = a.max_ctas;
  dim3 grid(t.n_items < ctas ? t.n_items : ctas);
  return launch_pdl(k_attn_tc<D>, grid, dim3(NUM_THREADS), smem_bytes<D>(), s, t, m_q, m_kc, m_vc, m_kt, m_vt, m_o,
                    m_po);
}

}  // namespace

cudaError_t attn_tc_prepare() {
  // per-process opt-in to the large shared-memory carve-out (not a stream
  // operation; done outside any capture by the first call)
  cudaError_t e = cudaFuncSetAttribute(k_attn_tc<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_bytes<128>());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_attn_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<64>());
}

cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t s) {
  return a.D == 128 ? launch_tc<128>(a, s) : launch_tc<64>(a, s);
}

}  // namespace ts
