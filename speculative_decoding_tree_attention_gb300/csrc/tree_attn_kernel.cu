// tree_attn_kernel.cu -- tree attention over a shared paged prefix on sm_103a.
//
// Sources (titles abbreviated):
//   [EC]  "端云协同推测解码中草稿模型动态生成与验证并行化：探究树形注意力机制与显存碎片整理联合加速":
//         §2.2.2 the tree mask M_tree[i,j] = 0 iff j is an ancestor of i or
//         j = i, else -inf; appendix B (a tree FlashAttention loop): parent
//         index per node, per-node ancestor bitmap, fp32 accumulators and an
//         online softmax.
//   [MM]  "端侧多模态大模型推测解码草稿模型动态剪枝：详解基于重要性采样的树形验证并行加速策略":
//         §3.2 the prefix KV is stored once and reached by index; all
//         branches flattened into one varlen kernel.
//   [LLM] "端侧大模型推测解码草稿模型动态剪枝策略：详解基于重要性采样的树形验证并行加速机制":
//         §2.3.1 variable-length batches through cuSeqLens and block_table.
//
// GB300 design.  One CTA computes a 128-row tile of packed query rows of one
// (sequence, KV head): row R = node * g + head-in-group, so every tree node
// and every query head of a GQA group share each K/V tile that is staged in
// shared memory.  The CTA walks its key range in 64-key tiles:
//   warp 4  (TMA)      loads K and V tiles into a 4-stage ring: four 16-token
//                      pages per tile through the block table (2D tensor map
//                      over the pool), or 64 tree nodes (3D tensor map);
//                      pages past the sequence load as zeros (out of bounds).
//   warp 5  (MMA)      one thread issues tcgen05.mma: S = Q K^T into a
//                      double-buffered TMEM tile (128 x 64 fp32), and
//                      O += P V into a TMEM accumulator (128 x D fp32) with
//                      P read from TMEM as the A operand.
//   warps 0-3          one thread per row: tcgen05.ld of S, the tree mask
//                      from a per-node ancestor bitmask (shared memory), fp32
//                      online softmax in base 2, rescale of O in TMEM only
//                      when the running max grows by more than 2^8, and P as
//                      bf16 pairs stored back to a double-buffered TMEM tile.
// Q, K and V use the 128-byte swizzle that TMA writes, so the MMA reads them
// straight from the ring; P never touches shared memory.  Long prefixes are split over CTAs (split-KV):
// each split writes (O, m, l) in fp32 and a merge kernel combines them.
// Every wait on an mbarrier is bounded; on expiry the CTA reports
// TV_ERR_DEVICE_TIMEOUT for its sequence, drains its copies and returns.
#include <climits>

#include "tv_device.cuh"
#include "tv_launch.h"

namespace tv {
namespace {

constexpr int BM = 128;           // packed query rows per CTA
constexpr int BN = 128;           // keys per tile
constexpr int kSoftmaxThreads = 256;  // warps 0-7
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;     // 8 softmax warps + TMA warp + MMA warp
constexpr int kMaxAncWords = 16;  // 512-node trees
constexpr float kRescaleLog2 = 8.0f;

// Shared-memory layout of a K or V tile: 16 groups of 8 keys; a group holds
// the 64-column halves of its 8 rows one after the other, each half an
// 8 x 128-byte swizzle atom: [group][half][row][128 B].  A 16-token page is
// two consecutive groups, so one TMA box brings a whole page, and for a fixed
// half the 8-row groups sit at a uniform stride (kGroupBytes), which is what
// the MMA descriptors need (K-major for K, MN-major for V).
template <int D>
struct Layout {
  static constexpr int kHalves = D / 64;
  static constexpr int kStages = D == 128 ? 3 : 6;     // K/V ring depth (128-key tiles)
  static constexpr int kGroupBytes = kHalves * 1024;   // 8 keys, all columns
  static constexpr int kTileBytes = BN * D * 2;        // one K or V tile (16 groups)
  static constexpr int kStage0 = 0;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kAnc = kStage0 + kStages * kStageBytes;
  static constexpr int kAncBytes = BM * kMaxAncWords * 4;
  static constexpr int kParent = kAnc + kAncBytes;
  static constexpr int kParentBytes = 512 * 4;
  static constexpr int kXchg = kParent + kParentBytes;  // row max / sum exchange
  static constexpr int kXchgBytes = 3 * 2 * BM * 4;  // slots 0, 1: per-tile max; 2: row sum
  static constexpr int kBar = kXchg + kXchgBytes;
  // full[kStages], empty[kStages], s_full[2], p_full[2], o_done[2], drain,
  // q_ready, s_free[2]
  static constexpr int kNumBars = 2 * kStages + 10;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kTotal = kMisc + 64;
  static constexpr int kAlloc = kTotal + 1024;  // slack for 1024-byte alignment
  // TMEM columns: S[2] at 0 and 128 (fp32), O at 256 (D columns), P at 384
  // (bf16 pairs, 64 columns), Q at 448 (bf16 pairs, D/2 columns)
  static constexpr int kTmemCols = 512;
};

struct Misc {
  uint32_t tmem_base;
  int abort;
  int bad;
};

struct Work {
  int b, kvh, mtile, split;
  int n0, N, L;
  int rows;      // N * g
  int nsplit;    // splits of this sequence
  int k_begin, k_end;
  int n_prefix_tiles, n_node_tiles, T;
  bool last_split;
};

// TMEM lane offset of a softmax warp (its 32-lane quarter).
__device__ __forceinline__ uint32_t lane_off_q(int warp) {
  return static_cast<uint32_t>((warp & 3) * 32) << 16;
}

// Named barriers among the 8 softmax warps (ids 1 and 2; 0 is __syncthreads).
__device__ __forceinline__ void softmax_group_sync() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}
__device__ __forceinline__ void softmax_pair_sync() {
  asm volatile("bar.sync 2, 256;" ::: "memory");
}

__device__ __forceinline__ void record_status(int32_t* status, int b, int code) {
  atomicMax(status + b, code);
}

// Zeros output row r (0..127) of this tile if it is a live row.
template <int D>
__device__ __forceinline__ void zero_rows(const AttnArgs& a, const Work& w, int r) {
  const int R = w.mtile * BM + r;
  if (R >= w.rows) return;
  const int i = R / a.group, h = w.kvh * a.group + R % a.group;
  uint4* dst = reinterpret_cast<uint4*>(a.out + (static_cast<size_t>(w.n0 + i) * a.hq + h) * D);
#pragma unroll
  for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    tree_attn_kernel(const AttnArgs a, const __grid_constant__ AttnMaps maps) {
  using Ly = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ly::kBar);
  constexpr int kStages = Ly::kStages;
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* s_full = bars + 2 * kStages;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 2;
  uint64_t* drain = o_done + 2;
  uint64_t* q_ready = drain + 1;
  uint64_t* s_free = q_ready + 1;
  Misc* misc = reinterpret_cast<Misc*>(smem + Ly::kMisc);
  uint32_t* anc = reinterpret_cast<uint32_t*>(smem + Ly::kAnc);
  int32_t* par = reinterpret_cast<int32_t*>(smem + Ly::kParent);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ------------------------------------------------------------ work item
  Work w;
  w.mtile = blockIdx.x;
  w.split = blockIdx.y;
  w.b = blockIdx.z / a.hkv;
  w.kvh = blockIdx.z % a.hkv;
  w.n0 = a.node_offsets[w.b];
  w.N = a.node_offsets[w.b + 1] - w.n0;
  w.L = max(0, a.prefix_lens[w.b]);
  w.rows = w.N * a.group;
  w.nsplit = max(1, (w.L + a.chunk - 1) / a.chunk);
  if (w.N < 1 || w.mtile * BM >= w.rows || w.split >= w.nsplit) return;  // no work here
  w.last_split = (w.split == w.nsplit - 1);
  w.k_begin = w.split * a.chunk;
  w.k_end = min(w.L, w.k_begin + a.chunk);
  w.n_prefix_tiles = (w.k_end - w.k_begin + BN - 1) / BN;
  w.n_node_tiles = w.last_split ? (w.N + BN - 1) / BN : 0;
  w.T = w.n_prefix_tiles + w.n_node_tiles;
  const int node_lo = (w.mtile * BM) / a.group;
  const int g = a.group;

  // ------------------------------------------------------------ prologue
  // Barriers and TMEM first, so that the TMA warp starts streaming K/V at
  // once; the softmax warps stage Q, validate the tree and build the ancestor
  // masks meanwhile, and release the first MMA through q_ready.
  if (tid == 0) {
    misc->abort = 0;
    misc->bad = (w.N > a.max_nodes || w.N > 512 || w.L > a.max_prefix_len || w.n0 < 0 ||
                 w.n0 + w.N > a.total_nodes) ? 1 : 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&s_full[k], 1);
      mbar_init(&p_full[k], kSoftmaxThreads);
      mbar_init(&o_done[k], 1);
    }
    mbar_init(drain, 1);
    mbar_init(q_ready, kSoftmaxThreads);
    mbar_init(&s_free[0], kSoftmaxThreads);
    mbar_init(&s_free[1], kSoftmaxThreads);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&misc->tmem_base, Ly::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;
  if (misc->bad) {  // the sequence's extent itself is malformed: nothing to read
    if (tid == 0) record_status(a.status, w.b, kBadTree);
    const bool rows_addressable = w.n0 >= 0 && w.N <= a.max_nodes && w.n0 + w.N <= a.total_nodes;
    if (w.nsplit == 1 && rows_addressable && warp < 4) zero_rows<D>(a, w, tid);
    if (warp == kMmaWarp) tmem_dealloc(tmem, Ly::kTmemCols);
    return;
  }
  const uint32_t tmem_s0 = tmem;        // S buffers at columns 0 and 128
  const uint32_t tmem_o = tmem + 256;   // O accumulator at columns 256 .. 256+D-1
  const uint32_t tmem_p = tmem + 384;   // P (A operand of P.V)
  const uint32_t tmem_q = tmem + 448;   // Q tile (A operand of Q.K^T)
  volatile int* abort_flag = &misc->abort;

  if (warp == kTmaWarp) {
    // ---------------------------------------------------------- TMA producer
    // The whole warp issues: lane 0 arms the stage's barrier, then each lane
    // issues one box: a prefix tile is 8 pages x {K, V} (one 5-D box per page
    // and tensor), a node tile is 16 groups of 8 nodes x {K, V}.
    if (lane == 0) {
      prefetch_tmap(&maps.k_pool);
      prefetch_tmap(&maps.v_pool);
      prefetch_tmap(&maps.k_nodes);
      prefetch_tmap(&maps.v_nodes);
    }
    constexpr int kPages = BN / 16;
    constexpr int kPastEnd = INT_MIN;                 // page past the prefix end -> zeros
    const int my_kv = lane & 1;
    const int my_unit = lane >> 1;                    // page (prefix) or 8-node group (nodes)
    const bool prefix_lane = my_unit < kPages;
    const int pool_pages = a.num_blocks * a.hkv;
    const int32_t* btab = a.block_table + static_cast<size_t>(w.b) * a.max_blocks_per_seq;
    auto fetch_block = [&](int t) -> int {
      const int lp = (w.k_begin + t * BN) / 16 + my_unit;
      return (prefix_lane && lp * 16 < w.k_end) ? __ldg(btab + lp) : kPastEnd;
    };
    int blk_next = w.n_prefix_tiles > 0 ? fetch_block(0) : kPastEnd;
    int issued = 0;
    bool ok = true;
    for (int t = 0; t < w.T; ++t) {
      const int st = t % kStages;
      const int blk = blk_next;
      if (t + 1 < w.n_prefix_tiles) blk_next = fetch_block(t + 1);  // overlaps the wait
      if (lane == 0) ok = mbar_wait(&empty[st], ((t / kStages) & 1) ^ 1, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane == 0) mbar_arrive_expect_tx(&full[st], 2 * Ly::kTileBytes);
      __syncwarp();
      uint8_t* tile = smem + Ly::kStage0 + st * Ly::kStageBytes + my_kv * Ly::kTileBytes;
      if (t < w.n_prefix_tiles) {
        if (prefix_lane) {
          int page = pool_pages;  // out of bounds: zero fill
          if (blk >= 0 && blk < a.num_blocks) {
            page = blk * a.hkv + w.kvh;
          } else if (blk != kPastEnd && !misc->bad) {  // malformed block id: zeros, reported
            misc->bad = 1;
            record_status(a.status, w.b, kBadTree);
          }
          tma_load_5d(tile + my_unit * 2 * Ly::kGroupBytes, my_kv ? &maps.v_pool : &maps.k_pool,
                      &full[st], 0, 0, 0, 0, page);
        }
      } else {
        const int node0 = w.n0 + (t - w.n_prefix_tiles) * BN + my_unit * 8;
        tma_load_4d(tile + my_unit * Ly::kGroupBytes, my_kv ? &maps.v_nodes : &maps.k_nodes,
                    &full[st], 0, node0, 0, w.kvh);
      }
      ++issued;
    }
    if (lane == 0) {
      if (!ok) {
        record_status(a.status, w.b, kDeviceTimeout);
        misc->abort = 1;
      }
      // drain: every issued copy has landed before the CTA may exit
      for (int t = max(0, issued - kStages); t < issued; ++t)
        mbar_wait(&full[t % kStages], (t / kStages) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(BM, BN, 0);  // M=128, N=128: full-rate shape
      constexpr uint32_t idesc_o = idesc_bf16(BM, D, 1);
      bool ok = true;
      // Descriptors are built once; each MMA adds a compile-time offset to the
      // start-address field (16-byte units; shared addresses stay < 2^18).
      // K (K-major): 8-row groups at kGroupBytes, halves at +1024.
      // V (MN-major): 8-key groups at kGroupBytes, column halves at +1024.
      const uint64_t dk0 = smem_desc(smem_u32(smem + Ly::kStage0), 16, Ly::kGroupBytes);
      const uint64_t dv0 = smem_desc(smem_u32(smem + Ly::kStage0 + Ly::kTileBytes), 1024, Ly::kGroupBytes);
      // S(t) = Q K(t)^T into S buffer t&1 (caller checked K(t) landed and the
      // buffer is free)
      auto issue_s = [&](int t) {
        const uint64_t dk = dk0 + static_cast<uint64_t>((t % kStages) * (Ly::kStageBytes >> 4));
        const uint32_t d = tmem_s0 + (t & 1) * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // A = Q from TMEM (16 dims = 8 columns per step), B = K from the ring
          const uint32_t boff = ((kk >> 2) * 1024 + (kk & 3) * 32) >> 4;
          mma_bf16_ts(d, tmem_q + kk * 8, dk + boff, idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[t & 1]);
      };
      // O += P(t) V(t) (caller checked P(t) is in TMEM)
      auto issue_pv = [&](int t) {
        const int st = t % kStages;
        const uint64_t dv = dv0 + static_cast<uint64_t>(st * (Ly::kStageBytes >> 4));
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // A = P from TMEM: 16 keys = 8 columns of bf16 pairs = 2 groups of V
          mma_bf16_ts(tmem_o, tmem_p + kk * 8, dv + ((kk * 2 * Ly::kGroupBytes) >> 4), idesc_o,
                      (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&o_done[t & 1]);
        mma_commit(&empty[st]);
      };
      // Issue in whichever order the inputs become ready: S(t) needs K(t) in
      // the ring and S buffer t&1 released by the softmax of tile t-2
      // (s_free, right after it loaded S(t-2) into registers), so the tensor
      // core computes S two tiles ahead; P(t).V(t) needs P(t) (p_full).
      ok = mbar_wait(q_ready, 0, abort_flag);
      tc_fence_after();
      int ns = 0, npv = 0;
      unsigned long long t_idle = 0;
      while (ok && npv < w.T) {
        bool progressed = false;
        if (ns < w.T && ns < npv + 3 &&
            (ns < 2 || mbar_test_wait(&s_free[ns & 1], ((ns - 2) >> 1) & 1)) &&
            mbar_test_wait(&full[ns % kStages], (ns / kStages) & 1)) {
          tc_fence_after();
          issue_s(ns);
          ++ns;
          progressed = true;
        }
        if (npv < ns && mbar_test_wait(&p_full[npv & 1], (npv >> 1) & 1)) {
          tc_fence_after();
          issue_pv(npv);
          ++npv;
          progressed = true;
        }
        if (progressed) {
          t_idle = 0;
        } else if (t_idle == 0) {
          t_idle = global_ns();
        } else if (global_ns() - t_idle > kWaitLimitNs || misc->abort) {
          ok = false;
        }
      }
      if (!ok) {
        record_status(a.status, w.b, kDeviceTimeout);
        misc->abort = 1;
      }
      // drain: all MMAs issued by this thread complete before TMEM is freed
      mma_commit(drain);
      mbar_wait(drain, 0);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- softmax warps
    // Warps 0-7: warp w owns rows 32*(w%4)..+31 (its TMEM lane quarter) and
    // column half hc = w/4 of every 64-key tile, so two threads share a row
    // and each scheduler runs two softmax warps.
    const int r = (warp & 3) * 32 + lane;  // row of the tile == TMEM lane
    const int hc = warp >> 2;              // which 32 keys of each tile
    const int sid = hc * 128 + r;          // 0..255
    const int R = w.mtile * BM + r;
    const bool live = R < w.rows;
    float* xchg = reinterpret_cast<float*>(smem + Ly::kXchg);  // [3 slots][2 halves][128 rows]
    // tree of this sequence into shared memory, validated
    for (int i = sid; i < w.N; i += kSoftmaxThreads) {
      const int p = __ldg(a.parent + w.n0 + i);
      par[i] = p;
      if (!(i == 0 ? p == -1 : (p >= 0 && p < i))) misc->bad = 1;
    }
    // Q tile -> TMEM (one row per lane, bf16 pairs; this thread stores the
    // half hc of its row); padding rows are zero.
    {
      constexpr int kWords = D / 4;  // 32-bit words per half row
      uint32_t qw[kWords];
      if (live) {
        const int i = R / g, h = w.kvh * g + R % g;
        const uint4* src = reinterpret_cast<const uint4*>(
            a.q + (static_cast<size_t>(w.n0 + i) * a.hq + h) * D + hc * (D / 2));
#pragma unroll
        for (int c = 0; c < kWords / 4; ++c) {
          const uint4 v = __ldg(src + c);
          qw[4 * c] = v.x;
          qw[4 * c + 1] = v.y;
          qw[4 * c + 2] = v.z;
          qw[4 * c + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int c = 0; c < kWords; ++c) qw[c] = 0u;
      }
      if constexpr (kWords == 32) {
        tmem_st32(tmem_q + hc * 32 + lane_off_q(warp), qw);
      } else {
        tmem_st16(tmem_q + hc * 16 + lane_off_q(warp), qw);
      }
      tmem_st_wait();
    }
    softmax_group_sync();
    const bool tree_ok = misc->bad == 0;
    if (!tree_ok && sid == 0) record_status(a.status, w.b, kBadTree);
    // ancestor-or-self bitmask of the tile's nodes (node tiles only)
    if (w.last_split && hc == 0) {
      const int i = node_lo + r;
      uint32_t* row = anc + r * kMaxAncWords;
#pragma unroll
      for (int k = 0; k < kMaxAncWords; ++k) row[k] = 0u;
      if (tree_ok && i < w.N) {
        for (int k = i; k >= 0; k = par[k]) row[k >> 5] |= 1u << (k & 31);
      }
    }
    tc_fence_before();  // Q is in TMEM before the MMA warp is released
    mbar_arrive(q_ready);
    softmax_group_sync();      // ancestor rows are read across threads
    const int i_node = live ? R / g : 0;  // local node of this row
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t* my_anc = anc + (i_node - node_lo) * kMaxAncWords;
    float m_run = -INFINITY;  // reference max (log2 units), shared by the pair
    float l_run = 0.0f;       // this thread's half of the row sum
    bool ok = true;
    // Every softmax warp passes the same sequence of named barriers (one per
    // tile): after a failed (timed-out) wait a warp keeps looping but skips
    // the work, so that its partner warp can never block on it.
    for (int t = 0; t < w.T; ++t) {
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t & 1], (t >> 1) & 1, abort_flag));
      // this thread's 64 scores of the tile (keys hc*64 .. hc*64+63)
      float x[64];
      if (ok) {
        uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&x[0]);
        uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&x[32]);
        tc_fence_after();
        tmem_ld32(tmem_s0 + (t & 1) * BN + hc * 64 + lane_off, lo);
        tmem_ld32(tmem_s0 + (t & 1) * BN + hc * 64 + 32 + lane_off, hi);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&s_free[t & 1]);  // S buffer t&1 may now take S(t+2)
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = 0.0f;
      }
      // mask (scores stay unscaled; the scale is folded into the exponent)
      int valid_keys = BN;
      if (t < w.n_prefix_tiles) {
        valid_keys = min(BN, w.k_end - (w.k_begin + t * BN));
        if (valid_keys < BN) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (hc * 64 + c >= valid_keys) x[c] = -INFINITY;
        }
      } else {
        const int j0 = (t - w.n_prefix_tiles) * BN + hc * 64;
        const uint32_t b0 = live ? my_anc[j0 >> 5] : 0u;
        const uint32_t b1 = live ? my_anc[(j0 >> 5) + 1] : 0u;
        const int nvalid = w.N - j0;  // node columns past the tree are masked
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const uint32_t bit = c < 32 ? (b0 >> c) & 1u : (b1 >> (c - 32)) & 1u;
          if (!bit || c >= nvalid) x[c] = -INFINITY;
        }
      }
      float mx[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) mx[c] = fmaxf(x[c], x[c + 32]);
#pragma unroll
      for (int h = 16; h >= 1; h >>= 1)
#pragma unroll
        for (int c = 0; c < h; ++c) mx[c] = fmaxf(mx[c], mx[c + h]);
      // the row max of both halves (exchange slot t&1, so that the next
      // tile's write cannot overtake the partner's read)
      xchg[((t & 1) * 2 + hc) * 128 + r] = mx[0];
      softmax_pair_sync();
      if (!ok) continue;  // skip the work, keep the barrier sequence
      const float tmax = fmaxf(mx[0], xchg[((t & 1) * 2 + (hc ^ 1)) * 128 + r]) * a.scale_log2;
      // online softmax with a lazily rescaled reference max (same decision
      // in both threads of a row)
      float alpha = 1.0f;
      bool rescale = false;
      if (tmax != -INFINITY) {
        if (m_run == -INFINITY) {
          m_run = tmax;
        } else if (tmax > m_run + kRescaleLog2) {
          alpha = exp2f(m_run - tmax);
          m_run = tmax;
          rescale = true;
        }
      }
      // P(t-1).V(t-1) must be complete: it reads the single P buffer and
      // accumulates into O
      if (t >= 1) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, abort_flag));
        if (!ok) continue;
        tc_fence_after();
      }
      if (t >= 1 && __any_sync(0xffffffffu, rescale)) {
        // this thread rescales its half of the O row
#pragma unroll
        for (int c0 = hc * (D / 2); c0 < (hc + 1) * (D / 2); c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tmem_o + c0 + lane_off, o);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tmem_st32(tmem_o + c0 + lane_off, o);
        }
      }
      l_run *= alpha;
      const float mref = (m_run == -INFINITY) ? 0.0f : m_run;
      uint32_t pk[32];  // bf16 pairs: column c of this half holds keys 2c (low), 2c+1
      float ls[8];
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        float part = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          // p = 2^(s * scale * log2(e) - m); masked scores are -inf -> 0
          const float p0 = ex2_approx(fmaf(x[c8 * 8 + 2 * k], a.scale_log2, -mref));
          const float p1 = ex2_approx(fmaf(x[c8 * 8 + 2 * k + 1], a.scale_log2, -mref));
          pk[c8 * 4 + k] = pack_bf16x2(p0, p1);
          part += p0 + p1;
        }
        ls[c8] = part;
      }
      tmem_st32(tmem_p + hc * 32 + lane_off, pk);
      l_run += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      // keys past the prefix end in this tile: clear their V rows (page tails
      // may hold stale data; P is 0 there but 0 * NaN would poison O)
      if (valid_keys < BN) {
        const int st = t % kStages;
        mbar_wait(&full[st], (t / kStages) & 1);  // acquire the TMA writes
        uint8_t* vt = smem + Ly::kStage0 + st * Ly::kStageBytes + Ly::kTileBytes;
        for (int idx = sid; idx < (BN - valid_keys) * Ly::kHalves; idx += kSoftmaxThreads) {
          const int row = valid_keys + idx / Ly::kHalves, h = idx % Ly::kHalves;
          uint4* p = reinterpret_cast<uint4*>(vt + (row >> 3) * Ly::kGroupBytes + h * 1024 +
                                              (row & 7) * 128);
#pragma unroll
          for (int k = 0; k < 8; ++k) p[k] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();  // generic writes, read by the MMA
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[t & 1]);
    }
    // the row sum of both halves (slot 2: the max slots may still be read)
    xchg[(2 * 2 + hc) * 128 + r] = l_run;
    softmax_pair_sync();
    const float l_row = l_run + xchg[(2 * 2 + (hc ^ 1)) * 128 + r];
    if (!ok) {
      record_status(a.status, w.b, kDeviceTimeout);
      misc->abort = 1;
    } else if (w.T > 0 && __all_sync(0xffffffffu, mbar_wait(&o_done[(w.T - 1) & 1],
                                                            ((w.T - 1) >> 1) & 1, abort_flag))) {
      tc_fence_after();
      // ------------------------------------------------------------ epilogue
      const bool final_out = (w.nsplit == 1);
      const float inv_l = (l_row > 0.0f) ? 1.0f / l_row : 0.0f;
      const size_t unit = (static_cast<size_t>(w.b) * a.hkv + w.kvh) * a.mtiles_max + w.mtile;
      const size_t prow_idx = (unit * a.max_splits + w.split) * BM + r;
#pragma unroll
      for (int c0 = hc * (D / 2); c0 < (hc + 1) * (D / 2); c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tmem_o + c0 + lane_off, o);
        tmem_ld_wait();
        if (!live) continue;
        if (final_out) {
          const int h = w.kvh * g + R % g;
          uint4* dst = reinterpret_cast<uint4*>(a.out + (static_cast<size_t>(w.n0 + i_node) * a.hq + h) * D + c0);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * k + 0]) * inv_l, __uint_as_float(o[8 * k + 1]) * inv_l);
            v.y = pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv_l, __uint_as_float(o[8 * k + 3]) * inv_l);
            v.z = pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv_l, __uint_as_float(o[8 * k + 5]) * inv_l);
            v.w = pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv_l, __uint_as_float(o[8 * k + 7]) * inv_l);
            dst[k] = v;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(a.ws_o + prow_idx * D + c0);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                 __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]));
        }
      }
      if (live && !final_out && hc == 0) a.ws_ml[prow_idx] = make_float2(m_run, l_row);
    } else if (w.T > 0) {
      record_status(a.status, w.b, kDeviceTimeout);
      misc->abort = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // a malformed tree or block id: the only writer of these rows writes zeros
  // (each row by the thread that wrote it in the epilogue, so zeros win)
  if (misc->bad && w.nsplit == 1 && warp < 4) zero_rows<D>(a, w, tid);
  if (warp == kMmaWarp) tmem_dealloc(tmem, Ly::kTmemCols);
}

// Combines the split partials: one warp per packed output row,
// O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s, lanes over D (float4).
constexpr int kMergeWarps = 8;
template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32) tree_attn_merge(const AttnArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x / (BM / kMergeWarps);
  const int r = (blockIdx.x % (BM / kMergeWarps)) * kMergeWarps + warp;
  const int mtile = unit % a.mtiles_max;
  const int bk = unit / a.mtiles_max;
  const int b = bk / a.hkv, kvh = bk % a.hkv;
  const int n0 = a.node_offsets[b];
  const int N = a.node_offsets[b + 1] - n0;
  const int L = max(0, a.prefix_lens[b]);
  const int nsplit = max(1, (L + a.chunk - 1) / a.chunk);
  const int rows = N * a.group;
  if (nsplit == 1 || N < 1 || N > a.max_nodes || L > a.max_prefix_len || n0 < 0 ||
      n0 + N > a.total_nodes)
    return;
  const int R = mtile * BM + r;
  if (R >= rows) return;
  const int i = R / a.group, h = kvh * a.group + R % a.group;
  uint16_t* dst = a.out + (static_cast<size_t>(n0 + i) * a.hq + h) * D;
  constexpr int kPer = D / 32;  // elements per lane (4 for D=128, 2 for D=64)
  if (a.status[b] == kBadTree) {
    for (int d = lane; d < D; d += 32) dst[d] = 0;
    return;
  }
  const size_t base = (static_cast<size_t>(unit) * a.max_splits) * BM + r;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, a.ws_ml[base + static_cast<size_t>(s) * BM].x);
  const float mref = (M == -INFINITY) ? 0.0f : M;
  float acc[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) acc[k] = 0.0f;
  float lsum = 0.0f;
  for (int s = 0; s < nsplit; ++s) {
    const size_t pr = base + static_cast<size_t>(s) * BM;
    const float2 ml = a.ws_ml[pr];
    const float wgt = (ml.x == -INFINITY) ? 0.0f : exp2f(ml.x - mref);
    lsum += wgt * ml.y;
    const float* src = a.ws_o + pr * D + lane * kPer;
    if constexpr (kPer == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      acc[0] += wgt * v.x;
      acc[1] += wgt * v.y;
      acc[2] += wgt * v.z;
      acc[3] += wgt * v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2*>(src);
      acc[0] += wgt * v.x;
      acc[1] += wgt * v.y;
    }
  }
  const float inv = (lsum > 0.0f) ? 1.0f / lsum : 0.0f;
  if constexpr (kPer == 4) {
    uint2 o;
    o.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    o.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst + lane * 4) = o;
  } else {
    *reinterpret_cast<uint32_t*>(dst + lane * 2) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
}

}  // namespace

size_t tree_attention_smem_bytes(int head_dim) {
  return head_dim == 64 ? Layout<64>::kAlloc : Layout<128>::kAlloc;
}

int launch_tree_attention(const AttnArgs& a, const AttnMaps& maps, cudaStream_t stream) {
  const dim3 grid(a.mtiles_max, a.max_splits, a.batch * a.hkv);
  cudaError_t e;
  static thread_local int attr_set_device = -1;  // the attribute is set once per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_set_device != dev) {
    cudaFuncSetAttribute(tree_attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         Layout<128>::kAlloc);
    cudaFuncSetAttribute(tree_attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         Layout<64>::kAlloc);
    attr_set_device = dev;
  }
  if (a.head_dim == 128) {
    const int smem = Layout<128>::kAlloc;
    tree_attn_kernel<128><<<grid, kThreads, smem, stream>>>(a, maps);
    e = cudaGetLastError();
    if (e == cudaSuccess && a.max_splits > 1) {
      tree_attn_merge<128><<<a.batch * a.hkv * a.mtiles_max * (BM / kMergeWarps),
                             kMergeWarps * 32, 0, stream>>>(a);
      e = cudaGetLastError();
    }
  } else {
    const int smem = Layout<64>::kAlloc;
    tree_attn_kernel<64><<<grid, kThreads, smem, stream>>>(a, maps);
    e = cudaGetLastError();
    if (e == cudaSuccess && a.max_splits > 1) {
      tree_attn_merge<64><<<a.batch * a.hkv * a.mtiles_max * (BM / kMergeWarps),
                            kMergeWarps * 32, 0, stream>>>(a);
      e = cudaGetLastError();
    }
  }
  return e == cudaSuccess ? 0 : -1;
}

}  // namespace tv
