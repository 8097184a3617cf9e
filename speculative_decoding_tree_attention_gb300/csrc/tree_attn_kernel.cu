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
// shared memory.  The CTA walks its key range in 128-key tiles:
//   warp 8  (TMA)      loads K and V tiles into two shared-memory rings: one 5-D
//                      box per 16-token page through the block table (eight
//                      pages per tile and tensor), or 16 boxes of 8 tree nodes;
//                      pages past the sequence load as zeros (out of bounds).
//   warps 9, 10 (MMA)  one thread each issues tcgen05.mma: warp 9 S(t) = Q K^T
//                      into one of two TMEM score buffers (128 x 128 fp32)
//                      with Q read from TMEM, warp 10 O += P(t) V into a TMEM
//                      accumulator (128 x D fp32) with P read from TMEM.
//   warps 0-7          two softmax lanes: warps 0-3 take the even tiles,
//                      warps 4-7 the odd ones, one thread per row.  Per
//                      tile: tcgen05.ld of S (the buffer is released at
//                      once), the tree mask from a per-node ancestor bitmask
//                      (shared memory), the row max, fp32 online softmax in
//                      base 2 against a running max that the two lanes hand
//                      to each other through mbarriers and that moves only
//                      when it grows by more than 2^8 (O is then rescaled in
//                      TMEM), and P as bf16 pairs into TMEM.  Each scheduler
//                      runs one warp of each lane, so the exponentials of one
//                      tile overlap the loads and maxima of the next.
// K and V use the 128-byte swizzle that TMA writes, so the MMA reads them
// straight from the ring; Q and P never touch shared memory.  Long prefixes
// may be split over CTAs (split-KV): the splits of a tile run as one
// thread-block cluster, each keeps its (O, m, l) in fp32 in its own shared
// memory, and the cluster combines them through distributed shared memory.
// Every wait on an mbarrier is bounded; on expiry the CTA reports
// TV_ERR_DEVICE_TIMEOUT for its sequence, drains its copies and returns.
#include <climits>

#include <cooperative_groups.h>

#include "tv_device.cuh"
#include "tv_launch.h"

namespace tv {
namespace {

constexpr int BM = 128;           // packed query rows per CTA
constexpr int BN = 128;           // keys per tile
constexpr int kSoftmaxThreads = 256;  // warps 0-7: two lanes of four warps
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;       // issues S = Q K^T; owns the TMEM allocation
constexpr int kPvWarp = 10;       // issues O += P V
constexpr int kThreads = 352;     // 8 softmax warps + TMA warp + 2 MMA warps
constexpr int kMaxAncWords = 16;  // 512-node trees
constexpr int kAncStride = kMaxAncWords + 1;  // odd word stride: rows of a warp hit distinct banks
constexpr float kRescaleLog2 = 8.0f;
constexpr int kOrderMax = 256;    // batches up to this size run longest sequence first

// Shared-memory layout of a K or V tile: 16 groups of 8 keys; a group holds
// the 64-column halves of its 8 rows one after the other, each half an
// 8 x 128-byte swizzle atom: [group][half][row][128 B].  A 16-token page is
// two consecutive groups, so one TMA box brings a whole page, and for a fixed
// half the 8-row groups sit at a uniform stride (kGroupBytes), which is what
// the MMA descriptors need (K-major for K, MN-major for V).
template <int D>
struct Layout {
  static constexpr int kHalves = D / 64;
  static constexpr int kStages = D == 128 ? 3 : 6;     // depth of the K ring and of the V ring
  static constexpr int kGroupBytes = kHalves * 1024;   // 8 keys, all columns
  static constexpr int kTileBytes = BN * D * 2;        // one K or V tile (16 groups)
  static constexpr int kKRing = 0;                     // kStages K tiles
  static constexpr int kVRing = kKRing + kStages * kTileBytes;  // kStages V tiles
  static constexpr int kAnc = kVRing + kStages * kTileBytes;
  static constexpr int kAncBytes = BM * kAncStride * 4;
  static constexpr int kParent = kAnc + kAncBytes;
  static constexpr int kParentBytes = 512 * 4;
  static constexpr int kXchg = kParent + kParentBytes;  // row max / sum exchange
  // running max after tile t (slot t & 1, 2 x 128 floats), then the
  // final (reference max, row sum) of each lane (2 x 128 float2)
  static constexpr int kXchgBytes = 2 * BM * 4 + 2 * BM * 8;
  // block ids of the pages of the last 8 K tiles issued (8 per tile), reused
  // by the V copies of the same tiles
  static constexpr int kBlk = kXchg + kXchgBytes;
  static constexpr int kBlkBytes = 8 * 8 * 4;
  // per-sequence (prefix length, first node, last node + 1) and the
  // longest-first order of the sequences (batches up to kOrderMax)
  static constexpr int kSeq = kBlk + kBlkBytes;
  static constexpr int kSeqBytes = 4 * kOrderMax * 4;
  static constexpr int kBar = kSeq + kSeqBytes;
  // kfull[kStages], kempty[kStages], vfull[kStages], vempty[kStages],
  // s_full[2], s_free[2], p_full, o_done[2], drain[2], chain[2][4], q_ready
  static constexpr int kNumBars = 4 * kStages + 18;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kTotal = kMisc + 64;
  static constexpr int kAlloc = kTotal + 1024;  // slack for 1024-byte alignment
  // TMEM columns: S buffers (128 x 128 fp32) at 0 and 128; O at 256 (D
  // columns); P (128 keys as bf16 pairs, 64 columns) at 384; Q at 448 (bf16
  // pairs, D/2 columns).
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

// max of three (NaN operands are ignored, as in fmaxf)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Named barrier 1 joins the 8 softmax warps (0 is __syncthreads).
__device__ __forceinline__ void softmax_group_sync() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
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

// Split-KV partials: each split of a tile keeps its raw O rows (fp32, rows
// padded by 4 floats so that a warp's row stores and reads are free of bank
// conflicts) and per-row (m, l) in its own shared memory, over the K ring,
// which is idle once the last S = Q K^T has completed.
template <int D>
struct Partial {
  static constexpr int kStride = D + 4;                 // floats per row
  static constexpr int kO = 0;                          // offset in the K ring
  static constexpr int kMl = BM * kStride * 4;
  static constexpr int kBytes = kMl + BM * 8;
  static_assert(kBytes <= Layout<D>::kStages * Layout<D>::kTileBytes, "partial exceeds the K ring");
};

// Combines the NS splits of this tile (the CTAs of the cluster) for the rows
// r = rank, rank + NS, ... : O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M)
// l_s, reading every split's partial through distributed shared memory.  A
// warp takes a group of rows, four columns per lane, and issues all of the
// group's loads before combining them (16 partial rows in flight per lane).
// A tile whose sequence was found malformed by any split (`bad` flag of any
// CTA of the cluster) gets zeros.
template <int D, int NS>
__device__ __forceinline__ void merge_rows_ns(const AttnArgs& a, const Work& w, uint8_t* ring,
                                              const int* bad_flag, int sid, int rank) {
  namespace cg = cooperative_groups;
  using Pt = Partial<D>;
  constexpr int kWarps = kSoftmaxThreads / 32;
  constexpr int kRows = (16 / NS) > 0 ? 16 / NS : 1;  // rows per warp and group
  cg::cluster_group cluster = cg::this_cluster();
  bool bad = false;
#pragma unroll
  for (int s = 0; s < NS; ++s) bad |= *cluster.map_shared_rank(bad_flag, s) != 0;
  const float* o_peer[NS];
  const float2* ml_peer[NS];
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    o_peer[s] = cluster.map_shared_rank(reinterpret_cast<const float*>(ring + Pt::kO), s);
    ml_peer[s] = cluster.map_shared_rank(reinterpret_cast<const float2*>(ring + Pt::kMl), s);
  }
  const int lane = sid & 31;
  for (int r0 = rank + (sid >> 5) * NS; r0 < BM; r0 += kRows * kWarps * NS) {
    int rr[kRows];
    bool ok_row[kRows];
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      rr[k] = r0 + k * kWarps * NS;
      ok_row[k] = rr[k] < BM && w.mtile * BM + rr[k] < w.rows;
    }
    for (int c = lane * 4; c < D; c += 128) {
      float2 ml[kRows][NS];
      float4 v[kRows][NS];
#pragma unroll
      for (int k = 0; k < kRows; ++k)
#pragma unroll
        for (int s = 0; s < NS; ++s)
          if (ok_row[k]) {
            ml[k][s] = ml_peer[s][rr[k]];
            v[k][s] = *reinterpret_cast<const float4*>(o_peer[s] + rr[k] * Pt::kStride + c);
          }
#pragma unroll
      for (int k = 0; k < kRows; ++k) {
        if (!ok_row[k]) continue;
        float M = -INFINITY;
#pragma unroll
        for (int s = 0; s < NS; ++s) M = fmaxf(M, ml[k][s].x);
        const float mref = (M == -INFINITY) ? 0.0f : M;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float lsum = 0.0f;
#pragma unroll
        for (int s = 0; s < NS; ++s) {
          const float wgt = (ml[k][s].x == -INFINITY) ? 0.0f : exp2f(ml[k][s].x - mref);
          lsum += wgt * ml[k][s].y;
          acc.x += wgt * v[k][s].x;
          acc.y += wgt * v[k][s].y;
          acc.z += wgt * v[k][s].z;
          acc.w += wgt * v[k][s].w;
        }
        const float inv = (lsum > 0.0f) ? __frcp_rn(lsum) : 0.0f;
        uint2 o = make_uint2(0u, 0u);
        if (!bad) {
          o.x = pack_bf16x2(acc.x * inv, acc.y * inv);
          o.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        }
        const int R = w.mtile * BM + rr[k];
        const int i = R / a.group, h = w.kvh * a.group + R % a.group;
        *reinterpret_cast<uint2*>(a.out + (static_cast<size_t>(w.n0 + i) * a.hq + h) * D + c) = o;
      }
    }
  }
}

template <int D>
__device__ __forceinline__ void merge_rows(const AttnArgs& a, const Work& w, uint8_t* ring,
                                           const int* bad_flag, int sid, int rank) {
  switch (w.nsplit) {
    case 2: merge_rows_ns<D, 2>(a, w, ring, bad_flag, sid, rank); break;
    case 3: merge_rows_ns<D, 3>(a, w, ring, bad_flag, sid, rank); break;
    case 4: merge_rows_ns<D, 4>(a, w, ring, bad_flag, sid, rank); break;
    case 5: merge_rows_ns<D, 5>(a, w, ring, bad_flag, sid, rank); break;
    case 6: merge_rows_ns<D, 6>(a, w, ring, bad_flag, sid, rank); break;
    case 7: merge_rows_ns<D, 7>(a, w, ring, bad_flag, sid, rank); break;
    case 8: merge_rows_ns<D, 8>(a, w, ring, bad_flag, sid, rank); break;
    default: break;
  }
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
  uint64_t* kfull = bars;
  uint64_t* kempty = bars + kStages;
  uint64_t* vfull = bars + 2 * kStages;
  uint64_t* vempty = bars + 3 * kStages;
  uint64_t* s_full = bars + 4 * kStages;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  // o_done[t & 1] completes with P(t).V.  A wait for P(t-1).V comes after the
  // same lane has seen P(t-2).V (or before any), so the phase of P(t-3).V is
  // complete and the parity ((t-1) >> 1) & 1 cannot alias an older phase
  // (one barrier for all tiles could: P(t-2).V may still be in flight).
  uint64_t* o_done = p_full + 1;
  uint64_t* drain = o_done + 2;  // one per MMA-issuing thread
  // running-max hand-off: chain[l][q] completes once per tile of lane l
  // for the rows of lane quarter q (arrived by the warp of lane l, awaited by
  // the warp of the other lane that owns the same rows)
  uint64_t* chain = drain + 2;
  uint64_t* q_ready = chain + 8;
  Misc* misc = reinterpret_cast<Misc*>(smem + Ly::kMisc);
  uint32_t* anc = reinterpret_cast<uint32_t*>(smem + Ly::kAnc);
  int32_t* par = reinterpret_cast<int32_t*>(smem + Ly::kParent);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ------------------------------------------------------------ work item
  // Grid z enumerates (sequence rank, KV head).  For batches of 2 up to
  // kOrderMax the rank orders the sequences by decreasing work (prefix plus
  // tree keys, ties by index), so that the CTAs that run longest are
  // dispatched first and the launch does not end on a tail of long CTAs.
  // The extents of all sequences are loaded first; barrier set-up and the
  // TMEM allocation below overlap the load latency.
  int* seq = reinterpret_cast<int*>(smem + Ly::kSeq);  // [4][kOrderMax]
  const bool ordered = a.batch > 1 && a.batch <= kOrderMax;
  if (ordered && tid < a.batch) {
    seq[tid] = max(0, __ldg(a.prefix_lens + tid));
    seq[kOrderMax + tid] = __ldg(a.node_offsets + tid);
    seq[2 * kOrderMax + tid] = __ldg(a.node_offsets + tid + 1);
  }
  Work w;
  w.mtile = blockIdx.x;
  w.split = blockIdx.y;
  w.kvh = blockIdx.z % a.hkv;

  // ------------------------------------------------------------ prologue
  if (tid == 0) {
    misc->abort = 0;
    misc->bad = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&s_full[k], 1);
      mbar_init(&s_free[k], kSoftmaxThreads / 2);
    }
    mbar_init(p_full, kSoftmaxThreads / 2);
    mbar_init(&o_done[0], 1);
    mbar_init(&o_done[1], 1);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    for (int k = 0; k < 8; ++k) mbar_init(&chain[k], 32);
    mbar_init(q_ready, kSoftmaxThreads);
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
  if (ordered) {
    if (tid < a.batch) {
      const int key = seq[tid] + seq[2 * kOrderMax + tid] - seq[kOrderMax + tid];
      int rank = 0;
      for (int u = 0; u < a.batch; ++u) {
        const int ku = seq[u] + seq[2 * kOrderMax + u] - seq[kOrderMax + u];
        rank += (ku > key) || (ku == key && u < tid);
      }
      seq[3 * kOrderMax + rank] = tid;
    }
    __syncthreads();
    w.b = seq[3 * kOrderMax + blockIdx.z / a.hkv];
    w.n0 = seq[kOrderMax + w.b];
    w.N = seq[2 * kOrderMax + w.b] - w.n0;
    w.L = seq[w.b];
  } else {
    w.b = blockIdx.z / a.hkv;
    w.n0 = __ldg(a.node_offsets + w.b);
    w.N = __ldg(a.node_offsets + w.b + 1) - w.n0;
    w.L = max(0, __ldg(a.prefix_lens + w.b));
  }

  w.rows = w.N * a.group;
  // Split-KV: the prefix of each sequence is cut into at most max_splits
  // ranges of whole 128-key tiles; the splits of one tile form a cluster
  // (grid y), and a member whose sequence has fewer splits only joins the
  // cluster barriers.
  const int chunk = max(BN, ((w.L + a.max_splits - 1) / a.max_splits + BN - 1) / BN * BN);
  w.nsplit = max(1, (w.L + chunk - 1) / chunk);
  if (w.N < 1 || w.mtile * BM >= w.rows) {  // no work for the whole cluster
    if (warp == kMmaWarp) tmem_dealloc(tmem, Ly::kTmemCols);
    return;
  }
  const bool idle = w.split >= w.nsplit;
  w.last_split = (w.split == w.nsplit - 1);
  w.k_begin = w.split * chunk;
  w.k_end = min(w.L, w.k_begin + chunk);
  w.n_prefix_tiles = idle ? 0 : (w.k_end - w.k_begin + BN - 1) / BN;
  w.n_node_tiles = w.last_split ? (w.N + BN - 1) / BN : 0;
  w.T = w.n_prefix_tiles + w.n_node_tiles;
  const int node_lo = (w.mtile * BM) / a.group;
  const int g = a.group;
  // the sequence's extent itself is malformed: nothing to read
  if (w.N > a.max_nodes || w.N > 512 || w.L > a.max_prefix_len || w.n0 < 0 ||
      w.n0 + w.N > a.total_nodes) {
    if (tid == 0) record_status(a.status, w.b, kBadTree);
    const bool rows_addressable = w.n0 >= 0 && w.N <= a.max_nodes && w.n0 + w.N <= a.total_nodes;
    // every CTA of the cluster takes this branch; split 0 writes the zeros
    if (w.split == 0 && rows_addressable && warp < 4) zero_rows<D>(a, w, tid);
    if (warp == kMmaWarp) tmem_dealloc(tmem, Ly::kTmemCols);
    return;
  }
  const uint32_t tmem_o = tmem + 256;   // O accumulator at columns 256 .. 256+D-1
  const uint32_t tmem_p = tmem + 384;   // P at columns 384 .. 447
  const uint32_t tmem_q = tmem + 448;   // Q tile (A operand of Q.K^T)
  volatile int* abort_flag = &misc->abort;

  if (idle) {
    // a cluster member without keys: straight to the cluster barriers
  } else if (warp == kTmaWarp) {
    // ---------------------------------------------------------- TMA producer
    // K and V stream through separate rings: a K slot is free again as soon
    // as S = Q K^T has read it, a V slot once P.V has, so K runs ahead of V.
    // The whole warp issues a tile: lane 0 arms the slot's barrier, then lane
    // u issues box u: page u of a prefix tile (one 5-D box per 16-token page,
    // 8 per tile) or the u-th group of 8 nodes of a node tile (16 per tile).
    if (lane == 0) {
      prefetch_tmap(&maps.k_pool);
      prefetch_tmap(&maps.v_pool);
      prefetch_tmap(&maps.k_nodes);
      prefetch_tmap(&maps.v_nodes);
    }
    constexpr int kPages = BN / 16;
    constexpr int kPastEnd = INT_MIN;                 // page past the prefix end -> zeros
    const bool prefix_lane = lane < kPages;
    const int pool_pages = a.num_blocks * a.hkv;
    const int32_t* btab = a.block_table + static_cast<size_t>(w.b) * a.max_blocks_per_seq;
    auto fetch_block = [&](int t) -> int {
      const int lp = (w.k_begin + t * BN) / 16 + lane;
      return (prefix_lane && t < w.n_prefix_tiles && lp * 16 < w.k_end) ? __ldg(btab + lp) : kPastEnd;
    };
    // issues tile t of tensor kv (0 = K, 1 = V) into its slot
    auto issue = [&](int t, int kv, int blk) {
      const int st = t % kStages;
      uint64_t* bar = kv ? &vfull[st] : &kfull[st];
      if (lane == 0) mbar_arrive_expect_tx(bar, Ly::kTileBytes);
      __syncwarp();
      uint8_t* tile = smem + (kv ? Ly::kVRing : Ly::kKRing) + st * Ly::kTileBytes;
      if (t < w.n_prefix_tiles) {
        if (prefix_lane) {
          int page = pool_pages;  // out of bounds: zero fill
          if (blk >= 0 && blk < a.num_blocks) {
            page = blk * a.hkv + w.kvh;
          } else if (blk != kPastEnd && kv == 0 && !misc->bad) {  // malformed block id: zeros, reported
            misc->bad = 1;
            record_status(a.status, w.b, kBadTree);
          }
          tma_load_5d(tile + lane * 2 * Ly::kGroupBytes, kv ? &maps.v_pool : &maps.k_pool, bar,
                      0, 0, 0, 0, page);
        }
      } else if (lane < BN / 8) {
        const int node0 = w.n0 + (t - w.n_prefix_tiles) * BN + lane * 8;
        tma_load_4d(tile + lane * Ly::kGroupBytes, kv ? &maps.v_nodes : &maps.k_nodes, bar, 0,
                    node0, 0, w.kvh);
      }
    };
    // The block-table reads run two K tiles ahead of the K copies (a global
    // read under load takes about a microsecond), and the ids of every K
    // tile issued stay in shared memory until its V copy: V(t) is issued
    // before K(t+8) can be (K(t+8) needs S(t+5), hence the softmax of tile
    // t+3, which waits for P(t+1).V and so for V(t)).
    int* blk_ring = reinterpret_cast<int*>(smem + Ly::kBlk);  // [tile & 7][page]
    int blk_k = fetch_block(0), blk_k2 = fetch_block(1);
    int tk = 0, tv = 0;
    bool ok = true;
    unsigned long long t_idle = 0;
    while (tv < w.T) {
      bool progressed = false;
      if (tk < w.T) {
        int ready = lane == 0 ? mbar_test_wait(&kempty[tk % kStages], ((tk / kStages) & 1) ^ 1) : 0;
        if (__shfl_sync(0xffffffffu, ready, 0)) {
          if (prefix_lane) blk_ring[(tk & 7) * 8 + lane] = blk_k;
          issue(tk, 0, blk_k);
          ++tk;
          blk_k = blk_k2;
          blk_k2 = fetch_block(tk + 1);
          progressed = true;
        }
      }
      if (tv < tk) {
        int ready = lane == 0 ? mbar_test_wait(&vempty[tv % kStages], ((tv / kStages) & 1) ^ 1) : 0;
        if (__shfl_sync(0xffffffffu, ready, 0)) {
          issue(tv, 1, prefix_lane ? blk_ring[(tv & 7) * 8 + lane] : kPastEnd);
          ++tv;
          progressed = true;
        }
      }
      int stop = 0;
      if (lane == 0) {
        if (progressed) {
          t_idle = 0;
        } else if (t_idle == 0) {
          t_idle = global_ns();
        } else if (global_ns() - t_idle > kWaitLimitNs || misc->abort) {
          stop = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) {
        ok = false;
        break;
      }
    }
    if (lane == 0) {
      if (!ok) {
        record_status(a.status, w.b, kDeviceTimeout);
        misc->abort = 1;
      }
      // drain: every issued copy has landed before the CTA may exit (at most
      // kStages of each ring can still be in flight)
      for (int t = max(0, tk - kStages); t < tk; ++t)
        mbar_wait(&kfull[t % kStages], (t / kStages) & 1);
      for (int t = max(0, tv - kStages); t < tv; ++t)
        mbar_wait(&vfull[t % kStages], (t / kStages) & 1);
    }
  } else if (warp == kMmaWarp || warp == kPvWarp) {
    // ---------------------------------------------------------- MMA issuers
    // Two threads issue to the tensor core: S = Q K^T from warp 9 and
    // O += P V from warp 10.  Issuing a tcgen05.mma stalls its thread while
    // the tensor pipe is busy, so one thread issuing both would hold P(t).V(t)
    // back behind S(t+1); with two threads each kind goes out as soon as its
    // inputs are ready and the pipe interleaves them.
    if (lane == 0) {
      bool ok = mbar_wait(q_ready, 0, abort_flag);
      tc_fence_after();
      if (warp == kMmaWarp) {
        constexpr uint32_t idesc_s = idesc_bf16(BM, BN, 0);  // M=128, N=128
        // Descriptors are built once; each MMA adds an offset to the
        // start-address field (16-byte units; shared addresses stay < 2^18).
        // K (K-major): 8-row groups at kGroupBytes, halves at +1024.
        const uint64_t dk0 = smem_desc(smem_u32(smem + Ly::kKRing), 16, Ly::kGroupBytes);
        for (int t = 0; ok && t < w.T; ++t) {
          // S(t) = Q K(t)^T into buffer t & 1, once K(t) has landed and the
          // softmax has read S(t-2) out of that buffer
          ok = mbar_wait(&kfull[t % kStages], (t / kStages) & 1, abort_flag);
          if (ok && t >= 2) ok = mbar_wait(&s_free[t & 1], ((t - 2) >> 1) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dk = dk0 + static_cast<uint64_t>((t % kStages) * (Ly::kTileBytes >> 4));
          const uint32_t d = tmem + (t & 1) * BN;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // A = Q from TMEM (16 dims = 8 columns per step), B = K from the ring
            const uint32_t boff = ((kk >> 2) * 1024 + (kk & 3) * 32) >> 4;
            mma_bf16_ts(d, tmem_q + kk * 8, dk + boff, idesc_s, kk > 0 ? 1u : 0u);
          }
          mma_commit(&s_full[t & 1]);
          mma_commit(&kempty[t % kStages]);  // the K slot is free once S(t) is done
        }
      } else {
        constexpr uint32_t idesc_o = idesc_bf16(BM, D, 1);
        // V (MN-major): 8-key groups at kGroupBytes, column halves at +1024.
        const uint64_t dv0 = smem_desc(smem_u32(smem + Ly::kVRing), 1024, Ly::kGroupBytes);
        for (int t = 0; ok && t < w.T; ++t) {
          // O += P(t) V(t), once P(t) is in TMEM and V(t) has landed
          ok = mbar_wait(p_full, t & 1, abort_flag);
          if (ok) ok = mbar_wait(&vfull[t % kStages], (t / kStages) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const int st = t % kStages;
          const uint64_t dv = dv0 + static_cast<uint64_t>(st * (Ly::kTileBytes >> 4));
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            // A = P from TMEM: 16 keys = 8 columns of bf16 pairs; B = 2 groups of V
            mma_bf16_ts(tmem_o, tmem_p + kk * 8, dv + ((kk * 2 * Ly::kGroupBytes) >> 4), idesc_o,
                        (t > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&o_done[t & 1]);
          mma_commit(&vempty[st]);
        }
      }
      if (!ok) {
        record_status(a.status, w.b, kDeviceTimeout);
        misc->abort = 1;
      }
      // drain: all MMAs issued by this thread complete before TMEM is freed
      uint64_t* dr = &drain[warp == kMmaWarp ? 0 : 1];
      mma_commit(dr);
      mbar_wait(dr, 0);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- softmax warps
    // Warps 0-7: warp w owns rows 32*(w%4)..+31 (its TMEM lane quarter) in
    // lane hc = w/4, which takes the tiles t = hc, hc + 2, ...; the two
    // warps of a scheduler belong to different lanes.  In the prologue and
    // the epilogue hc selects the half of the Q and O columns a thread moves.
    const int r = (warp & 3) * 32 + lane;  // row of the tile == TMEM lane
    const int hc = warp >> 2;              // softmax lane
    const int sid = hc * 128 + r;          // 0..255
    const int R = w.mtile * BM + r;
    const bool live = R < w.rows;
    float* m_slot = reinterpret_cast<float*>(smem + Ly::kXchg);           // [2][128]
    float2* fin = reinterpret_cast<float2*>(smem + Ly::kXchg + 2 * BM * 4);  // [2 lanes][128]
    // Q tile -> TMEM (one row per lane, bf16 pairs; this thread stores the
    // half hc of its row); padding rows are zero.  The Q loads are issued
    // before the tree loads so that both latencies overlap.
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
      // tree of this sequence into shared memory, validated
      for (int i = sid; i < w.N; i += kSoftmaxThreads) {
        const int p = __ldg(a.parent + w.n0 + i);
        par[i] = p;
        if (!(i == 0 ? p == -1 : (p >= 0 && p < i))) misc->bad = 1;
      }
      if constexpr (kWords == 32) {
        tmem_st32(tmem_q + hc * 32 + lane_off_q(warp), qw);
      } else {
        tmem_st16(tmem_q + hc * 16 + lane_off_q(warp), qw);
      }
      tmem_st_wait();
    }
    tc_fence_before();  // Q is in TMEM before the MMA warp is released
    mbar_arrive(q_ready);
    softmax_group_sync();
    const bool tree_ok = misc->bad == 0;
    if (!tree_ok && sid == 0) record_status(a.status, w.b, kBadTree);
    // ancestor-or-self bitmask of the tile's nodes (node tiles only)
    if (w.last_split && hc == 0) {
      const int i = node_lo + r;
      uint32_t* row = anc + r * kAncStride;
#pragma unroll
      for (int k = 0; k < kMaxAncWords; ++k) row[k] = 0u;
      if (tree_ok && i < w.N) {
        for (int k = i; k >= 0; k = par[k]) row[k >> 5] |= 1u << (k & 31);
      }
    }
    softmax_group_sync();      // ancestor rows are read across threads
    const int i_node = live ? R / g : 0;  // local node of this row
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t* my_anc = anc + (i_node - node_lo) * kAncStride;
    // Online softmax over the tiles of this lane.  The running max m(t)
    // (log2 units) is a chain through all tiles of both lanes: it moves only
    // when a tile's max exceeds it by more than 2^8, and P(t) is taken
    // against m(t).  O always holds sum P V against the latest m (a move
    // rescales it after the previous P.V); each lane keeps its part of the
    // row sum against the reference of its own last tile.
    float m_lane = -INFINITY;  // reference of l_run
    float l_run = 0.0f;
    bool ok = true;
    // The warp of the other lane hands over m(t-1) through chain[1-hc][q]:
    // its k-th completion is tile 2k + (1-hc), and it cannot complete again
    // before this warp has handed back m(t), so the phase parity of tile t-1
    // is ((t-1) >> 1) & 1.  After a failed (timed-out) wait a warp keeps
    // looping and arriving but skips the work.
    uint64_t* chain_in = &chain[(1 - hc) * 4 + (warp & 3)];
    uint64_t* chain_out = &chain[hc * 4 + (warp & 3)];
    for (int t = hc; t < w.T; t += 2) {
      if (ok) {
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[t & 1], (t >> 1) & 1, abort_flag));
        if (!ok) misc->abort = 1;
      }
      // this thread's 128 scores of the tile
      float x[128];
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tmem + (t & 1) * BN + 32 * c + lane_off,
                    *reinterpret_cast<uint32_t(*)[32]>(&x[32 * c]));
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&s_free[t & 1]);  // S(t+2) may overwrite the buffer
      } else {
#pragma unroll
        for (int c = 0; c < 128; ++c) x[c] = 0.0f;
      }
      // mask (scores stay unscaled; the scale is folded into the exponent)
      int valid_keys = BN;
      if (t < w.n_prefix_tiles) {
        valid_keys = min(BN, w.k_end - (w.k_begin + t * BN));
        if (valid_keys < BN) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= valid_keys) x[c] = -INFINITY;
        }
      } else {
        const int j0 = (t - w.n_prefix_tiles) * BN;
        // only ancestors-or-self of this node carry a bit, all of them < N,
        // so node columns past the tree are masked as well
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t b = live ? my_anc[(j0 >> 5) + k] : 0u;
#pragma unroll
          for (int c = 0; c < 32; ++c) x[32 * k + c] = (b & (1u << c)) ? x[32 * k + c] : -INFINITY;
        }
      }
      // max of the 128 scores: eight running three-input maxima over the
      // columns j, j+8, ..., j+120 (few live temporaries next to x)
      float mx[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        mx[j] = fmax3(x[j], x[j + 8], x[j + 16]);
#pragma unroll
        for (int k = 3; k < 15; k += 2) mx[j] = fmax3(mx[j], x[j + 8 * k], x[j + 8 * k + 8]);
        mx[j] = fmaxf(mx[j], x[j + 120]);
      }
      const float smax =
          fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) *
          a.scale_log2;
      // the running max after the previous tile (the other lane's)
      float m_prev = -INFINITY;
      if (t >= 1) {
        if (ok) {
          ok = __all_sync(0xffffffffu, mbar_wait(chain_in, ((t - 1) >> 1) & 1, abort_flag));
          if (!ok) misc->abort = 1;
        }
        m_prev = m_slot[((t - 1) & 1) * BM + r];
      }
      float m_new = m_prev, alpha = 1.0f;
      bool rescale = false;
      if (smax != -INFINITY) {
        if (m_prev == -INFINITY) {
          m_new = smax;
        } else if (smax > m_prev + kRescaleLog2) {
          m_new = smax;
          alpha = exp2f(m_prev - smax);
          rescale = true;
        }
      }
      m_slot[(t & 1) * BM + r] = m_new;
      mbar_arrive(chain_out);  // release: m_slot is visible to the waiter
      if (!ok) continue;  // skip the work, keep the hand-off sequence
      if (m_lane != m_new) {  // this lane's row sum follows the reference
        if (l_run > 0.0f) l_run *= exp2f(m_lane - m_new);
        m_lane = m_new;
      }
      const float mref = (m_new == -INFINITY) ? 0.0f : m_new;
      // P(t) = 2^(s * scale * log2(e) - m) as bf16 pairs (column c holds keys
      // 2c, 2c+1); masked scores are -inf -> 0
      uint32_t pk[64];
      float ls[16];
#pragma unroll
      for (int c8 = 0; c8 < 16; ++c8) {
        float part = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float p0 = ex2_approx(fmaf(x[c8 * 8 + 2 * k], a.scale_log2, -mref));
          const float p1 = ex2_approx(fmaf(x[c8 * 8 + 2 * k + 1], a.scale_log2, -mref));
          pk[c8 * 4 + k] = pack_bf16x2(p0, p1);
          part += p0 + p1;
        }
        ls[c8] = part;
      }
      // P(t-1).V is the last reader of the P buffer and the last
      // accumulation into O
      if (t >= 1) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, abort_flag));
        if (!ok) {
          misc->abort = 1;
          continue;
        }
      }
      tc_fence_after();
      if (__any_sync(0xffffffffu, rescale)) {  // O holds P(0..t-1).V against m_prev
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tmem_o + c0 + lane_off, o);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tmem_st32(tmem_o + c0 + lane_off, o);
        }
      }
      tmem_st32(tmem_p + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st32(tmem_p + 32 + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      float lsum = 0.0f;
#pragma unroll
      for (int k = 0; k < 16; ++k) lsum += ls[k];
      l_run += lsum;
      // keys past the prefix end in this tile: clear their V rows (page
      // tails may hold stale data; P is 0 there but 0 * NaN would poison O)
      if (valid_keys < BN) {
        const int st = t % kStages;
        mbar_wait(&vfull[st], (t / kStages) & 1);  // acquire the TMA writes
        uint8_t* vt = smem + Ly::kVRing + st * Ly::kTileBytes;
        for (int idx = r; idx < (BN - valid_keys) * Ly::kHalves; idx += BM) {
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
      mbar_arrive(p_full);
    }
    // the row sum: both lanes' parts against the final running max
    fin[hc * BM + r] = make_float2(m_lane, l_run);
    softmax_group_sync();
    const float2 f0 = fin[r], f1 = fin[BM + r];
    const float m_run = fmaxf(f0.x, f1.x);  // the chain only grows: the final max
    float l_row = 0.0f;
    if (f0.y > 0.0f) l_row += f0.y * exp2f(f0.x - m_run);
    if (f1.y > 0.0f) l_row += f1.y * exp2f(f1.x - m_run);
    if (!ok) {
      record_status(a.status, w.b, kDeviceTimeout);
      misc->abort = 1;
    } else if (w.T > 0 && __all_sync(0xffffffffu, mbar_wait(&o_done[(w.T - 1) & 1],
                                                            ((w.T - 1) >> 1) & 1, abort_flag))) {
      tc_fence_after();
      // ------------------------------------------------------------ epilogue
      const bool final_out = (w.nsplit == 1);
      const float inv_l = (l_row > 0.0f) ? 1.0f / l_row : 0.0f;
      using Pt = Partial<D>;
      float* part_o = reinterpret_cast<float*>(smem + Ly::kKRing + Pt::kO) + r * Pt::kStride;
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
          float4* dst = reinterpret_cast<float4*>(part_o + c0);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                 __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]));
        }
      }
      if (live && !final_out && hc == 0)
        reinterpret_cast<float2*>(smem + Ly::kKRing + Pt::kMl)[r] = make_float2(m_run, l_row);
    } else if (w.T > 0) {
      record_status(a.status, w.b, kDeviceTimeout);
      misc->abort = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (a.max_splits > 1) {
    // launched as clusters of max_splits CTAs: merge this tile's splits
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();  // every split's partial is in its shared memory
    if (w.nsplit > 1 && !idle && warp < kSoftmaxThreads / 32)
      merge_rows<D>(a, w, smem + Ly::kKRing, &misc->bad, tid,
                    static_cast<int>(cluster.block_rank()));
    cluster.sync();  // no CTA leaves while another may still read its shared memory
  }
  // a malformed tree or block id: the only writer of these rows writes zeros
  // (each row by the thread that wrote it in the epilogue, so zeros win)
  if (misc->bad && w.nsplit == 1 && warp < 4) zero_rows<D>(a, w, tid);
  if (warp == kMmaWarp) tmem_dealloc(tmem, Ly::kTmemCols);
}

}  // namespace

size_t tree_attention_smem_bytes(int head_dim) {
  return head_dim == 64 ? Layout<64>::kAlloc : Layout<128>::kAlloc;
}

int launch_tree_attention(const AttnArgs& a, const AttnMaps& maps, cudaStream_t stream) {
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
  if (a.max_splits < 1 || a.max_splits > 8) return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.mtiles_max, a.max_splits, a.batch * a.hkv);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  // the splits of one tile (grid y) run as one cluster
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = a.max_splits;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.max_splits > 1 ? 1 : 0;
  cudaError_t e;
  if (a.head_dim == 128) {
    cfg.dynamicSmemBytes = Layout<128>::kAlloc;
    e = cudaLaunchKernelEx(&cfg, tree_attn_kernel<128>, a, maps);
  } else {
    cfg.dynamicSmemBytes = Layout<64>::kAlloc;
    e = cudaLaunchKernelEx(&cfg, tree_attn_kernel<64>, a, maps);
  }
  return e == cudaSuccess ? 0 : -1;
}

}  // namespace tv
