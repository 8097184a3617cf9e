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
// GB300 design.
//
// Rows.  The packed query rows of one (sequence, KV head) are R = node * g +
// head-in-group, so every tree node and every query head of a GQA group share
// each K/V tile.  A unit is 256 consecutive rows (two 128-row m-tiles, an
// "m-tile pair") of one (sequence, KV head); its keys are the prefix (128-key
// tiles) followed by the tree nodes (128-node tiles).
//
// Work.  The grid is persistent: at most one CTA per SM.  The key tiles of all
// units are laid out in one line, ordered (sequence, KV head, layer, key
// tile), where a layer holds `lanes` consecutive m-tile pairs of a (sequence,
// KV head).  The line is cut into `vctas` contiguous ranges of equal length,
// one per virtual CTA of `lanes` CTAs; CTA lane i of a virtual CTA computes
// m-tile pair layer * lanes + i of every (sequence, KV head, layer) in its
// range.  So every CTA gets the same number of tiles, and the CTAs that read
// the same K/V tiles (the m-tile pairs of one KV head) walk them at the same
// time, which keeps the repeated reads in L2.  A range boundary inside a unit
// splits it into pieces: each piece leaves its unnormalised O and (m, l) in a
// workspace slot, and the last piece to finish (an arrival counter per unit)
// merges the slots in a fixed order, so results do not depend on timing.
//
// One CTA has 320 threads (384 for E4M3 inputs):
//   warp 8  (TMA)      loads K and V tiles into two shared-memory rings: one 5-D
//                      box per 16-token page through the block table (eight
//                      pages per tile and tensor), or 16 boxes of 8 tree nodes;
//                      pages past the sequence load as zeros (out of bounds).
//   warp 9  (MMA)      one thread issues tcgen05.mma for both m-tiles h:
//                      S_h = Q_h K^T into TMEM (Q_h and K from shared memory),
//                      O_h += P_h V with P_h read from TMEM, in the order
//                      PV_0(t), S_0(t+1), PV_1(t), S_1(t+1).  P_h(t) is written
//                      over the columns of S_h(t); the tensor pipe runs the
//                      MMAs of one thread in order, so S_h(t+1) overwrites them
//                      only after PV_h(t) has read them.  While one m-tile's
//                      softmax runs, the tensor pipe works on the other's.
//   warps 0-3, 4-7     the softmax of m-tile 0 and of m-tile 1, one thread per
//                      row: tcgen05.ld of S, the tree mask from a per-row
//                      ancestor bitmask, the row max, fp32 online softmax in
//                      base 2 against a running max that moves only when it
//                      grows by more than 2^8 (O is then rescaled in TMEM), and
//                      P as 16-bit pairs into TMEM; the row sum adds the rounded
//                      P, so O / l weights V exactly as the P V product did.
//                      They also load Q (cp.async, in the 128-byte swizzled
//                      layout the MMA reads), build the ancestor masks and
//                      write or merge the results.
//   warps 10-11        (E4M3 inputs) convert V tiles to fp16 with their row
//                      scales.
// TMEM (512 columns): S_0/P_0 at 0, S_1/P_1 at 128, O_0 at 256, O_1 at 256+D.
// Every wait on an mbarrier is bounded; on expiry the CTA reports
// TV_ERR_DEVICE_TIMEOUT for its sequence, drains its copies and returns.
#include <climits>

#include "tv_device.cuh"
#include "tv_launch.h"

namespace tv {
namespace {

constexpr int BM = 128;               // rows of one m-tile
constexpr int BN = 128;               // keys per tile
constexpr int kUnitRows = 2 * BM;     // rows of one m-tile pair
constexpr int kSoftmaxThreads = 256;  // warps 0-7: two groups of four warps
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;           // issues every MMA; owns the TMEM allocation
constexpr int kConvWarp = 10;         // E4M3 inputs: warps 10-11 convert V tiles to fp16
constexpr int kConvThreads = 64;
constexpr int kThreads = 320;
constexpr int kThreadsF8 = 384;       // (registers are allocated for 12 warps either way)
constexpr int kMaxNodes = 512;
constexpr int kMaxAncWords = kMaxNodes / 32;
constexpr int kAncStride = kMaxAncWords + 1;  // odd word stride: rows of a warp hit distinct banks
constexpr float kRescaleLog2 = 8.0f;
constexpr int kMaxPieces = 32;        // pieces per scheduling round
constexpr int kSclSlots = 8;          // E4M3: scale slots (tile tau in slot tau % 8)

// Named barriers (0 is __syncthreads): one per softmax group, both groups.
constexpr int kBarGroup0 = 1;         // group h uses kBarGroup0 + h
constexpr int kBarPair = 3;

// A piece: the key tiles [t0, t1) of one unit that this CTA computes.
struct Piece {
  int b, kvh, mp;   // sequence, KV head, m-tile pair
  int t0, t1;       // key tiles of the unit
  int P;            // prefix tiles of the sequence (node tiles follow)
  int L, n0, N;     // prefix length, first node, nodes of the sequence
  int rows;         // packed rows of the unit (1 .. 256)
  int nm;           // m-tiles with rows (1 or 2)
  int slot;         // partial-result slot, -1 when the piece is the whole unit
  int cnt;          // arrival counter of a split unit
  int npieces;      // pieces of a split unit
  int vfirst;       // virtual CTA of the unit's first piece
  int pad;
};

// Shared memory of one CTA.  bf16 inputs: K and V tiles of 128 keys x D bf16
// in 2-stage rings.  E4M3 inputs (F8, D = 128): K and raw V tiles of 128 keys
// x 128 one-byte codes (a K ring of 3, a raw V ring of 3), two converted fp16
// V tiles, and 8 slots of per-key scales (K scales, V scales).
template <int D, bool F8>
struct Layout {
  static_assert(!F8 || D == 128, "E4M3 inputs need D = 128");
  static constexpr int kHalves = D / 64;               // 64-column halves of a 16-bit row
  static constexpr int kStages = F8 ? 3 : (D == 128 ? 2 : 4);  // K ring depth
  static constexpr int kVStages = F8 ? 3 : kStages;    // V (raw) ring depth
  static constexpr int kGroupBytes = kHalves * 1024;   // 8 rows of a 16-bit tile
  static constexpr int kTileBytes = BN * D * 2;        // a 16-bit (bf16 or fp16) K or V tile
  static constexpr int kKTileBytes = F8 ? BN * D : kTileBytes;  // a K or raw V tile as loaded
  static constexpr int kQBytes = F8 ? BM * D : BM * D * 2;     // Q of one m-tile
  static constexpr int kQ = 0;                         // Q_0, Q_1
  static constexpr int kKRing = kQ + 2 * kQBytes;
  static constexpr int kVRing = kKRing + kStages * kKTileBytes;
  static constexpr int kV16 = kVRing + kVStages * kKTileBytes;  // F8: converted V, 2 slots
  static constexpr int kV16Bytes = F8 ? 2 * kTileBytes : 0;
  static constexpr int kScl = kV16 + kV16Bytes;        // F8: [8][2][128] floats
  static constexpr int kSclBytes = F8 ? kSclSlots * 2 * BN * 4 : 0;
  static constexpr int kAnc = kScl + kSclBytes;        // [2][128][kAncStride] words
  static constexpr int kAncBytes = 2 * BM * kAncStride * 4;
  static constexpr int kParent = kAnc + kAncBytes;     // [2][512]
  static constexpr int kParentBytes = 2 * kMaxNodes * 4;
  static constexpr int kPieces = kParent + kParentBytes;
  static constexpr int kPiecesBytes = kMaxPieces * static_cast<int>(sizeof(Piece));
  static constexpr int kScan = kPieces + kPiecesBytes; // 8 warp sums
  static constexpr int kScanBytes = 128;
  // block ids of the pages of the last 8 K tiles issued (8 per tile), reused
  // by the V copies (and, for E4M3 inputs, the V conversion) of the same tiles
  static constexpr int kBlk = kScan + kScanBytes;
  static constexpr int kBlkBytes = 8 * 8 * 4;
  static constexpr int kBar = kBlk + kBlkBytes;
  // kfull[S], kempty[S], vfull[VS], vempty[VS], s_full[2], p_full[2],
  // o_done[2], q_full[2], drain, v16full[2], v16empty[2], sfull[8]
  static constexpr int kNumBars = 2 * kStages + 2 * kVStages + 13 + kSclSlots;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kMiscBytes = 256;
  static constexpr int kTotal = kMisc + kMiscBytes;
  static constexpr int kAlloc = kTotal + 1024;  // slack for 1024-byte alignment
  static constexpr int kTmemCols = 512;
  static_assert(kAlloc <= 232448, "shared memory per CTA");
};

struct Misc {
  uint32_t tmem_base;
  int abort;
  int npieces;                // pieces of this round
  int more;                   // another round follows
  int merge;                  // this CTA merges the current split unit
  int zero_needed;            // a malformed sequence's rows are zeroed by this CTA
  int tree_bad[2];            // per group: the tree of its current piece is malformed
  int piece_bad[kMaxPieces];  // a block id of the piece was out of range
};
static_assert(sizeof(Misc) <= Layout<128, true>::kMiscBytes, "Misc fits its area");

// Partial-result slot: unnormalised O (fp32) as float4 [D/4][256 rows], so
// that the lanes of a warp (consecutive rows) store and load consecutive 16
// bytes; (m, l) per row; a flag.
template <int D>
struct Slot {
  static constexpr size_t kO = 0;
  static constexpr size_t kMl = static_cast<size_t>(kUnitRows) * D * 4;
  static constexpr size_t kFlag = kMl + kUnitRows * 8;
  static constexpr size_t kBytes = kFlag + 256;
};

__device__ __forceinline__ uint32_t lane_off_q(int warp) {
  return static_cast<uint32_t>((warp & 3) * 32) << 16;
}

// max of three (NaN operands are ignored, as in fmaxf)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void record_status(int32_t* status, int b, int code) {
  atomicMax(status + b, code);
}

// ---------------------------------------------------------------- schedule
struct SeqInfo {
  int L, n0, N;
  int P, T;          // prefix tiles; key tiles of a unit (prefix + node tiles)
  int mpairs;        // m-tile pairs (units per KV head)
  int layers;        // ceil(mpairs / lanes)
  int valid;         // extent well formed
  int W;             // tiles of the sequence on the line (the host bounds the
                     // whole line below 2^31)
};

__device__ __forceinline__ SeqInfo seq_info(const AttnArgs& a, int b) {
  SeqInfo s;
  s.L = max(0, __ldg(a.prefix_lens + b));
  s.n0 = __ldg(a.node_offsets + b);
  s.N = __ldg(a.node_offsets + b + 1) - s.n0;
  s.valid = s.N >= 1 && s.N <= a.max_nodes && s.N <= kMaxNodes && s.n0 >= 0 &&
            s.n0 + s.N <= a.total_nodes && s.L <= a.max_prefix_len;
  s.P = (s.L + BN - 1) / BN;
  s.T = s.P + (s.N + BN - 1) / BN;
  s.mpairs = s.valid ? (s.N * a.group + kUnitRows - 1) / kUnitRows : 0;
  s.layers = (s.mpairs + a.lanes - 1) / a.lanes;
  s.W = s.valid ? a.hkv * s.layers * s.T : 0;
  return s;
}

// Exclusive scan over the 256 softmax threads; *total = the sum.
__device__ __forceinline__ int scan256(int v, int* scratch, int sid, int* total) {
  const int lane = sid & 31, w = sid >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[w] = x;
  named_sync(kBarPair, kSoftmaxThreads);
  int before = 0, all = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int s = scratch[k];
    if (k < w) before += s;
    all += s;
  }
  named_sync(kBarPair, kSoftmaxThreads);  // scratch may be reused
  *total = all;
  return before + x - v;
}

// Range boundaries of the V virtual CTAs on a line of W tiles: virtual CTA v
// takes [start(v), start(v+1)) with start(v) = floor(v W / V), computed as
// v q + floor(v r / V) with W = q V + r.  floor(v r / V) (v r <= V^2 < 2^24)
// comes from the fp32 product with 1/V, within one of the quotient, and one
// exact integer correction: no division on the schedule's critical path.
struct Line {
  int W, V, q, r;
  float rV;  // 1 / V
  __device__ __forceinline__ int start(int v) const {
    const int n = v * r;
    int k = static_cast<int>(static_cast<float>(n) * rV);
    if (k * V > n) {
      --k;
    } else if ((k + 1) * V <= n) {
      ++k;
    }
    return v * q + k;
  }
  float VW;  // V / W
  // the virtual CTA whose range holds position p (0 <= p < W): the fp32
  // estimate p V / W is within two of it; exact integer steps finish it
  __device__ __forceinline__ int owner(int p) const {
    int o = min(V - 1, max(0, static_cast<int>(static_cast<float>(p) * VW)));
#pragma unroll 1
    for (int k = 0; k < 4 && o > 0 && start(o) > p; ++k) --o;
#pragma unroll 1
    for (int k = 0; k < 4 && o + 1 < V && start(o + 1) <= p; ++k) ++o;
    return o;
  }
};

// Builds this CTA's pieces of scheduling round `round` into shared memory
// (run by the 256 softmax threads).  In round 0 it also zeroes the output of
// sequences whose extent is malformed (every row it can address) and records
// their status.
template <int D, bool F8>
__device__ void build_schedule(const AttnArgs& a, uint8_t* smem, int round, int sid) {
  using Ly = Layout<D, F8>;
  Misc* misc = reinterpret_cast<Misc*>(smem + Ly::kMisc);
  Piece* pieces = reinterpret_cast<Piece*>(smem + Ly::kPieces);
  int* scratch = reinterpret_cast<int*>(smem + Ly::kScan);
  const size_t out_elem = a.out_fp32 ? 4 : 2;
  // the length of the line; malformed sequences of this CTA (b mod grid).  A
  // batch of at most 256 is read once and kept in registers for the second
  // pass.
  const bool one_chunk = a.batch <= kSoftmaxThreads;
  SeqInfo kept;
  kept.W = 0;
  kept.T = 1;
  kept.layers = 1;
  int W = 0;
  for (int base = 0; base < a.batch; base += kSoftmaxThreads) {
    const int b = base + sid;
    int w = 0;
    if (b < a.batch) {
      const SeqInfo s = seq_info(a, b);
      w = s.W;
      if (one_chunk) kept = s;
      if (round == 0 && !s.valid && s.N >= 1 && b % gridDim.x == blockIdx.x) {
        record_status(a.status, b, kBadTree);
        misc->zero_needed = 1;
      }
    }
    int tot;
    scan256(w, scratch, sid, &tot);
    W += tot;
  }
  if (round == 0 && misc->zero_needed) {
    // the rows of a malformed sequence that can be addressed get zeros
    for (int b = blockIdx.x; b < a.batch; b += gridDim.x) {
      const SeqInfo s = seq_info(a, b);
      if (s.valid || s.N < 1 || s.n0 < 0 || s.n0 + s.N > a.total_nodes) continue;
      const size_t n = static_cast<size_t>(s.N) * a.hq * D * out_elem / 16;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) +
                                            static_cast<size_t>(s.n0) * a.hq * D * out_elem);
      for (size_t k = sid; k < n; k += kSoftmaxThreads) dst[k] = make_uint4(0, 0, 0, 0);
    }
  }
  const int lanes = a.lanes;
  const int v = static_cast<int>(blockIdx.x) / lanes, li = static_cast<int>(blockIdx.x) % lanes;
  Line line;
  line.W = W;
  line.V = max(1, min(a.vctas, W / max(1, a.min_tiles)));
  line.q = W / line.V;
  line.r = W % line.V;
  line.rV = 1.0f / static_cast<float>(line.V);
  line.VW = W > 0 ? static_cast<float>(line.V) / static_cast<float>(W) : 0.0f;
  const int V = line.V;
  int count = 0;  // pieces of this CTA before the current chunk (all rounds)
  if (W > 0 && v < V) {
    const int s_v = line.start(v), e_v = line.start(v + 1);
    int cum = 0;
    for (int base = 0; base < a.batch; base += kSoftmaxThreads) {
      const int b = base + sid;
      SeqInfo s = kept;
      if (!one_chunk) {
        s.W = 0;
        s.T = 1;
        s.layers = 1;
        if (b < a.batch) s = seq_info(a, b);
      }
      int tot;
      const int c0 = cum + scan256(s.W, scratch, sid, &tot);
      // the units of b that meet [s_v, e_v), in line order; the unit of a
      // lane past the sequence's m-tile pairs is idle and skipped
      int mine = 0;
      int lo = 0, hi = 0;
      if (s.W > 0) {
        lo = max(s_v, c0) - c0;
        hi = min(e_v, c0 + s.W) - c0;
        if (lo < hi)
          for (int ui = lo / s.T; ui <= (hi - 1) / s.T; ++ui)
            if ((ui % s.layers) * lanes + li < s.mpairs) ++mine;
      }
      int ptot;
      const int first = count + scan256(mine, scratch, sid, &ptot);
      if (mine > 0) {
        int k = first;
        for (int ui = lo / s.T; ui <= (hi - 1) / s.T; ++ui) {
          const int kvh = ui / s.layers, layer = ui % s.layers;
          const int mp = layer * lanes + li;
          if (mp >= s.mpairs) continue;
          const int slot_i = k - round * kMaxPieces;
          ++k;
          if (slot_i < 0 || slot_i >= kMaxPieces) continue;
          Piece pc;
          const int u0 = c0 + ui * s.T;  // line position of the unit's first tile
          pc.b = b;
          pc.kvh = kvh;
          pc.mp = mp;
          pc.t0 = max(lo, ui * s.T) - ui * s.T;
          pc.t1 = min(hi, (ui + 1) * s.T) - ui * s.T;
          pc.P = s.P;
          pc.L = s.L;
          pc.n0 = s.n0;
          pc.N = s.N;
          pc.rows = min(kUnitRows, s.N * a.group - mp * kUnitRows);
          pc.nm = pc.rows > BM ? 2 : 1;
          if (pc.t0 == 0 && pc.t1 == s.T) {
            pc.slot = -1;
            pc.cnt = -1;
            pc.npieces = 1;
            pc.vfirst = v;
          } else {
            // the first piece (it holds tile 0) uses the CTA's slot 1, every
            // later piece (it starts the CTA's range) slot 0
            const int vf = line.owner(u0), vl = line.owner(u0 + s.T - 1);
            pc.vfirst = vf;
            pc.npieces = vl - vf + 1;
            pc.cnt = vf * lanes + li;
            pc.slot = 2 * static_cast<int>(blockIdx.x) + (pc.t0 > 0 ? 0 : 1);
          }
          pc.pad = 0;
          pieces[slot_i] = pc;
        }
      }
      count += ptot;
      cum += tot;
    }
  }
  if (sid == 0) {
    const int n = count - round * kMaxPieces;
    misc->npieces = max(0, min(kMaxPieces, n));
    misc->more = n > kMaxPieces;
    for (int k = 0; k < kMaxPieces; ++k) misc->piece_bad[k] = 0;
  }
}

// ---------------------------------------------------------------- output
// Writes 32 values of one output row (fp32 or bf16) at column c0.
template <int D>
__device__ __forceinline__ void store_row_chunk(const AttnArgs& a, size_t row, int c0,
                                                const float (&v)[32]) {
  if (a.out_fp32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + row * D + c0);
#pragma unroll
    for (int k = 0; k < 8; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + row * D + c0);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint4 w;
      w.x = pack_bf16x2(v[8 * k + 0], v[8 * k + 1]);
      w.y = pack_bf16x2(v[8 * k + 2], v[8 * k + 3]);
      w.z = pack_bf16x2(v[8 * k + 4], v[8 * k + 5]);
      w.w = pack_bf16x2(v[8 * k + 6], v[8 * k + 7]);
      dst[k] = w;
    }
  }
}

__device__ __forceinline__ int piece_slot(const AttnArgs& a, const Piece& pc, int s) {
  const int cta = (pc.vfirst + s) * a.lanes + static_cast<int>(blockIdx.x) % a.lanes;
  return s == 0 ? 2 * cta + 1 : 2 * cta;
}

// Merges the pieces of a split unit: O = sum_s 2^(m_s - M) O_s /
// sum_s 2^(m_s - M) l_s in piece order.  Thread `ur` of the participants
// takes row ur of the unit.  Piece `own` is this CTA's: its (m, l) and O come
// from registers and TMEM (the values it would have written), the others'
// from their slots; the lanes of a warp read consecutive rows (coalesced).
// Half a row of a piece is loaded at a time (all its loads in flight
// together), so a piece costs two round trips to L2, not one per 32 columns.
template <int D>
__device__ void merge_unit(const AttnArgs& a, const Piece& pc, int ur, size_t out_row, int own,
                           float m_own, float l_own, bool bad_own, uint32_t tmem_o) {
  using Sl = Slot<D>;
  constexpr int kH = D / 2;
  const bool row_ok = ur < pc.rows;
  bool bad = bad_own;
  float M = -INFINITY, l = 0.0f;
  for (int s = 0; s < pc.npieces; ++s) {
    float2 ml = make_float2(m_own, l_own);
    if (s != own) {
      const uint8_t* base = a.slots + static_cast<size_t>(piece_slot(a, pc, s)) * Sl::kBytes;
      bad |= __ldcg(reinterpret_cast<const int*>(base + Sl::kFlag)) != 0;
      ml = row_ok ? __ldcg(reinterpret_cast<const float2*>(base + Sl::kMl) + ur) : make_float2(-INFINITY, 0.0f);
    }
    if (ml.x > M) {
      l = (M == -INFINITY ? 0.0f : l * exp2f(M - ml.x)) + ml.y;
      M = ml.x;
    } else if (ml.x != -INFINITY) {
      l += ml.y * exp2f(ml.x - M);
    }
  }
  const float inv = (l > 0.0f && !bad) ? 1.0f / l : 0.0f;
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += kH) {
    float acc[kH];
#pragma unroll
    for (int k = 0; k < kH; ++k) acc[k] = 0.0f;
#pragma unroll 1
    for (int s = 0; s < pc.npieces; ++s) {
      float v[kH];
      float ms = m_own;
      if (s == own) {
        // every thread of the warp loads TMEM together (a warp-wide load)
#pragma unroll
        for (int c = 0; c < kH; c += 32)
          tmem_ld32(tmem_o + c0 + c, *reinterpret_cast<uint32_t(*)[32]>(&v[c]));
        tmem_ld_wait();
      } else if (row_ok) {
        const uint8_t* base = a.slots + static_cast<size_t>(piece_slot(a, pc, s)) * Sl::kBytes;
        ms = __ldcg(reinterpret_cast<const float2*>(base + Sl::kMl) + ur).x;
        const float4* o4 = reinterpret_cast<const float4*>(base + Sl::kO) + static_cast<size_t>(c0 / 4) * kUnitRows + ur;
#pragma unroll
        for (int k = 0; k < kH / 4; ++k) {
          const float4 x = __ldcg(o4 + k * kUnitRows);
          v[4 * k] = x.x;
          v[4 * k + 1] = x.y;
          v[4 * k + 2] = x.z;
          v[4 * k + 3] = x.w;
        }
      }
      if (!row_ok) continue;
      const float wgt = ms == -INFINITY ? 0.0f : exp2f(ms - M);
#pragma unroll
      for (int k = 0; k < kH; ++k) acc[k] += wgt * v[k];
    }
    if (!row_ok) continue;
#pragma unroll
    for (int k = 0; k < kH; ++k) acc[k] *= inv;
#pragma unroll
    for (int c = 0; c < kH; c += 32)
      store_row_chunk<D>(a, out_row, c0 + c, *reinterpret_cast<const float(*)[32]>(&acc[c]));
  }
}

// ---------------------------------------------------------------- the kernel
// F8: E4M3 inputs (tv_tree_attention_fp8): S = Q K^T on kind::f8f6f4 over the
// codes, the K and Q row scales applied to the scores; the keys' scales come
// with the K tile (4-byte asynchronous copies by the TMA warp); V rows
// converted to fp16 with their scale (one rounding of code x scale) by warps
// 10-11; P in fp16 and P V on kind::f16.
template <int D, bool F8>
__global__ void __launch_bounds__(F8 ? kThreadsF8 : kThreads, 1)
    tree_attn_kernel(const AttnArgs a, const __grid_constant__ AttnMaps maps) {
  using Ly = Layout<D, F8>;
  using Sl = Slot<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int kStages = Ly::kStages;
  constexpr int kVStages = Ly::kVStages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ly::kBar);
  uint64_t* kfull = bars;
  uint64_t* kempty = bars + kStages;
  uint64_t* vfull = bars + 2 * kStages;
  uint64_t* vempty = vfull + kVStages;    // F8: the converters have read the raw V
  uint64_t* s_full = vempty + kVStages;   // [2]: S_h(t) complete (and every MMA before it)
  uint64_t* p_full = s_full + 2;          // [2]: P_h(t) in TMEM (128 arrivals)
  uint64_t* o_done = p_full + 2;          // [2]: the last P_h V of a piece complete
  uint64_t* q_full = o_done + 2;          // [2]: Q_h of a piece in shared memory (128 arrivals)
  uint64_t* drain = q_full + 2;           // every MMA issued so far complete (once per round)
  uint64_t* v16full = drain + 1;          // F8 [2]: V(t) converted and its scales staged (64 arrivals)
  uint64_t* v16empty = v16full + 2;       // F8 [2]: the P V of tile t complete
  uint64_t* sfull = v16empty + 2;         // F8 [8]: the K and V scales of tile t landed (32 arrivals)
  Misc* misc = reinterpret_cast<Misc*>(smem + Ly::kMisc);
  Piece* pieces = reinterpret_cast<Piece*>(smem + Ly::kPieces);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    misc->abort = 0;
    misc->zero_needed = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], F8 ? kConvThreads : 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&v16full[k], kConvThreads);
      mbar_init(&v16empty[k], 1);
    }
    for (int k = 0; k < kSclSlots; ++k) mbar_init(&sfull[k], 32);
    for (int h = 0; h < 2; ++h) {
      mbar_init(&s_full[h], 1);
      mbar_init(&p_full[h], BM);
      mbar_init(&o_done[h], 1);
      mbar_init(&q_full[h], BM);
    }
    mbar_init(drain, 1);
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
  volatile int* abort_flag = &misc->abort;
  const int g = a.group;

  // Progress kept across pieces and rounds (ring slots and barrier phases):
  // g_tile = K/V tiles of every earlier round; in a role, the tiles and the
  // pieces of m-tile h so far (MMA: both m-tiles; softmax: its own).
  int g_tile = 0;
  int tiles_h0 = 0, tiles_h1 = 0, pieces_h0 = 0, pieces_h1 = 0;

  for (int round = 0;; ++round) {
    if (warp < kTmaWarp) build_schedule<D, F8>(a, smem, round, tid);
    __syncthreads();
    const int npieces = misc->npieces;
    const bool more = misc->more != 0;
    if (npieces == 0 || misc->abort) break;

    if (warp == kTmaWarp) {
      // ------------------------------------------------------ TMA producer
      // The whole warp issues a tile: lane 0 arms the slot's barrier, then
      // lane u issues box u: page u of a prefix tile (one 5-D box per
      // 16-token page, 8 per tile) or the u-th group of 8 nodes of a node
      // tile (16 per tile).  K runs ahead of V: a K slot is free again once
      // the last S of its tile is done, a V slot once the last P V is.
      if (round == 0 && lane == 0) {
        prefetch_tmap(&maps.k_pool);
        prefetch_tmap(&maps.v_pool);
        prefetch_tmap(&maps.k_nodes);
        prefetch_tmap(&maps.v_nodes);
      }
      constexpr int kPages = BN / 16;
      constexpr int kPastEnd = INT_MIN;  // page past the prefix end -> zeros
      const bool page_lane = lane < kPages;
      const int pool_pages = a.num_blocks * a.hkv;
      int* blk_ring = reinterpret_cast<int*>(smem + Ly::kBlk);  // [tile & 7][page]
      volatile int* piece_bad = misc->piece_bad;
      auto fetch_block = [&](int p, int t) -> int {
        if (p >= npieces || !page_lane) return kPastEnd;
        const Piece& pc = pieces[p];
        if (t >= pc.P) return kPastEnd;
        const int lp = t * kPages + lane;
        return lp * 16 < pc.L
                   ? __ldg(a.block_table + static_cast<size_t>(pc.b) * a.max_blocks_per_seq + lp)
                   : kPastEnd;
      };
      // issues tile t of piece p (global tile tau) of tensor kv (0 = K, 1 = V)
      auto issue = [&](int p, int t, int tau, int kv, int blk) {
        const Piece& pc = pieces[p];
        const int st = kv ? tau % kVStages : tau % kStages;
        uint64_t* bar = kv ? &vfull[st] : &kfull[st];
        if (lane == 0) mbar_arrive_expect_tx(bar, Ly::kKTileBytes);
        __syncwarp();
        uint8_t* tile = smem + (kv ? Ly::kVRing : Ly::kKRing) + st * Ly::kKTileBytes;
        if constexpr (F8) {
          // E4M3 codes: a page is 16 rows of 128 bytes (2 KB), a node box 8
          if (t < pc.P) {
            if (page_lane) {
              int page = pool_pages;  // out of bounds: zero fill
              if (blk >= 0 && blk < a.num_blocks) {
                page = blk * a.hkv + pc.kvh;
              } else if (blk != kPastEnd && kv == 0) {
                piece_bad[p] = 1;
                record_status(a.status, pc.b, kBadTree);
              }
              tma_load_3d(tile + lane * 2048, kv ? &maps.v_pool : &maps.k_pool, bar, 0, 0, page);
            }
          } else if (lane < BN / 8) {
            const int node0 = pc.n0 + (t - pc.P) * BN + lane * 8;
            tma_load_3d(tile + lane * 1024, kv ? &maps.v_nodes : &maps.k_nodes, bar, 0, node0, pc.kvh);
          }
          if (kv == 0) {
            // the tile's K and V scales into slot tau % 8, lane u the keys
            // 4u .. 4u+3 (page u / 4 of a prefix tile); keys past the prefix
            // end or the tree, and pages with a bad block id, get 0
            float* sc = reinterpret_cast<float*>(smem + Ly::kScl) + (tau % kSclSlots) * 2 * BN;
            const bool prefix = t < pc.P;
            const int valid = prefix ? min(BN, pc.L - t * BN) : min(BN, pc.N - (t - pc.P) * BN);
            const int pblk = __shfl_sync(0xffffffffu, blk, lane >> 2);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int key = 4 * lane + j;
              const float* sk = a.kp_scale;
              const float* sv = a.vp_scale;
              uint32_t n = 0;
              if (key < valid) {
                if (prefix) {
                  if (pblk >= 0 && pblk < a.num_blocks) {
                    const size_t idx = (static_cast<size_t>(pblk) * a.hkv + pc.kvh) * 16 + (key & 15);
                    sk += idx;
                    sv += idx;
                    n = 4;
                  }
                } else {
                  const size_t idx = static_cast<size_t>(pc.n0 + (t - pc.P) * BN + key) * a.hkv + pc.kvh;
                  sk = a.kn_scale + idx;
                  sv = a.vn_scale + idx;
                  n = 4;
                }
              }
              cpa4_zfill(sc + key, sk, n);
              cpa4_zfill(sc + BN + key, sv, n);
            }
            cpa_arrive_noinc(&sfull[tau % kSclSlots]);
          }
          return;
        }
        if (t < pc.P) {
          if (page_lane) {
            int page = pool_pages;  // out of bounds: zero fill
            if (blk >= 0 && blk < a.num_blocks) {
              page = blk * a.hkv + pc.kvh;
            } else if (blk != kPastEnd && kv == 0) {  // malformed block id: zeros, reported
              piece_bad[p] = 1;
              record_status(a.status, pc.b, kBadTree);
            }
            tma_load_5d(tile + lane * 2 * Ly::kGroupBytes, kv ? &maps.v_pool : &maps.k_pool, bar,
                        0, 0, 0, 0, page);
          }
        } else if (lane < BN / 8) {
          const int node0 = pc.n0 + (t - pc.P) * BN + lane * 8;
          tma_load_4d(tile + lane * Ly::kGroupBytes, kv ? &maps.v_nodes : &maps.k_nodes, bar, 0,
                      node0, 0, pc.kvh);
        }
      };
      auto advance = [&](int& p, int& t) {
        if (++t >= pieces[p].t1) {
          ++p;
          if (p < npieces) t = pieces[p].t0;
        }
      };
      int kp = 0, kt = pieces[0].t0, vp = 0, vt = pieces[0].t0;
      int blk_k = fetch_block(kp, kt);  // the block ids of the next K tile, read ahead
      int tk = g_tile, tv = g_tile;
      bool ok = true;
      unsigned long long t_idle = 0;
      while (vp < npieces) {
        bool progressed = false;
        // V before K: the next P V needs its V tile about a tile period
        // before the S after it needs its K tile, and the copies of one warp
        // land in issue order
        if (tv < tk) {
          int ready = lane == 0 ? mbar_test_wait(&vempty[tv % kVStages], ((tv / kVStages) & 1) ^ 1) : 0;
          if (__shfl_sync(0xffffffffu, ready, 0)) {
            issue(vp, vt, tv, 1, page_lane ? blk_ring[(tv & 7) * 8 + lane] : kPastEnd);
            ++tv;
            advance(vp, vt);
            progressed = true;
          }
        }
        if (kp < npieces) {
          // a K tile only when no V copy could be issued now instead
          int ready = 0;
          if (lane == 0) {
            const bool v_free = tv < tk && mbar_test_wait(&vempty[tv % kVStages], ((tv / kVStages) & 1) ^ 1);
            ready = !v_free && mbar_test_wait(&kempty[tk % kStages], ((tk / kStages) & 1) ^ 1);
          }
          if (__shfl_sync(0xffffffffu, ready, 0)) {
            if (page_lane) blk_ring[(tk & 7) * 8 + lane] = blk_k;
            issue(kp, kt, tk, 0, blk_k);
            ++tk;
            advance(kp, kt);
            blk_k = fetch_block(kp, kt);
            progressed = true;
          }
        }
        int stop = 0;
        if (!progressed && lane == 0) {
          // sleep (at most about 200 ns) in try_wait on the slot likely to
          // free first (bf16: the MMAs free K(x) after V(x - 1) and before
          // V(x)) instead of polling, which takes issue slots from the
          // softmax warps of this SM sub-partition
          const bool k_next = kp < npieces;
          const bool v_next = tv < tk;
          if (v_next && (!k_next || tv - kVStages < tk - kStages))
            mbar_try_wait_ns(&vempty[tv % kVStages], ((tv / kVStages) & 1) ^ 1, 200);
          else if (k_next)
            mbar_try_wait_ns(&kempty[tk % kStages], ((tk / kStages) & 1) ^ 1, 200);
        }
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
      if constexpr (F8) cpa_wait_all();  // this lane's scale copies have landed
      if (lane == 0) {
        if (!ok) {
          record_status(a.status, pieces[min(vp, npieces - 1)].b, kDeviceTimeout);
          misc->abort = 1;
        }
        // every issued copy has landed before the ring is reused or the CTA
        // exits (at most kStages of each ring can still be in flight)
        for (int t = max(g_tile, tk - kStages); t < tk; ++t)
          mbar_wait(&kfull[t % kStages], (t / kStages) & 1);
        for (int t = max(g_tile, tv - kVStages); t < tv; ++t)
          mbar_wait(&vfull[t % kVStages], (t / kVStages) & 1);
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // ------------------------------------------------------ MMA issuer
      if (lane == 0) {
        // bf16: S and P V on kind::f16 in bf16.  E4M3: S on kind::f8f6f4 over
        // the codes, P V on kind::f16 in fp16 (P' and the converted V).
        constexpr uint32_t idesc_s = F8 ? idesc_e4m3(BM, BN) : idesc_bf16(BM, BN, 0);
        constexpr uint32_t idesc_o = F8 ? idesc_f16(BM, D, 1) : idesc_bf16(BM, D, 1);
        // Descriptors are built once; each MMA adds an offset to the start
        // address field (16-byte units).  K and Q (K-major): 8-row groups at
        // kGroupBytes (16-bit) or 1024 (8-bit: one 128-byte line per row),
        // 64-column halves at +1024.  V (MN-major): 8-key groups at
        // kGroupBytes, column halves at +1024.
        constexpr uint32_t kKRow8 = F8 ? 1024 : Ly::kGroupBytes;
        const uint64_t dk0 = smem_desc(smem_u32(smem + Ly::kKRing), 16, kKRow8);
        const uint64_t dv0 = smem_desc(smem_u32(smem + (F8 ? Ly::kV16 : Ly::kVRing)), 1024, Ly::kGroupBytes);
        const uint64_t dq0 = smem_desc(smem_u32(smem + Ly::kQ), 16, kKRow8);
        auto issue_s = [&](int h, int t) {  // S_h = Q_h K(t)^T into columns 128 h
          const uint64_t dk = dk0 + static_cast<uint64_t>((t % kStages) * (Ly::kKTileBytes >> 4));
          const uint64_t dq = dq0 + static_cast<uint64_t>(h * (Ly::kQBytes >> 4));
          if constexpr (F8) {
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk)  // 32 codes (bytes) of each row per MMA
              mma_f8_ss(tmem + h * BN, dq + kk * 2, dk + kk * 2, idesc_s, kk > 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = ((kk >> 2) * 1024 + (kk & 3) * 32) >> 4;
              mma_bf16_ss(tmem + h * BN, dq + off, dk + off, idesc_s, kk > 0 ? 1u : 0u);
            }
          }
          mma_commit(&s_full[h]);
        };
        auto issue_pv = [&](int h, int t, bool acc) {  // O_h (+)= P_h V(t)
          const uint64_t dv = dv0 + static_cast<uint64_t>((F8 ? (t & 1) : (t % kStages)) * (Ly::kTileBytes >> 4));
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_bf16_ts(tmem + 256 + h * D, tmem + h * BN + kk * 8,
                        dv + ((kk * 2 * Ly::kGroupBytes) >> 4), idesc_o, (acc || kk > 0) ? 1u : 0u);
        };
        bool ok = true;
        int tau = g_tile;
        for (int p = 0; p < npieces && ok; ++p) {
          const Piece& pc = pieces[p];
          const int nm = pc.nm, T = pc.t1 - pc.t0;
          // the piece's first S of each m-tile, once its Q is loaded and K has landed
          for (int h = 0; h < nm && ok; ++h) {
            ok = mbar_wait(&q_full[h], (h ? pieces_h1 : pieces_h0) & 1, abort_flag);
            if (ok && h == 0) ok = mbar_wait(&kfull[tau % kStages], (tau / kStages) & 1, abort_flag);
            if (!ok) break;
            tc_fence_after();
            issue_s(h, tau);
          }
          if (!ok) break;
          mma_commit(&kempty[tau % kStages]);
          for (int i = 0; i < T && ok; ++i) {
            const int t = tau + i;
            for (int h = 0; h < nm; ++h) {
              ok = mbar_wait(&p_full[h], (h ? tiles_h1 : tiles_h0) & 1, abort_flag);
              if (ok && h == 0) {
                if constexpr (F8) {
                  ok = mbar_wait(&v16full[t & 1], (t >> 1) & 1, abort_flag);  // V(t) in fp16
                } else {
                  ok = mbar_wait(&vfull[t % kStages], (t / kStages) & 1, abort_flag);
                }
              }
              if (!ok) break;
              tc_fence_after();
              issue_pv(h, t, i > 0);
              if (i + 1 < T) {
                if (h == 0) {
                  ok = mbar_wait(&kfull[(t + 1) % kStages], ((t + 1) / kStages) & 1, abort_flag);
                  if (!ok) break;
                  tc_fence_after();
                }
                issue_s(h, t + 1);
              }
              if (h) ++tiles_h1; else ++tiles_h0;
            }
            if (!ok) break;
            if constexpr (F8) {
              mma_commit(&v16empty[t & 1]);  // the converted V slot may take tile t + 2
            } else {
              mma_commit(&vempty[t % kStages]);
            }
            if (i + 1 < T) mma_commit(&kempty[(t + 1) % kStages]);
          }
          if (!ok) break;
          mma_commit(&o_done[0]);
          ++pieces_h0;
          if (nm == 2) {
            mma_commit(&o_done[1]);
            ++pieces_h1;
          }
          tau += T;
        }
        if (!ok) {
          record_status(a.status, pieces[0].b, kDeviceTimeout);
          misc->abort = 1;
        }
        // every MMA issued so far completes before the next round or the exit
        mma_commit(drain);
        mbar_wait(drain, round & 1);
      }
      __syncwarp();
    } else if (F8 && warp >= kConvWarp) {
      // ------------------------------------------------------ V conversion (E4M3)
      // Per tile, once its raw V and its scales have landed and the converted
      // slot is free (the P V of tile t - 2 is complete): each key's row as
      // fp16 of code x V scale (one rounding of the exact product) into
      // converted slot t % 2, in the MN-major layout the P V MMA reads.  Keys
      // past the prefix end or the tree get zero rows (page tails may hold
      // stale codes).
      if constexpr (F8) {
        const int ct = tid - kConvWarp * 32;  // 0 .. 63
        const float* scl = reinterpret_cast<const float*>(smem + Ly::kScl);
        bool ok = true;
        int tau = g_tile;
        for (int p = 0; p < npieces; ++p) {
          const Piece& pc = pieces[p];
          for (int t = pc.t0; t < pc.t1; ++t, ++tau) {
            const int vs = tau % kVStages;
            if (ok) ok = mbar_wait(&vfull[vs], (tau / kVStages) & 1, abort_flag);
            if (ok) ok = mbar_wait(&sfull[tau % kSclSlots], (tau / kSclSlots) & 1, abort_flag);
            if (ok && tau >= 2) ok = mbar_wait(&v16empty[tau & 1], ((tau - 2) >> 1) & 1, abort_flag);
            if (!ok) {
              misc->abort = 1;
            } else {
              const float* sv = scl + (tau % kSclSlots) * 2 * BN + BN;
              const bool prefix = t < pc.P;
              const int valid = prefix ? min(BN, pc.L - t * BN) : min(BN, pc.N - (t - pc.P) * BN);
              // thread ct: the 16 codes of columns 16c .. 16c+15 (c = ct % 8)
              // of keys k0 + 8i, k0 = ct / 8, i = 0 .. 15.  Raw: 128 bytes a
              // key, 16-byte chunk c at chunk c ^ (key % 8); fp16: [8-key
              // group][64-column half][key][128 B], 16-byte chunk q of a
              // line at chunk q ^ (key % 8).  key % 8 = k0 for every i.
              const int k0 = ct >> 3, c = ct & 7;
              const uint8_t* raw = smem + Ly::kVRing + vs * Ly::kKTileBytes + k0 * 128 + ((c ^ k0) << 4);
              uint8_t* v16 = smem + Ly::kV16 + (tau & 1) * Ly::kTileBytes + (c >> 2) * 1024 + k0 * 128;
              const int q0 = (((2 * c) & 7) ^ k0) << 4, q1 = (((2 * c + 1) & 7) ^ k0) << 4;
              auto convert = [&](int i, bool live) {
                uint32_t h[8];
                if (live) {
                  const uint4 w = *reinterpret_cast<const uint4*>(raw + i * 1024);
                  const float s1 = sv[k0 + 8 * i];
                  const float2 s2 = make_float2(s1, s1);
                  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    // codes -> fp16 (exact) -> fp32, times the scale, -> fp16
                    uint32_t c01, c23;
                    e4m3x4_to_f16x2x2(ww[k], c01, c23);
                    const float2 v01 = mul2(unpack_f16x2(c01), s2);
                    const float2 v23 = mul2(unpack_f16x2(c23), s2);
                    h[2 * k] = pack_f16x2(v01.x, v01.y);
                    h[2 * k + 1] = pack_f16x2(v23.x, v23.y);
                  }
                } else {
#pragma unroll
                  for (int k = 0; k < 8; ++k) h[k] = 0u;
                }
                uint8_t* dst = v16 + i * Ly::kGroupBytes;
                *reinterpret_cast<uint4*>(dst + q0) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4*>(dst + q1) = make_uint4(h[4], h[5], h[6], h[7]);
              };
              // a rolled loop: unrolled, the converter's bursts of independent
              // instructions crowd out the softmax warps it shares an SM
              // sub-partition with (measured slower)
              if (valid == BN) {
#pragma unroll 1
                for (int i = 0; i < 16; ++i) convert(i, true);
              } else {
#pragma unroll 1
                for (int i = 0; i < 16; ++i) convert(i, k0 + 8 * i < valid);
              }
              fence_proxy_async_smem();  // generic writes, read by the MMA
            }
            mbar_arrive(&v16full[tau & 1]);
            mbar_arrive(&vempty[vs]);
          }
        }
        if (!ok) record_status(a.status, pieces[0].b, kDeviceTimeout);
      }
    } else {
      // ------------------------------------------------------ softmax groups
      // Warps 4h .. 4h+3 own m-tile h; warp w's rows are its TMEM lane
      // quarter 32 (w % 4) .. +31.
      const int h = warp >> 2;
      const int r = (warp & 3) * 32 + lane;  // row of the m-tile == TMEM lane
      const uint32_t lane_off = lane_off_q(warp);
      const uint32_t tmem_s = tmem + h * BN;
      const uint32_t tmem_o = tmem + 256 + h * D;
      uint32_t* anc = reinterpret_cast<uint32_t*>(smem + Ly::kAnc) + (h * BM + r) * kAncStride;
      int32_t* par = reinterpret_cast<int32_t*>(smem + Ly::kParent) + h * kMaxNodes;
      uint8_t* qh = smem + Ly::kQ + h * Ly::kQBytes;
      volatile int* piece_bad = misc->piece_bad;
      int my_tiles = h ? tiles_h1 : tiles_h0;
      int my_pieces = h ? pieces_h1 : pieces_h0;
      bool ok = true;
      int tau = g_tile;  // global index of the piece's first tile
      for (int p = 0; p < npieces; ++p) {
        const Piece pc = pieces[p];
        const int T = pc.t1 - pc.t0;
        if (h >= pc.nm) {  // this m-tile has no rows in the unit
          tau += T;
          continue;
        }
        const int bar_group = kBarGroup0 + h;
        const int ur = h * BM + r;                 // row of the unit
        const int R = pc.mp * kUnitRows + ur;      // packed row of the (sequence, KV head)
        const bool live = ur < pc.rows;
        const int i_node = live ? R / g : 0;
        const size_t out_row = static_cast<size_t>(pc.n0 + i_node) * a.hq + pc.kvh * g + R % g;
        // Q rows -> shared memory in the 128-byte swizzled K-major layout
        // (the 16-byte chunk c of row r sits at chunk c ^ (r % 8)); rows past
        // the unit are zero.  The buffer is free: the previous piece's last
        // S_h completed before its epilogue.  E4M3: one 128-byte line of
        // codes a row, and the row's scale folded into the exponent factor.
        float cq = a.scale_log2;
        {
          constexpr int kRowBytes = F8 ? D : 2 * D;
          constexpr int kLineBytes = F8 ? 1024 : Ly::kGroupBytes;  // 8 rows
          uint8_t* dst = qh + (r >> 3) * kLineBytes + (r & 7) * 128;
          if (live) {
            const uint8_t* src = reinterpret_cast<const uint8_t*>(a.q) + out_row * kRowBytes;
#pragma unroll
            for (int k = 0; k < kRowBytes / 16; ++k)
              cpa16(dst + (k >> 3) * 1024 + (((k & 7) ^ (r & 7)) << 4), src + k * 16);
            if constexpr (F8) cq = a.scale_log2 * __ldg(a.q_scale + out_row);
          } else {
#pragma unroll
            for (int k = 0; k < kRowBytes / 16; ++k)
              *reinterpret_cast<uint4*>(dst + (k >> 3) * 1024 + k % 8 * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        // the next piece's Q row of this thread (and its tree's parents)
        // into L2, so that its prologue after this piece's epilogue is short
        if (p + 1 < npieces && h < pieces[p + 1].nm) {
          const Piece& nx = pieces[p + 1];
          if (nx.t1 > nx.P && r * 32 < nx.N) prefetch_l2(a.parent + nx.n0 + r * 32);
          const int nr = nx.mp * kUnitRows + ur;
          if (ur < nx.rows) {
            const uint8_t* q = reinterpret_cast<const uint8_t*>(a.q) +
                               (static_cast<size_t>(nx.n0 + nr / g) * a.hq + nx.kvh * g + nr % g) * (F8 ? D : 2 * D);
#pragma unroll
            for (int k = 0; k < (F8 ? D : 2 * D); k += 128) prefetch_l2(q + k);
          }
        }
        // the tree of the sequence (pieces with node tiles): parents, the
        // check 0 <= parent[i] < i (parent[0] = -1), and this row's
        // ancestor-or-self bitmask
        const bool has_nodes = pc.t1 > pc.P;
        bool tree_bad = false;
        if (has_nodes) {
          if (r == 0) misc->tree_bad[h] = 0;
          named_sync(bar_group, BM);
          for (int k = r; k < pc.N; k += BM) {
            const int q = __ldg(a.parent + pc.n0 + k);
            par[k] = q;
            if (!(k == 0 ? q == -1 : (q >= 0 && q < k))) misc->tree_bad[h] = 1;
          }
          named_sync(bar_group, BM);
          tree_bad = misc->tree_bad[h] != 0;
#pragma unroll
          for (int k = 0; k < kMaxAncWords; ++k) anc[k] = 0u;
          if (!tree_bad && live)
            for (int k = i_node; k >= 0; k = par[k]) anc[k >> 5] |= 1u << (k & 31);
          if (tree_bad && r == 0) record_status(a.status, pc.b, kBadTree);
          named_sync(bar_group, BM);  // tree_bad is reset by the next piece
        }
        cpa_wait_all();
        fence_proxy_async_smem();  // generic writes of Q, read by the MMA
        mbar_arrive(&q_full[h]);

        float m_run = -INFINITY;  // running max (log2 units)
        float l_run = 0.0f;       // row sum against m_run
        for (int i = 0; i < T; ++i) {
          const int t = pc.t0 + i;  // tile of the unit
          const int gt = tau + i;   // global tile (ring slot)
          if (ok) {
            ok = __all_sync(0xffffffffu, mbar_wait(&s_full[h], my_tiles & 1, abort_flag));
            if (!ok) misc->abort = 1;
          }
          ++my_tiles;
          if (!ok) {
            mbar_arrive(&p_full[h]);
            continue;
          }
          float x[128];
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tmem_ld32(tmem_s + 32 * c + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&x[32 * c]));
          tmem_ld_wait();
          if constexpr (F8) {
            // the keys' K scales (landed with the K tile, slot gt % 8)
            if (!__all_sync(0xffffffffu, mbar_wait(&sfull[gt % kSclSlots], (gt / kSclSlots) & 1,
                                                   abort_flag))) {
              ok = false;
              misc->abort = 1;
              mbar_arrive(&p_full[h]);
              continue;
            }
            const float* sk = reinterpret_cast<const float*>(smem + Ly::kScl) + (gt % kSclSlots) * 2 * BN;
#pragma unroll
            for (int c = 0; c < 128; c += 4) {
              const float4 s4 = *reinterpret_cast<const float4*>(sk + c);
              const float2 a2 = mul2(make_float2(x[c], x[c + 1]), make_float2(s4.x, s4.y));
              const float2 b2 = mul2(make_float2(x[c + 2], x[c + 3]), make_float2(s4.z, s4.w));
              x[c] = a2.x;
              x[c + 1] = a2.y;
              x[c + 2] = b2.x;
              x[c + 3] = b2.y;
            }
          }
          // mask (scores stay unscaled by the softmax scale, which is folded
          // into the exponent)
          int valid_keys = BN;
          if (t < pc.P) {
            valid_keys = min(BN, pc.L - t * BN);
            if (valid_keys < BN) {
#pragma unroll
              for (int c = 0; c < 128; ++c)
                if (c >= valid_keys) x[c] = -INFINITY;
            }
          } else {
            // only ancestors-or-self of this node carry a bit, all of them
            // < N, so node columns past the tree are masked as well
            const int j0 = (t - pc.P) * BN;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t bits = live ? anc[(j0 >> 5) + k] : 0u;
#pragma unroll
              for (int c = 0; c < 32; ++c) x[32 * k + c] = (bits & (1u << c)) ? x[32 * k + c] : -INFINITY;
            }
          }
          // max of the 128 scores: eight running three-input maxima
          float mx[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            mx[j] = fmax3(x[j], x[j + 8], x[j + 16]);
#pragma unroll
            for (int k = 3; k < 15; k += 2) mx[j] = fmax3(mx[j], x[j + 8 * k], x[j + 8 * k + 8]);
            mx[j] = fmaxf(mx[j], x[j + 120]);
          }
          const float smax =
              fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * cq;
          float alpha = 1.0f;
          bool rescale = false;
          if (smax != -INFINITY) {
            if (m_run == -INFINITY) {
              m_run = smax;
            } else if (smax > m_run + kRescaleLog2) {
              alpha = exp2f(m_run - smax);
              m_run = smax;
              rescale = true;
            }
          }
          const float mref = m_run == -INFINITY ? 0.0f : m_run;
          // P = 2^(s * scale * log2(e) - m) as 16-bit pairs (column c holds
          // keys 2c, 2c+1), written over S_h in four 16-column stores; masked
          // scores are -inf -> 0.  bf16 P for bf16 inputs, fp16 P for E4M3
          // inputs (the converted V is fp16).  The row sum adds the rounded
          // values, so that O / l weights V exactly as the P V product did
          // (with the unrounded sum the rounding of a dominant P biases the
          // output by up to 2^-9 of its V row in bf16).  Exponent arguments
          // and sums take two lanes per instruction.
          const float2 sc2 = make_float2(cq, cq);
          const float2 nm2 = make_float2(-mref, -mref);
          float2 lacc[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const float2 e = fma2(make_float2(x[32 * q4 + 2 * k], x[32 * q4 + 2 * k + 1]), sc2, nm2);
              const float2 pp = make_float2(ex2_approx(e.x), ex2_approx(e.y));
              if constexpr (F8) {
                // P in fp16 (the V scales are in the converted V rows)
                const uint32_t ph = pack_f16x2(pp.x, pp.y);
                pk[k] = ph;
                acc_f16x2(ph, lacc[k & 1]);
              } else {
                const uint32_t pb = pack_bf16x2(pp.x, pp.y);
                pk[k] = pb;
                acc_bf16x2(pb, lacc[k & 1]);
              }
            }
            tmem_st16(tmem_s + 16 * q4 + lane_off, pk);
          }
          const float lsum = (lacc[0].x + lacc[1].x) + (lacc[0].y + lacc[1].y);
          if (__any_sync(0xffffffffu, rescale)) {
            // O holds P(..t-1) V against the old max; P_h(t-1) V is complete
            // (S_h(t), which this thread has seen complete, was issued after it)
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t o[32];
              tmem_ld32(tmem_o + c0 + lane_off, o);
              tmem_ld_wait();
#pragma unroll
              for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
              tmem_st32(tmem_o + c0 + lane_off, o);
            }
            l_run *= alpha;  // (this tile's sum is added below, against the new max)
          }
          l_run += lsum;
          // keys past the prefix end in this tile: clear their V rows (page
          // tails may hold stale data; P is 0 there but 0 * NaN would poison
          // O).  Group 0 does it before P_0(t) V(t), the tile's first reader.
          if (!F8 && h == 0 && valid_keys < BN) {
            const int st = gt % kStages;
            mbar_wait(&vfull[st], (gt / kStages) & 1, abort_flag);  // acquire the TMA writes
            uint8_t* vtile = smem + Ly::kVRing + st * Ly::kTileBytes;
            for (int idx = r; idx < (BN - valid_keys) * Ly::kHalves; idx += BM) {
              const int row = valid_keys + idx / Ly::kHalves, hf = idx % Ly::kHalves;
              uint4* pz = reinterpret_cast<uint4*>(vtile + (row >> 3) * Ly::kGroupBytes + hf * 1024 +
                                                   (row & 7) * 128);
#pragma unroll
              for (int k = 0; k < 8; ++k) pz[k] = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();  // generic writes, read by the MMA
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&p_full[h]);
        }
        // -------------------------------------------------- piece epilogue
        bool done = false;
        if (ok) {
          done = __all_sync(0xffffffffu, mbar_wait(&o_done[h], my_pieces & 1, abort_flag));
          if (!done) {
            ok = false;
            misc->abort = 1;
            record_status(a.status, pc.b, kDeviceTimeout);
          }
        }
        ++my_pieces;
        const bool bad = tree_bad || piece_bad[p] != 0;
        tc_fence_after();
        if (pc.slot < 0) {
          // the whole unit: normalise and write
          const float inv_l = (l_run > 0.0f && !bad) ? 1.0f / l_run : 0.0f;
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = 0u;
            if (done) {
              tmem_ld32(tmem_o + c0 + lane_off, o);
              tmem_ld_wait();
            }
            float v[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(o[k]) * inv_l;
            if (live && done) store_row_chunk<D>(a, out_row, c0, v);
          }
        } else {
          // a piece of a split unit.  Every piece takes a ticket; all but
          // the last write raw O and (m, l) to their slot and then count
          // themselves done; the last waits until the others are done and
          // merges every piece of the unit, its own from TMEM.
          const int nthr = pc.nm * BM;
          const int bar = pc.nm == 2 ? kBarPair : kBarGroup0;
          int* ticket = a.counters + 2 * pc.cnt;
          int* finished = ticket + 1;
          named_sync(bar, nthr);
          if (ur == 0) misc->merge = atomicAdd(ticket, 1) == pc.npieces - 1;
          named_sync(bar, nthr);
          const bool last = misc->merge != 0;
          if (!last) {
            uint8_t* sl = a.slots + static_cast<size_t>(pc.slot) * Sl::kBytes;
            float4* so4 = reinterpret_cast<float4*>(sl + Sl::kO) + ur;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t o[32];
#pragma unroll
              for (int k = 0; k < 32; ++k) o[k] = 0u;
              if (done) {
                tmem_ld32(tmem_o + c0 + lane_off, o);
                tmem_ld_wait();
              }
              if (live) {
#pragma unroll
                for (int k = 0; k < 8; ++k)
                  so4[(c0 / 4 + k) * kUnitRows] =
                      make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                  __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]));
              }
            }
            if (live) reinterpret_cast<float2*>(sl + Sl::kMl)[ur] = make_float2(m_run, l_run);
            if (ur == 0) *reinterpret_cast<int*>(sl + Sl::kFlag) = (bad || !done) ? 1 : 0;
            __threadfence();
            named_sync(bar, nthr);
            if (ur == 0) atomicAdd(finished, 1);
          } else {
            if (ur == 0) {
              // the other pieces hold tickets, so they are running; each
              // only has its slot write left
              const unsigned long long t0 = global_ns();
              while (atomicAdd(finished, 0) < pc.npieces - 1) {
                if (global_ns() - t0 > kWaitLimitNs || *abort_flag) {
                  record_status(a.status, pc.b, kDeviceTimeout);
                  misc->abort = 1;
                  break;
                }
              }
            }
            named_sync(bar, nthr);
            __threadfence();
            merge_unit<D>(a, pc, ur, out_row, static_cast<int>(blockIdx.x) / a.lanes - pc.vfirst,
                          m_run, l_run, bad || !done, tmem_o + lane_off);
          }
          named_sync(bar, nthr);  // misc->merge is rewritten by the next split piece
        }
        tc_fence_before();
        tau += T;
      }
      if (h) {
        tiles_h1 = my_tiles;
        pieces_h1 = my_pieces;
      } else {
        tiles_h0 = my_tiles;
        pieces_h0 = my_pieces;
      }
    }
    // every role has finished the round's pieces (the TMA copies have
    // landed, the MMAs are complete)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    for (int p = 0; p < npieces; ++p) g_tile += pieces[p].t1 - pieces[p].t0;
    __syncthreads();  // the piece list is rebuilt next round
    if (!more || misc->abort) break;
  }
  if (warp == kMmaWarp) tmem_dealloc(tmem, Ly::kTmemCols);
}

}  // namespace

size_t attn_slot_bytes(int head_dim) {
  return head_dim == 64 ? Slot<64>::kBytes : Slot<128>::kBytes;
}

int launch_tree_attention(const AttnArgs& a, const AttnMaps& maps, cudaStream_t stream) {
  static thread_local int attr_set_device = -1;  // the attribute is set once per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_set_device != dev) {
    cudaFuncSetAttribute(tree_attn_kernel<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         Layout<128, false>::kAlloc);
    cudaFuncSetAttribute(tree_attn_kernel<64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         Layout<64, false>::kAlloc);
    cudaFuncSetAttribute(tree_attn_kernel<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         Layout<128, true>::kAlloc);
    attr_set_device = dev;
  }
  const int ctas = a.vctas * a.lanes;
  if (ctas < 1) return -1;
  if (a.fp8 && a.head_dim != 128) return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(a.fp8 ? kThreadsF8 : kThreads, 1, 1);
  cfg.stream = stream;
  cudaError_t e;
  if (a.fp8) {
    cfg.dynamicSmemBytes = Layout<128, true>::kAlloc;
    e = cudaLaunchKernelEx(&cfg, tree_attn_kernel<128, true>, a, maps);
  } else if (a.head_dim == 128) {
    cfg.dynamicSmemBytes = Layout<128, false>::kAlloc;
    e = cudaLaunchKernelEx(&cfg, tree_attn_kernel<128, false>, a, maps);
  } else {
    cfg.dynamicSmemBytes = Layout<64, false>::kAlloc;
    e = cudaLaunchKernelEx(&cfg, tree_attn_kernel<64, false>, a, maps);
  }
  return e == cudaSuccess ? 0 : -1;
}

}  // namespace tv
