// accept_kernel.cu -- the fused accept pass.
//
// Sources (titles abbreviated):
//   [EC]  "端云协同推测解码中草稿模型动态生成与验证并行化：探究树形注意力机制与显存碎片整理联合加速",
//         §2.2.3 batch verification: p_accept = min(1, p_target/p_draft) per
//         node, parallel uniforms -> accept mask, root-first search cut at the
//         first rejection, longest accepted path, all inside GPU kernels with
//         no host round trip.
//   [LLM] "端侧大模型推测解码草稿模型动态剪枝策略：详解基于重要性采样的树形验证并行加速机制",
//         §2.2.1-§2.2.2 importance correction q~ = q 1_R / Z and the ScaleMask
//         step (add log(1/Z) on retained tokens, -inf elsewhere); §7.1 the
//         log-space chain (log w = -LSE of the kept draft mass); §1.2 step 3
//         resampling at the rejection.
//
// Two kernels, one call, no host round trip:
//   accept_rowstats_kernel  (only for logits input or a retained-set mask)
//       nparts CTAs per row of the batch (rows without children exit after
//       finding their tree); CTA k of a row takes every nparts-th 8K-entry
//       chunk, each with all its loads issued at once (128-bit), and keeps
//       per thread a running log-sum-exp (max, sum of exp) of the target
//       logits and/or the retained draft mass in exact 2^-40 fixed point;
//       one partial per CTA.  nparts gives about four CTAs per SM.
//   accept_tree_kernel      one thread-block cluster per tree, launched with
//       programmatic dependent launch so it is resident when the first kernel
//       ends.  Phase 1: every node's p~, q~ from the combined partials (fixed
//       combine order); the tests; warp ballots; each thread walks its node's
//       parent chain over the ballot bits; a block max over (depth, -index)
//       picks the cut node.  Phase 2: the bonus draw over the cut node's row,
//       split across the cluster with each thread holding 32 consecutive
//       entries in registers; exact fixed-point sums are combined in rank
//       order over distributed shared memory and the thread whose range
//       holds t = floor(u0 * S) finds the token.
// The multi-candidate walk (test 2) replaces the parallel tests and the cut:
// from the root, the children of the current node are tried in index order
// against the current target distribution cur (at first p~), the first
// accepted child becomes the current node, and every rejection replaces cur
// by its normalised residual fl32(r / N), r = max(0, fl32(cur - q~)), N the
// fp32 of the exact fixed-point sum of r, computed over the cluster's slices
// of the row (multi-step speculative sampling, SpecInfer, which the pages cite
// among their sources).  The bonus then comes from the last residual, or from
// p~ at a leaf.
// Every decision-carrying sum is an exact integer, so the result does not
// depend on the reduction order.
#include <cooperative_groups.h>

#include "tv_device.cuh"
#include "tv_launch.h"

namespace cg = cooperative_groups;

namespace tv {
namespace {

constexpr int kMaxN = 512;
constexpr int kTreeThreads = 512;
constexpr int kTreeWarps = kTreeThreads / 32;
constexpr int kMaxCluster = 16;        // CTAs per tree (non-portable cluster size)
constexpr int kChunkQuantum = 32 * kTreeWarps;  // a CTA's slice of the cut row: multiple of 512
constexpr int kMinChunk = 2048;        // entries per CTA before another CTA is worth it
// Entries of the cut row per CTA (multiple of kChunkQuantum) for C CTAs.
__host__ __device__ inline int bonus_chunk(int vocab, int C) {
  const int c = (vocab + C - 1) / C;
  return (c + kChunkQuantum - 1) / kChunkQuantum * kChunkQuantum;
}
// the cut row's target and draft chunks (and, for the multi-candidate walk,
// the residual chunk) plus its mask words
__host__ __device__ inline int tree_smem_bytes(int chunk, bool multi) {
  return (multi ? 3 : 2) * chunk * 4 + (chunk / 32) * 4;
}
constexpr int kRowThreads = 256;
constexpr int kRowVec = 8;             // float4 per thread per chunk (logits rows)
constexpr int kChunk = kRowThreads * kRowVec * 4;  // 8192 entries per row chunk (workspace unit)
constexpr float kTwo40 = 1099511627776.0f;
constexpr float kTwoM40 = 9.094947017729282379150390625e-13f;

__device__ __forceinline__ void lse_combine(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  if (m2 > m) {
    s = s * expf(m - m2) + s2;
    m = m2;
  } else {
    s = s + s2 * expf(m2 - m);
  }
}
__device__ __forceinline__ void lse_push(float& m, float& s, float x) {
  if (x == -INFINITY) return;  // contributes exp(-inf) = 0
  if (x > m) {
    s = s * expf(m - x) + 1.0f;
    m = x;
  } else {
    s += expf(x - m);  // NaN x propagates into s
  }
}
// floor(min(r, 32) * 2^40) for r > 0, else 0 (NaN -> 0)
__device__ __forceinline__ unsigned long long fix40(float r) {
  if (!(r > 0.0f)) return 0ull;
  r = fminf(r, 32.0f);
  return __float2ull_rz(__fmul_rn(r, kTwo40));
}
__device__ __forceinline__ float z_from_sum(unsigned long long S) {
  return __fmul_rn(__ull2float_rn(S), kTwoM40);  // exact scaling by 2^-40
}
// floor(u * S) exactly for u in [0,1), S < 2^64
__device__ __forceinline__ unsigned long long scaled_draw(float u, unsigned long long S) {
  if (!(u > 0.0f)) return 0ull;
  const uint32_t b = __float_as_uint(u);
  const uint32_t e = (b >> 23) & 0xFFu;
  const unsigned long long M = e ? ((b & 0x7FFFFFu) | 0x800000u) : (b & 0x7FFFFFu);
  const int sh = e ? 150 - static_cast<int>(e) : 149;  // u = M * 2^-sh, sh >= 24
  const unsigned long long lo = M * S;
  const unsigned long long hi = __umul64hi(M, S);
  if (sh >= 128) return 0ull;
  if (sh >= 64) return hi >> (sh - 64);
  return (lo >> sh) | (hi << (64 - sh));
}

// Does local node j of the tree starting at n0 (N nodes) have a child?
// (children have larger indices).  Block-wide; every thread gets the answer.
__device__ bool block_has_child(const int32_t* parent, int n0, int N, int j) {
  int found = 0;
  for (int i = j + 1 + static_cast<int>(threadIdx.x); i < N; i += blockDim.x)
    if (__ldg(parent + n0 + i) == j) found = 1;
  return __syncthreads_or(found) != 0;
}

// ============================================================ row statistics
// RV float4 per thread per chunk of kRowThreads * RV * 4 entries: 8 (three
// CTAs per SM) for logits rows alone; 4 (six CTAs per SM, more of them in
// flight) when draft rows and a mask are read as well.  nchunk counts chunks
// of that size.
template <int RV>
__global__ void __launch_bounds__(kRowThreads, RV == 8 ? 3 : 6)
    accept_rowstats_kernel(const AcceptArgs a, int nchunk, int nparts, float2* ws_ms,
                           unsigned long long* ws_z) {
  constexpr int kCh = kRowThreads * RV * 4;
  // the per-tree kernel may start now: its prologue (tree loads and checks)
  // overlaps this kernel; it waits for our results in griddepcontrol.wait
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long item = blockIdx.x;
  const int g = static_cast<int>(item / nparts);  // global row
  const int part = static_cast<int>(item % nparts);
  if (g >= a.total_nodes) return;
  // tree of row g (binary search over node_offsets)
  int lo = 0, hi = a.batch;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a.node_offsets + mid) <= g) lo = mid; else hi = mid;
  }
  const int n0 = __ldg(a.node_offsets + lo);
  const int N = min(__ldg(a.node_offsets + lo + 1) - n0, kMaxN);
  const int j = g - n0;
  if (N < 1 || j < 0 || j >= N) return;
  if (!block_has_child(a.parent, n0, N, j)) return;  // nobody reads this row's statistics

  const int V = a.vocab;
  const size_t rowbase = static_cast<size_t>(g) * V;
  const bool vec = (rowbase & 3) == 0;
  const bool logits = a.kind == 1;
  const bool masked = a.mask != nullptr;
  const int W = (V + 31) >> 5;
  const uint32_t* mrow = masked ? a.mask + static_cast<size_t>(g) * W : nullptr;

  // this CTA's chunks c = part, part + nparts, ...: each thread keeps one
  // running (max, sum of exp) and one exact fixed-point sum over all of them
  float m = -INFINITY, s = 0.0f;
  unsigned long long z = 0;
  for (int c = part; c < nchunk; c += nparts) {
    const int v0 = c * kCh, v1 = min(V, v0 + kCh);
    if (vec) {
      float4 tv[RV], dv[RV];
#pragma unroll
      for (int k = 0; k < RV; ++k) {
        const int v = v0 + (k * kRowThreads + threadIdx.x) * 4;
        tv[k] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        dv[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (v + 3 < v1) {
          if (logits) tv[k] = __ldg(reinterpret_cast<const float4*>(a.target + rowbase + v));
          if (masked) dv[k] = __ldg(reinterpret_cast<const float4*>(a.draft + rowbase + v));
        } else {
          float* tp = &tv[k].x;
          float* dp = &dv[k].x;
          for (int e = 0; e < 4 && v + e < v1; ++e) {
            if (logits) tp[e] = __ldg(a.target + rowbase + v + e);
            if (masked) dp[e] = __ldg(a.draft + rowbase + v + e);
          }
        }
      }
      if (logits) {  // the chunk's max first, then independent exponentials
        // as 2^((x - m) log2 e) on the special function unit (relative error
        // about 2^-22 a term: the LSE moves by far less than the 1e-5 that p~
        // is held to; terms below 2^-126 flush to zero)
        float cm = -INFINITY, cs = 0.0f;
#pragma unroll
        for (int k = 0; k < RV; ++k)
          cm = fmaxf(cm, fmaxf(fmaxf(tv[k].x, tv[k].y), fmaxf(tv[k].z, tv[k].w)));
        if (cm != -INFINITY) {
          constexpr float kLog2e = 1.4426950408889634f;
#pragma unroll
          for (int k = 0; k < RV; ++k)
            cs += (ex2_approx((tv[k].x - cm) * kLog2e) + ex2_approx((tv[k].y - cm) * kLog2e)) +
                  (ex2_approx((tv[k].z - cm) * kLog2e) + ex2_approx((tv[k].w - cm) * kLog2e));
        }
        if (cm != cm) cs = cm;  // a NaN logit makes the row NaN
        lse_combine(m, s, cm, cs);
      }
      if (masked) {
#pragma unroll
        for (int k = 0; k < RV; ++k) {
          const int v = v0 + (k * kRowThreads + threadIdx.x) * 4;
          if (v >= v1) continue;
          const uint32_t w = __ldg(mrow + (v >> 5)) >> (v & 31);
          if ((w & 1u) && v < v1) z += fix40(dv[k].x);
          if ((w & 2u) && v + 1 < v1) z += fix40(dv[k].y);
          if ((w & 4u) && v + 2 < v1) z += fix40(dv[k].z);
          if ((w & 8u) && v + 3 < v1) z += fix40(dv[k].w);
        }
      }
    } else {
      for (int e = v0 + threadIdx.x; e < v1; e += kRowThreads) {
        if (logits) lse_push(m, s, __ldg(a.target + rowbase + e));
        if (masked && ((__ldg(mrow + (e >> 5)) >> (e & 31)) & 1u)) z += fix40(__ldg(a.draft + rowbase + e));
      }
    }
  }
  // block reduction
  __shared__ float sm_m[kRowThreads / 32], sm_s[kRowThreads / 32];
  __shared__ unsigned long long sm_z[kRowThreads / 32];
  for (int o = 16; o; o >>= 1) {
    lse_combine(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
    z += __shfl_xor_sync(0xffffffffu, z, o);
  }
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    sm_m[w] = m;
    sm_s[w] = s;
    sm_z[w] = z;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -INFINITY, S = 0.0f;
    unsigned long long Z = 0;
    for (int k = 0; k < kRowThreads / 32; ++k) {
      lse_combine(M, S, sm_m[k], sm_s[k]);
      Z += sm_z[k];
    }
    ws_ms[item] = make_float2(M, S);
    ws_z[item] = Z;
  }
}

// ============================================================ per-tree pass
struct TreeSmem {
  int32_t parent[kMaxN];
  int32_t token[kMaxN];
  float u[kMaxN];
  float lse[kMaxN];  // log-sum-exp of the target logits row of each node with children
  float z[kMaxN];    // retained draft mass Z of each node with children
  uint8_t has_child[kMaxN];
  uint32_t acc_bits[kMaxN / 32];
  float red_f0[kTreeWarps], red_f1[kTreeWarps];
  unsigned long long red_u64[kTreeWarps];
  uint32_t red_u32[kTreeWarps];
  int red_i32[kTreeWarps];
  // cluster exchange slots (read by the other CTAs of the cluster); each is
  // written once per call, so no barrier is needed before a slot is reused
  float x_m, x_s;
  unsigned long long x_u64[2], x_z;
  float x_maxv;
  int x_maxi;
  int bad;
  int cut, cut_len;
  float x_p, x_q;    // multi-candidate walk: the tested child's p~, q~
  int x_next;        // multi-candidate walk: the next child
};

__device__ unsigned long long block_sum_u64(TreeSmem& sm, unsigned long long x) {
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.red_u64[w] = x;
  __syncthreads();
  unsigned long long t = 0;
  for (int i = 0; i < kTreeWarps; ++i) t += sm.red_u64[i];
  return t;
}
__device__ float block_max_f32(TreeSmem& sm, float x) {
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.red_f0[w] = x;
  __syncthreads();
  float t = -INFINITY;
  for (int i = 0; i < kTreeWarps; ++i) t = fmaxf(t, sm.red_f0[i]);
  return t;
}
__device__ float block_sum_f32(TreeSmem& sm, float x) {
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.red_f1[w] = x;
  __syncthreads();
  float t = 0.0f;
  for (int i = 0; i < kTreeWarps; ++i) t += sm.red_f1[i];
  return t;
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}
__device__ uint32_t block_max_u32(TreeSmem& sm, uint32_t x) {
  x = __reduce_max_sync(0xffffffffu, x);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.red_u32[w] = x;
  __syncthreads();
  uint32_t t = 0;
  for (int i = 0; i < kTreeWarps; ++i) t = max(t, sm.red_u32[i]);
  return t;
}
// max value, smallest index among equal maxima (NaN ignored)
__device__ void block_argmax(TreeSmem& sm, float& v, int& idx) {
  for (int o = 16; o; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    if (v2 > v || (v2 == v && i2 < idx)) {
      v = v2;
      idx = i2;
    }
  }
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    sm.red_f0[w] = v;
    sm.red_i32[w] = idx;
  }
  __syncthreads();
  v = -INFINITY;
  idx = 0x7fffffff;
  for (int i = 0; i < kTreeWarps; ++i) {
    if (sm.red_f0[i] > v || (sm.red_f0[i] == v && sm.red_i32[i] < idx)) {
      v = sm.red_f0[i];
      idx = sm.red_i32[i];
    }
  }
}

// Cluster-wide sum of a per-CTA slot, and the part of it held by ranks below
// `rank`: lane c of every warp reads CTA c's slot, so the C reads of
// distributed shared memory are in flight together.
template <typename T>
__device__ __forceinline__ T cluster_sum(cg::cluster_group& cluster, const T* slot, int C, int rank,
                                         T* below) {
  const int lane = threadIdx.x & 31;
  T v = lane < C ? *cluster.map_shared_rank(slot, lane) : T(0);
  T b = lane < rank ? v : T(0);
  for (int o = 16; o; o >>= 1) {
    v += __shfl_xor_sync(0xffffffffu, v, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  if (below) *below = b;
  return v;
}
__device__ __forceinline__ float cluster_max(cg::cluster_group& cluster, const float* slot, int C) {
  const int lane = threadIdx.x & 31;
  float v = lane < C ? *cluster.map_shared_rank(slot, lane) : -INFINITY;
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__global__ void __launch_bounds__(kTreeThreads, 1)
    accept_tree_kernel(const AcceptArgs a, int nparts, const float2* ws_ms,
                       const unsigned long long* ws_z) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.y;
  const int tid = threadIdx.x;
  __shared__ TreeSmem sm;

  const int n0 = a.node_offsets[b];
  const int N = a.node_offsets[b + 1] - n0;
  const int V = a.vocab;
  const int W = (V + 31) >> 5;
  const bool logits = a.kind == 1;
  const bool masked = a.mask != nullptr;
  const bool stats = logits || masked;
  extern __shared__ float4 smem_dyn[];
  float* smem_rows = reinterpret_cast<float*>(smem_dyn);

  // ---------------------------------------------------------------- tree
  if (tid == 0)
    sm.bad = (N < 1 || N > a.max_nodes || N > kMaxN || n0 < 0 || n0 + N > a.total_nodes ||
              (a.gamma && !(a.gamma[b] > 0.0f && a.gamma[b] <= 3.0e38f))) ? 1 : 0;
  __syncthreads();
  if (!sm.bad) {
    for (int i = tid; i < N; i += kTreeThreads) {
      const int p = a.parent[n0 + i];
      const int x = a.tokens[n0 + i];
      sm.parent[i] = p;
      sm.token[i] = x;
      sm.u[i] = a.uniforms[n0 + i];
      sm.has_child[i] = 0;
      const bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i && x >= 0 && x < V);
      if (!ok) sm.bad = 1;
    }
  }
  __syncthreads();
  if (sm.bad) {  // identical decision in every CTA of the cluster
    if (rank == 0) {
      for (int k = tid; k < a.max_nodes; k += kTreeThreads) a.path[(size_t)b * a.max_nodes + k] = -1;
      if (tid == 0) {
        a.accepted_len[b] = -1;
        a.bonus_token[b] = -1;
        a.status[b] = kBadTree;
      }
      if (a.debug_pq && N >= 1 && N <= kMaxN && n0 >= 0 && n0 + N <= a.total_nodes)
        for (int i = tid; i < N; i += kTreeThreads) {
          a.debug_pq[2 * (size_t)(n0 + i)] = 0.0f;
          a.debug_pq[2 * (size_t)(n0 + i) + 1] = 0.0f;
        }
    }
    return;
  }
  for (int i = tid + 1; i < N; i += kTreeThreads) sm.has_child[sm.parent[i]] = 1;
  // The tested entries do not depend on the row statistics: thread i reads
  // node i's target and draft entries (and mask bit) before waiting for them.
  // Everything before the row-statistics kernel in the stream has completed.
  const bool multi = a.test == 2;
  float raw_p = 0.0f, raw_q = 0.0f;
  uint32_t raw_in = 1u;
  if (!multi && tid >= 1 && tid < N) {
    const int j = sm.parent[tid], x = sm.token[tid];
    const size_t row = static_cast<size_t>(n0 + j) * V;
    raw_p = __ldg(a.target + row + x);
    raw_q = __ldg(a.draft + row + x);
    if (masked) raw_in = (__ldg(a.mask + static_cast<size_t>(n0 + j) * W + (x >> 5)) >> (x & 31)) & 1u;
  }
  // the row statistics come from the previous kernel in the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __syncthreads();

  // LSE / Z of local row j (a row with children) from the partials, fixed order
  auto row_lse = [&](int j) -> float {
    float m = -INFINITY, s = 0.0f;
    const float2* p = ws_ms + static_cast<size_t>(n0 + j) * nparts;
    for (int c = 0; c < nparts; ++c) {
      const float2 e = p[c];
      lse_combine(m, s, e.x, e.y);
    }
    return m + logf(s);
  };
  auto row_z = [&](int j) -> float {
    unsigned long long S = 0;
    const unsigned long long* p = ws_z + static_cast<size_t>(n0 + j) * nparts;
    for (int c = 0; c < nparts; ++c) S += p[c];
    return z_from_sum(S);
  };

  // LSE / Z of every row with children, once (thread j: row j)
  if (stats) {
    const int j = tid;  // kTreeThreads == kMaxN
    if (j < N && sm.has_child[j]) {
      if (logits) sm.lse[j] = row_lse(j);
      if (masked) sm.z[j] = row_z(j);
    }
    __syncthreads();
  }

  // p~, q~ of a tested entry of the rows of local node j (a node with
  // children) from its raw target value p, draft value q and mask bit
  auto tilde = [&](int j, float& p, float& q, uint32_t in) {
    if (logits) p = expf(p - sm.lse[j]);
    if (masked) {
      if (in) {
        const float z = sm.z[j];
        p = __fdiv_rn(p, z);
        q = __fdiv_rn(q, z);
      } else {
        p = 0.0f;
        q = 0.0f;
      }
    }
  };
  // the same for token x, read here
  auto node_pq = [&](int j, int x, float& p, float& q) {
    const size_t row = static_cast<size_t>(n0 + j) * V;
    p = __ldg(a.target + row + x);
    q = __ldg(a.draft + row + x);
    const uint32_t in =
        masked ? (__ldg(a.mask + static_cast<size_t>(n0 + j) * W + (x >> 5)) >> (x & 31)) & 1u : 1u;
    tilde(j, p, q, in);
  };
  const float gam = a.gamma ? a.gamma[b] : 1.0f;
  bool m_rejected = false;  // multi-candidate: the final node's children were all rejected

  // ---------------------------------------------------------------- tests
  float my_p = 0.0f, my_q = 0.0f;
  if (!multi) {
    const int i = tid;  // kTreeThreads == kMaxN: one node per thread
    bool acc = false;
    if (i >= 1 && i < N) {
      const int j = sm.parent[i];
      float p = raw_p, q = raw_q;
      tilde(j, p, q, raw_in);
      my_p = p;
      my_q = q;
      const float u = sm.u[i];
      const float g = gam;
      if (a.test == 0) {
        // u < min(1, g * p~ / q~) as fl32(u * q~) < fl32(g * p~)
        acc = __fmul_rn(u, q) < __fmul_rn(g, p);
      } else {
        // log space with a clamp: r = clamp(log p~ - log q~ + log g, -L, L),
        // accept iff u < (r >= 0 ? 1 : exp(r)); p~ = 0 or a NaN ratio rejects
        const float r = (logf(p) - logf(q)) + logf(g);
        if (!(p > 0.0f) || r != r) {
          acc = false;
        } else {
          const float rc = fmaxf(fminf(r, a.log_clamp), -a.log_clamp);
          acc = u < (rc >= 0.0f ? 1.0f : expf(rc));
        }
      }
    }
    const uint32_t bal = __ballot_sync(0xffffffffu, acc);
    if ((tid & 31) == 0) sm.acc_bits[tid >> 5] = bal;
  }
  __syncthreads();
  if (!multi) {
    uint32_t key = 0;
    const int i = tid;
    if (i < N) {
      int k = i, d = 0;
      bool ok = true;
      while (k > 0) {
        if (!((sm.acc_bits[k >> 5] >> (k & 31)) & 1u)) {
          ok = false;
          break;
        }
        k = sm.parent[k];
        ++d;
      }
      if (ok) key = (static_cast<uint32_t>(d) << 16) | (0xFFFFu - static_cast<uint32_t>(i));
    }
    key = block_max_u32(sm, key);
    if (tid == 0) {
      sm.cut = static_cast<int>(0xFFFFu - (key & 0xFFFFu));
      sm.cut_len = static_cast<int>(key >> 16);
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- rows
  // A row's chunk of this CTA, [lo, hi), goes to shared memory with
  // cp.async; every pass then reads it coalesced.  The exact find walks
  // contiguous 1024-entry warp spans in index order with warp scans.
  const int chunk = bonus_chunk(V, C);
  const int wspan = chunk / kTreeWarps;  // contiguous entries per warp (multiple of 32)
  float* tbuf = smem_rows;               // p~ (or the current target of the walk)
  float* dbuf = smem_rows + chunk;       // q~
  float* rbuf = smem_rows + 2 * chunk;   // the walk's last residual (multi only)
  uint32_t* mbuf = reinterpret_cast<uint32_t*>(smem_rows + (multi ? 3 : 2) * chunk);
  const int lo = min(V, rank * chunk), hi = min(V, lo + chunk);
  const int n = hi - lo;
  auto in_set = [&](int e) -> bool { return !masked || ((mbuf[e >> 5] >> (e & 31)) & 1u); };
  // Loads this CTA's chunk of local row `node` and turns it into p~, q~ in
  // place (0 off the retained set).  LSE / Z come from the partials if the
  // node has children (the same values its children were tested with), else
  // they are reduced here across the cluster (at most once per call: the
  // exchange slots are written once).  Called by every CTA of the cluster.
  auto load_row = [&](int node) {
    const size_t crow = static_cast<size_t>(n0 + node) * V;
    {
      const float* tsrc = a.target + crow + lo;
      const float* dsrc = a.draft + crow + lo;
      if (((crow + lo) & 3) == 0) {
        const int n4 = n >> 2;
        for (int k = tid; k < n4; k += kTreeThreads) {
          cp_async16(tbuf + 4 * k, tsrc + 4 * k);
          cp_async16(dbuf + 4 * k, dsrc + 4 * k);
        }
        for (int e = 4 * n4 + tid; e < n; e += kTreeThreads) {
          cp_async4(tbuf + e, tsrc + e);
          cp_async4(dbuf + e, dsrc + e);
        }
      } else {
        for (int e = tid; e < n; e += kTreeThreads) {
          cp_async4(tbuf + e, tsrc + e);
          cp_async4(dbuf + e, dsrc + e);
        }
      }
      if (masked) {  // lo is a multiple of 32: whole mask words
        const uint32_t* msrc = a.mask + static_cast<size_t>(n0 + node) * W + (lo >> 5);
        for (int k = tid; k < (n + 31) >> 5; k += kTreeThreads) mbuf[k] = __ldg(msrc + k);
      }
      cp_async_wait_all();
      __syncthreads();
    }
    float lse = 0.0f, z = 1.0f;
    if (stats) {
      if (sm.has_child[node]) {
        if (logits) lse = sm.lse[node];
        if (masked) z = sm.z[node];
      } else {
        float m = -INFINITY;
        unsigned long long zs = 0;
        for (int e = tid; e < n; e += kTreeThreads) {
          if (logits) m = fmaxf(m, tbuf[e]);
          if (masked && in_set(e)) zs += fix40(dbuf[e]);
        }
        if (logits) m = block_max_f32(sm, m);
        if (masked) zs = block_sum_u64(sm, zs);
        if (tid == 0) {
          sm.x_m = m;
          sm.x_z = zs;
        }
        cluster.sync();
        const float M = cluster_max(cluster, &sm.x_m, C);
        const unsigned long long Z = cluster_sum(cluster, &sm.x_z, C, rank,
                                                 static_cast<unsigned long long*>(nullptr));
        z = z_from_sum(Z);
        if (logits) {
          float ssum = 0.0f;
          if (M != -INFINITY)
            for (int e = tid; e < n; e += kTreeThreads) ssum += expf(tbuf[e] - M);
          ssum = block_sum_f32(sm, ssum);
          if (tid == 0) sm.x_s = ssum;
          cluster.sync();
          // the same reduction order in every CTA: the same value everywhere
          const float Ssum = cluster_sum(cluster, &sm.x_s, C, rank, static_cast<float*>(nullptr));
          lse = M + logf(Ssum);
        }
      }
    }
    // p~ and q~ in place (0 off the retained set)
    for (int e = tid; e < n; e += kTreeThreads) {
      const bool in = in_set(e);
      float p = logits ? expf(tbuf[e] - lse) : tbuf[e];
      float q = dbuf[e];
      if (masked) {
        p = __fdiv_rn(p, z);
        q = __fdiv_rn(q, z);
      }
      tbuf[e] = in ? p : 0.0f;
      dbuf[e] = in ? q : 0.0f;
    }
    __syncthreads();
  };

  // ------------------------------------------------------ multi-candidate walk
  // Every CTA of the cluster runs the same walk and takes the same decisions:
  // the tested values come from one place (the global rows before the first
  // rejection at a node, the owning CTA's chunk after it) and every sum is an
  // exact integer combined in rank order.
  if (multi) {
    // first child of node j after node `after` (children have larger indices)
    auto next_child = [&](int j, int after) -> int {
      const int i = tid;
      const uint32_t key = (i > after && i < N && sm.parent[i] == j) ? 0xFFFFu - static_cast<uint32_t>(i) : 0u;
      const uint32_t k = block_max_u32(sm, key);
      return k ? static_cast<int>(0xFFFFu - k) : -1;
    };
    int j = 0, len = 0;
    for (;;) {
      int c = next_child(j, j);
      bool loaded = false, accepted = false;
      m_rejected = false;
      while (c >= 0) {
        const int x = sm.token[c];
        if (!loaded) {
          if (tid == 0) {
            float p, q;
            node_pq(j, x, p, q);
            sm.x_p = p;
            sm.x_q = q;
          }
        } else if (tid == 0) {  // the current target lives in the chunk of CTA x / chunk
          const int owner = x / chunk;
          sm.x_p = *cluster.map_shared_rank(tbuf + (x - owner * chunk), owner);
          sm.x_q = *cluster.map_shared_rank(dbuf + (x - owner * chunk), owner);
        }
        __syncthreads();
        const float p = sm.x_p, q = sm.x_q;
        if (tid == c) {
          my_p = p;
          my_q = q;
        }
        if (__fmul_rn(sm.u[c], q) < __fmul_rn(gam, p)) {
          accepted = true;
          break;
        }
        // rejected: cur <- max(0, cur - q~) / N over the cluster
        if (loaded) cluster.sync();  // every CTA has read the tested value above
        if (!loaded) {
          load_row(j);
          loaded = true;
        }
        unsigned long long part = 0;
        for (int e = tid; e < n; e += kTreeThreads) {
          const float d = __fsub_rn(tbuf[e], dbuf[e]);
          const float r = d > 0.0f ? d : 0.0f;
          rbuf[e] = r;
          part += fix40(r);
        }
        part = block_sum_u64(sm, part);
        if (tid == 0) sm.x_u64[0] = part;
        cluster.sync();
        const unsigned long long S = cluster_sum(cluster, &sm.x_u64[0], C, rank,
                                                 static_cast<unsigned long long*>(nullptr));
        if (S > 0) {
          const float Nf = z_from_sum(S);
          for (int e = tid; e < n; e += kTreeThreads) tbuf[e] = __fdiv_rn(rbuf[e], Nf);
        }
        m_rejected = true;
        cluster.sync();  // the new current target and every slot read before reuse
        c = next_child(j, c);
      }
      if (accepted) {
        if (loaded) cluster.sync();  // the chunk is read before the next node's load
        ++len;
        j = c;
        continue;
      }
      if (tid == 0) {
        sm.cut = j;
        sm.cut_len = len;
      }
      __syncthreads();
      break;
    }
  }

  const int cut = sm.cut;
  const int len = sm.cut_len;
  if (rank == 0) {
    int32_t* path = a.path + static_cast<size_t>(b) * a.max_nodes;
    for (int k = len + tid; k < a.max_nodes; k += kTreeThreads) path[k] = -1;
    if (tid == 0) {
      for (int d = len - 1, v = cut; d >= 0; --d, v = sm.parent[v]) path[d] = v;
      a.accepted_len[b] = len;
      a.bonus_token[b] = -1;  // overwritten by the draw below (ordered by cluster barriers)
      a.status[b] = kOk;
    }
    if (a.debug_pq && tid < N) {
      a.debug_pq[2 * static_cast<size_t>(n0 + tid)] = my_p;
      a.debug_pq[2 * static_cast<size_t>(n0 + tid) + 1] = my_q;
    }
  }

  // ---------------------------------------------------------------- bonus
  // The cut row (already in shared memory when the walk rejected children
  // there); pass 0 draws from the residual, pass 1 from p~ (or the current
  // target of the walk).
  if (!(multi && m_rejected)) load_row(cut);
  const bool from_residual = multi ? m_rejected : (sm.has_child[cut] != 0);

  const float u0 = sm.u[0];
  bool drawn = false;
  const int warp = tid >> 5, lane = tid & 31;
  for (int pass = from_residual ? 0 : 1; pass < 2 && !drawn; ++pass) {
    auto quantum = [&](int e) -> unsigned long long {
      if (e >= n) return 0ull;
      if (pass == 1) return fix40(tbuf[e]);
      return fix40(multi ? rbuf[e] : __fsub_rn(tbuf[e], dbuf[e]));
    };
    // per-warp sums over contiguous spans [warp*wspan, +wspan)
    unsigned long long wsum = 0;
    for (int k = 0; k < wspan / 32; ++k) wsum += quantum(warp * wspan + k * 32 + lane);
    for (int o = 16; o; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    __syncthreads();
    if (lane == 0) sm.red_u64[warp] = wsum;
    __syncthreads();
    unsigned long long part = 0;
    for (int k = 0; k < kTreeWarps; ++k) part += sm.red_u64[k];
    if (tid == 0) sm.x_u64[pass] = part;
    cluster.sync();
    unsigned long long before = 0;
    const unsigned long long S = cluster_sum(cluster, &sm.x_u64[pass], C, rank, &before);
    if (S == 0) continue;  // the same decision in every CTA
    drawn = true;
    const unsigned long long t = scaled_draw(u0, S);
    if (t >= before && t - before < part) {  // this CTA holds the token
      unsigned long long cum = t - before;     // target offset within the CTA
      int w0 = 0;
      for (; w0 < kTreeWarps; ++w0) {
        const unsigned long long ws = sm.red_u64[w0];
        if (cum < ws) break;
        cum -= ws;
      }
      if (warp == w0) {  // walk the warp's span in steps of 32 entries
        unsigned long long acc = 0;
        for (int k = 0; k < wspan / 32; ++k) {
          const int e = warp * wspan + k * 32 + lane;
          const unsigned long long f = quantum(e);
          unsigned long long inc = f;
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
          }
          const bool hit = acc + inc > cum;
          const uint32_t hits = __ballot_sync(0xffffffffu, hit);
          if (hits) {
            if (lane == __ffs(hits) - 1) a.bonus_token[b] = lo + e;
            break;
          }
          acc += __shfl_sync(0xffffffffu, inc, 31);
        }
      }
    }
  }
  if (!drawn) {
    // no mass at all: smallest index of the largest p~ (NaN ignored)
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int e = tid; e < n; e += kTreeThreads)
      if (tbuf[e] > bv) {
        bv = tbuf[e];
        bi = lo + e;
      }
    block_argmax(sm, bv, bi);
    if (tid == 0) {
      sm.x_maxv = bv;
      sm.x_maxi = bi;
    }
    cluster.sync();
    if (rank == 0 && tid == 0) {
      float best = -INFINITY;
      int idx = 0;
      for (int c = 0; c < C; ++c) {
        const TreeSmem* o = cluster.map_shared_rank(&sm, c);
        if (o->x_maxv > best) {
          best = o->x_maxv;
          idx = o->x_maxi;
        }
      }
      a.bonus_token[b] = idx;
    }
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
}


// ============================================================ retained set
// The step before the accept pass: the retained set R of each draft row
// ([LLM] §2.1.2: tokens by descending draft probability, mass summed until it
// reaches 1 - Prune_Ratio, the crossing token kept; [LLM] §7.1 the same in log
// space), read exactly: order = key desc, id asc with key = q if q > 0 else 0;
// R = the shortest prefix of that order whose fixed-point mass sum of fix40
// quanta reaches T (the caller's floor(mass * 2^40)), or the whole row.
//
// One CTA of 1024 threads per row (or, when the rows fill at most half of the
// SMs, a cluster of two CTAs, half the row each): a wave of one CTA per SM
// holds about 150 rows (90 MB at V = 151936), so the row, read from HBM by
// the first pass, is still in L2 for the second.  A radix select over the key
// (the fp32 bit pattern, which orders non-negative floats) finds the key tau at
// which the cumulative mass crosses T, a digit at a time from the top: the
// exponent field (key bits 30..23), then bits 22..15, 14..7 and 6..0.  Every
// sum is an exact integer: within one exponent field e the fix40 weight of an
// entry is a << s, with m its 24-bit significand, a = m (e >= 110) or
// m >> (110 - e) (e < 110: the truncation of fix40) and s = max(e - 110, 0),
// so the mass of a digit is (the sum of a) << s.
//   pass 0 (the row): private u32 sums of a per thread for each of the 45
//     fields 87..131 that carry weight below the clamp (no conflicts: most
//     entries share a few fields, so shared buckets would; a thread reads at
//     most 256 entries, so a sum stays below 2^32); fields 132 and up (q >= 32
//     or +inf, weight clamped to 2^45) go to shared u64 buckets.
//   pass 1 (the row again): with the crossing field e* known, the mask bits
//     of the keys above it go to a bitmap in shared memory and those of the
//     keys of field e* to a second one, from which each warp lists the ids
//     of its run of mask words (a warp scan) in its slice of the id list.
//   Each warp gathers its keys again by id (from L2), each lane keeping
//     bits 30..15 of its keys in registers: the histogram of bits 22..15, then
//     a filter that sets the mask bits of the keys above the new 16-bit prefix
//     and copies the keys at it, with their ids, into a small list, whose
//     keys give tau (by pairwise mass sums for up to 256 keys in a one-CTA
//     row, else the histograms of bits 14..7 and 6..0).  The mask is the bitmap
//     plus the small list's keys above tau and its ties at tau: all of them
//     when their number is the number of ties to keep, c = ceil((T - mass
//     above tau) / fix40(tau)), else the c of lowest id.
// A row whose field e* holds more keys in some warp's words than its slice,
// or whose 16-bit prefix more than the small list, takes its remaining digits
// by passes over the row and its mask by a pass over the row that ranks the
// ties in id order with a block scan.  The two CTAs of a cluster row sum every
// histogram and count through distributed shared memory.
constexpr int kRsThreads = 1024;
constexpr int kRsWarps = kRsThreads / 32;
constexpr int kRsE0 = 87;                          // lowest field with weight (q >= 2^-40)
constexpr int kRsEBig = 132;                       // fields from here on: weight clamped to 2^45
constexpr int kRsExps = kRsEBig - kRsE0;           // pass 0's private sums per thread
constexpr int kRsPoolWords = kRsExps * kRsThreads; // ... as u32 [field][thread]
constexpr int kRsHists = kRsWarps / 2;             // later histograms: one per warp pair,
constexpr int kRsHistWords = kRsHists * 2 * 256;   // of two 16-bit weight parts
constexpr int kRsMaskWords = 8192;                 // a row's mask words (V <= 2^18)
constexpr int kRsSmallCap = 2048;                  // keys at the 16-bit prefix
constexpr int kRsDirect = 256;  // up to this many, tau is picked from the small list by pairwise sums
// ids of field e* the pool holds after the histograms, two bitmaps and the
// small list: at least 17408 (V = 2^18), 24296 at V = 151936
static_assert(kRsPoolWords - (kRsHistWords + 2 * kRsMaskWords + 2 * kRsSmallCap) >= 17408, "pool");
constexpr int kRsGather = 16;  // ids of field e* a thread gathers at once (kept in registers)

struct RsSmem {
  // pass 0: private sums [field][thread]; then the histograms, the mask
  // bitmaps and the small list (keys, ids)
  alignas(16) uint32_t pool[kRsPoolWords];
  unsigned long long big[256];  // pass 0: fields 132..255
  unsigned long long hist[256];
  int iscan[kRsWarps];
  int digit;
  int nsmall;
  int nties;
  int ovf;  // a warp's ids of field e* overflowed its slice
  unsigned long long above;
  unsigned long long total;
  unsigned long long xh[2][256];  // a CTA's histogram, read by the other CTAs of its row
  unsigned long long xs[2];       // ... and one value
};

// Key bits below digit p: digit 0 is bits 30..23, digits 1..3 bits 22..15,
// 14..7 and 6..0.
__device__ __forceinline__ int rs_shift(int p) { return max(23 - 8 * p, 0); }
__device__ __forceinline__ uint32_t rs_key(float x) { return x > 0.0f ? __float_as_uint(x) : 0u; }
// a of a key of field ex (weight = a << rs_wshift(ex)); 1 above the clamp
__device__ __forceinline__ uint32_t rs_addend(uint32_t key, int ex) {
  return ex >= kRsEBig ? 1u : (((key & 0x7fffffu) | 0x800000u) >> max(110 - ex, 0));
}
__device__ __forceinline__ int rs_wshift(int ex) { return ex >= kRsEBig ? 45 : max(ex - 110, 0); }

// Lane L of a warp reads id 32 word + L: a warp's load of one word is one
// 128-byte line, and the words w, w + 32, ... of the 32 warps make the CTA
// read 4 KB of consecutive ids at a time.  Ids past V read as 0.
__device__ __forceinline__ float rs_load(const float* q, int V, int id) {
  return id < V ? __ldcg(q + id) : 0.0f;
}

constexpr int kRsUnroll = 8;  // loads of a warp in flight

// The order-free passes on a 16-byte aligned row (V % 4 == 0): lane L of warp
// w reads float4 (32 g + L) for the groups g = w, w + 32, ..., so a warp load
// is 512 consecutive bytes and a CTA keeps 8 x 16 KB in flight.  Float4s past
// the row read as zeros.
__device__ __forceinline__ float4 rs_load4(const float* q, int nf, int f) {
  return f < nf ? __ldcg(reinterpret_cast<const float4*>(q) + f) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
}

// Pass 0's update for one entry (x as loaded, any value): a into this
// thread's private sum of its field (a shared atomic add: one instruction
// where a load, add and store take three; no other thread touches the
// word), or 2^45 into the shared bucket of a field above the clamp.  Non-positive entries (field >= 256 as bits), NaN,
// zeros, denormals and fields below 87 add nothing.
__device__ __forceinline__ void rs_count0(RsSmem& sm, int tid, float x) {
  const uint32_t k = __float_as_uint(x);
  const uint32_t e = k >> 23;
  const uint32_t b = e - kRsE0;
  if (b < static_cast<uint32_t>(kRsExps)) {
    const uint32_t m = (k & 0x7fffffu) | 0x800000u;
    atomicAdd(&sm.pool[b * kRsThreads + tid], m >> max(110 - static_cast<int>(e), 0));
  } else if (e - kRsEBig < static_cast<uint32_t>(256 - kRsEBig) && k <= 0x7f800000u) {
    atomicAdd(&sm.big[e], 1ull << 45);
  }
}

// Adds a (< 2^24) to digit d as two 16-bit parts: at most 16384 entries of a
// pass reach one histogram (two warps, each at most 8192 entries of a row for
// V <= 2^18), so the low part sums stay below 2^30 and the high below 2^22.
__device__ __forceinline__ void rs_add2(uint32_t* h, uint32_t d, uint32_t a) {
  if (a & 0xffffu) atomicAdd(h + d, a & 0xffffu);
  if (a >> 16) atomicAdd(h + 256 + d, a >> 16);
}

// sm.hist[d] = the warp-pair histograms' sum for digit d, times 2^wsh.
__device__ __forceinline__ void rs_reduce(RsSmem& sm, int tid, int wsh) {
  if (tid < 256) {
    unsigned long long h = 0;
    for (int g = 0; g < kRsHists; ++g) {
      const uint32_t* hg = sm.pool + g * 512;
      h += static_cast<unsigned long long>(hg[tid]) + (static_cast<unsigned long long>(hg[256 + tid]) << 16);
    }
    sm.hist[tid] = h << wsh;
  }
}

// The CTAs of a row in a cluster of C (C = 2: each takes half the row)
// combine their histograms and counts through distributed shared memory.  An
// exchange publishes into buffer xi & 1, meets the others at a cluster
// barrier and reads theirs: a CTA writes a buffer again two exchanges later,
// after the barrier of the exchange between, which the others reach only
// after reading it.
template <int C>
__device__ __forceinline__ void rs_done() {
  if constexpr (C > 1) cg::this_cluster().sync();  // no CTA leaves while another may read its buffers
}

// The sum over the row's CTAs of v (the same in every thread of a CTA);
// *lower = the sum over the CTAs of lower rank (the earlier ids).  Every
// thread calls it.
template <int C>
__device__ unsigned long long rs_xsum(RsSmem& sm, int& xi, unsigned long long v, unsigned long long* lower) {
  if constexpr (C == 1) {
    if (lower) *lower = 0ull;
    return v;
  } else {
    cg::cluster_group cl = cg::this_cluster();
    const int b = xi & 1;
    if (threadIdx.x == 0) sm.xs[b] = v;
    cl.sync();
    const int me = static_cast<int>(cl.block_rank());
    unsigned long long t = 0, lo = 0;
    for (int r = 0; r < C; ++r) {
      const unsigned long long y = *cl.map_shared_rank(&sm.xs[b], r);
      t += y;
      if (r < me) lo += y;
    }
    if (lower) *lower = lo;
    ++xi;
    return t;
  }
}

// The crossing digit of sm.hist (written before a barrier; summed over the
// row's CTAs): the one digit d with above + mass(digits > d) < T <= above +
// mass(digits >= d), where above is the mass of the keys above the current
// prefix range.  Sets sm.digit and sm.above (and sm.total, the whole row,
// when `first`).  Warp 0 alone scans: lane L holds digits 8L .. 8L + 7, a
// shuffle scan sums the lanes above, and each lane walks its own digits.
// Every thread calls it; it ends with a barrier.
template <int C>
__device__ void rs_pick(RsSmem& sm, int tid, unsigned long long above, unsigned long long T, bool first, int& xi) {
  const int lane = tid & 31;
  if constexpr (C > 1) {
    cg::cluster_group cl = cg::this_cluster();
    const int b = xi & 1;
    if (tid < 256) sm.xh[b][tid] = sm.hist[tid];
    cl.sync();
    if (tid < 256) {
      unsigned long long H = 0ull;
      for (int r = 0; r < C; ++r) H += *cl.map_shared_rank(&sm.xh[b][tid], r);
      sm.hist[tid] = H;
    }
    ++xi;
    __syncthreads();
  }
  if (tid < 32) {
    unsigned long long h[8], own = 0ull;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      h[k] = sm.hist[8 * lane + k];
      own += h[k];
    }
    unsigned long long incl = own;  // the digits of this lane and of the lanes above
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_down_sync(0xffffffffu, incl, o);
      if (lane + o < 32) incl += y;
    }
    const unsigned long long ge0 = above + incl;  // mass of digits >= 8 lane
    if (first && lane == 0) sm.total = ge0;       // digit 0: the whole row
    unsigned long long lower = 0ull;              // this lane's digits below k
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const unsigned long long gek = ge0 - lower;  // mass of digits >= 8 lane + k
      const unsigned long long gtk = gek - h[k];   // mass of digits > 8 lane + k
      if (gtk < T && gek >= T) {
        sm.digit = 8 * lane + k;
        sm.above = gtk;
      }
      lower += h[k];
    }
  }
  __syncthreads();
}

// Rows row0 + blockIdx.x / C; CTA h = blockIdx.x % C of a row (its rank in
// the cluster) takes mask words [h wp, h wp + wp) of it, wp = ceil(words / C)
// rounded up to 4 words (128 ids): V, words, q and mrow below are the part's.
template <int C>
__global__ void __launch_bounds__(kRsThreads, 1)
    retained_set_kernel(const RetainArgs a, int row0) {
  extern __shared__ __align__(16) uint8_t rs_raw[];
  RsSmem& sm = *reinterpret_cast<RsSmem*>(rs_raw);
  const int row = row0 + static_cast<int>(blockIdx.x) / C;
  const int h = static_cast<int>(blockIdx.x) % C;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t lt_mask = (1u << lane) - 1u;
  const int Vrow = a.vocab, wrow = (Vrow + 31) >> 5;
  const int wp = C == 1 ? wrow : (((wrow + C - 1) / C + 3) & ~3);
  const int wlo = min(h * wp, wrow);
  const int words = min(wlo + wp, wrow) - wlo;
  const int V = max(0, min(Vrow, 32 * (wlo + words)) - 32 * wlo);
  const bool vec = (Vrow & 3) == 0;  // the row (and so the part) starts 16-byte aligned
  const int nf = V >> 2;             // its float4s when vec
  const float* q = a.draft + static_cast<size_t>(row) * Vrow + 32 * wlo;
  uint32_t* mrow = a.mask + static_cast<size_t>(row) * wrow + wlo;
  int xi = 0;  // exchanges so far
  const unsigned long long T = a.threshold;
  uint32_t* whist = sm.pool;
  uint32_t* myh = whist + (warp >> 1) * 512;
  // the pool after pass 0: histograms, the two bitmaps, the small list, the ids
  uint32_t* bits = sm.pool + kRsHistWords;
  uint32_t* mbits = bits + words;
  uint32_t* skeys = mbits + words;
  uint32_t* sids = skeys + kRsSmallCap;
  uint32_t* ids = sids + kRsSmallCap;
  const int cap = kRsPoolWords - (kRsHistWords + 2 * words + 2 * kRsSmallCap);  // >= 17408

  // ---- pass 0: the field of every entry
#pragma unroll
  for (int b = 0; b < kRsExps; ++b) sm.pool[b * kRsThreads + tid] = 0u;
  if (tid < 256) sm.big[tid] = 0ull;
  __syncthreads();
  if (vec) {
    for (int g0 = warp; g0 * 32 < nf; g0 += kRsWarps * kRsUnroll) {
      float4 x[kRsUnroll];
#pragma unroll
      for (int u = 0; u < kRsUnroll; ++u) x[u] = rs_load4(q, nf, (g0 + u * kRsWarps) * 32 + lane);
#pragma unroll
      for (int u = 0; u < kRsUnroll; ++u) {
        rs_count0(sm, tid, x[u].x);
        rs_count0(sm, tid, x[u].y);
        rs_count0(sm, tid, x[u].z);
        rs_count0(sm, tid, x[u].w);
      }
    }
  } else {
    for (int w0 = warp; w0 < words; w0 += kRsWarps * kRsUnroll) {
      float x[kRsUnroll];
#pragma unroll
      for (int u = 0; u < kRsUnroll; ++u) {
        const int word = w0 + u * kRsWarps;
        x[u] = word < words ? rs_load(q, V, word * 32 + lane) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < kRsUnroll; ++u) rs_count0(sm, tid, x[u]);
    }
  }
  __syncthreads();
  // field masses: a warp per field sums the 1024 private sums (< 2^42: at
  // most 2^18 entries of a < 2^24), then shifts
  for (int b = warp; b < kRsExps; b += kRsWarps) {
    unsigned long long y = 0;
    for (int i = lane; i < kRsThreads; i += 32) y += sm.pool[b * kRsThreads + i];
    for (int o = 16; o; o >>= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
    if (lane == 0) sm.hist[kRsE0 + b] = y << max(kRsE0 + b - 110, 0);
  }
  if (tid < 256 && (tid < kRsE0 || tid >= kRsEBig)) sm.hist[tid] = tid < kRsE0 ? 0ull : sm.big[tid];
  __syncthreads();
  rs_pick<C>(sm, tid, 0ull, T, true, xi);
  if (sm.total < T) {  // the mass never reaches T: every token is kept
    const unsigned long long total = sm.total;
    for (int word = tid; word < words; word += kRsThreads) {
      const int v0 = word * 32;
      mrow[word] = (V - v0 >= 32) ? 0xffffffffu : ((1u << (V - v0)) - 1u);
    }
    if (tid == 0 && h == 0) {
      if (a.z_fixed) a.z_fixed[row] = total;
      if (a.z) a.z[row] = __fmul_rn(__ull2float_rn(total), kTwoM40);
      if (a.kept) a.kept[row] = Vrow;
    }
    rs_done<C>();
    return;
  }
  const int ex = sm.digit;  // e*: 87..255 (its mass is > 0)
  const int wsh = rs_wshift(ex);
  uint32_t prefix = static_cast<uint32_t>(ex);
  unsigned long long above = sm.above;  // mass of the keys above the prefix range

  // ---- pass 1: mask bits of the keys of fields above e* (bits) and of
  // field e* (mbits), each word written once; the histograms of the next
  // digit are cleared meanwhile (pass 0's sums are read)
  for (int i = tid; i < kRsHistWords; i += kRsThreads) whist[i] = 0u;
  if (tid == 0) {
    sm.nsmall = 0;
    sm.nties = 0;
    sm.ovf = 0;
  }
  {
    const uint32_t lim = static_cast<uint32_t>(ex + 1) << 23;  // keys of fields > e*
    const uint32_t lo = static_cast<uint32_t>(ex) << 23;       // keys of field e*: [lo, lim)
    // the same tests on the floats (false for NaN and for x <= 0): x above
    // field e* iff x >= flim (NaN bound for e* = 255: nothing is above), x
    // in it iff x >= flo and not above
    const float flim = __uint_as_float(ex < 255 ? lim : 0x7fc00000u);
    const float flo = __uint_as_float(lo);
    if (vec) {
      for (int g0 = warp; g0 * 32 < nf; g0 += kRsWarps * kRsUnroll) {
        float4 x[kRsUnroll];
#pragma unroll
        for (int u = 0; u < kRsUnroll; ++u) x[u] = rs_load4(q, nf, (g0 + u * kRsWarps) * 32 + lane);
#pragma unroll
        for (int u = 0; u < kRsUnroll; ++u) {
          const int f = (g0 + u * kRsWarps) * 32 + lane;  // ids 4f .. 4f + 3
          // mask word f / 8 holds the nibbles of lanes 8j .. 8j + 7, the
          // nibble of lane L at bit 4 (L % 8)
          const int sh = 4 * (lane & 7);
          const uint32_t an = static_cast<uint32_t>(x[u].x >= flim) | (static_cast<uint32_t>(x[u].y >= flim) << 1) |
                              (static_cast<uint32_t>(x[u].z >= flim) << 2) |
                              (static_cast<uint32_t>(x[u].w >= flim) << 3);
          const uint32_t gn = static_cast<uint32_t>(x[u].x >= flo) | (static_cast<uint32_t>(x[u].y >= flo) << 1) |
                              (static_cast<uint32_t>(x[u].z >= flo) << 2) |
                              (static_cast<uint32_t>(x[u].w >= flo) << 3);
          uint32_t av = an << sh;
          uint32_t mv = (gn & ~an) << sh;
#pragma unroll
          for (int o = 1; o < 8; o <<= 1) {
            av |= __shfl_xor_sync(0xffffffffu, av, o);
            mv |= __shfl_xor_sync(0xffffffffu, mv, o);
          }
          if ((lane & 7) == 0 && (f >> 3) < words) {
            bits[f >> 3] = av;
            mbits[f >> 3] = mv;
          }
        }
      }
    } else {
      for (int w0 = warp; w0 < words; w0 += kRsWarps * kRsUnroll) {
        float x[kRsUnroll];
#pragma unroll
        for (int u = 0; u < kRsUnroll; ++u) {
          const int word = w0 + u * kRsWarps;
          x[u] = word < words ? rs_load(q, V, word * 32 + lane) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kRsUnroll; ++u) {
          const int word = w0 + u * kRsWarps;
          const uint32_t av = __ballot_sync(0xffffffffu, x[u] >= flim);
          const uint32_t mv = __ballot_sync(0xffffffffu, x[u] >= flo) & ~av;
          if (lane == 0 && word < words) {
            bits[word] = av;
            mbits[word] = mv;
          }
        }
      }
    }
  }
  __syncthreads();
  // ---- the ids of field e*: warp w takes mask words [w wpw, w wpw + wpw),
  // 32 at a time (lane L word base + L), and lists their ids in id order in
  // its own slice of the list (a warp scan of the words' counts); no block
  // barrier until the histogram below is complete
  const int wpw = (words + kRsWarps - 1) / kRsWarps;
  const int slice = cap / kRsWarps;
  uint32_t* wids = ids + warp * slice;
  int n = 0;  // ids of field e* in this warp's words (the same in every lane)
  {
    const int wb = min(warp * wpw, words), we = min(wb + wpw, words);
    for (int base = wb; base < we; base += 32) {
      const int w = base + lane;
      const uint32_t v0 = w < we ? mbits[w] : 0u;
      const int c = __popc(v0);
      int incl = c;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int pos = n + incl - c;
      for (uint32_t v = v0; v; v &= v - 1u, ++pos)
        if (pos < slice) wids[pos] = 32u * static_cast<uint32_t>(w) + static_cast<uint32_t>(__ffs(v) - 1);
      n += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0 && n > slice) sm.ovf = 1;
  }
  const int nw = min(n, slice);

  // ---- digit 1 (bits 22..15) over the listed keys, gathered again by id:
  // lane L of a warp takes its slice's entries L + 32 u, and keeps bits
  // 30..15 of the keys of the first round in registers (two to a register)
  // for the filter.  (A warp whose slice overflowed makes the whole row take
  // the passes over the row below, so its partial sums do not matter.)
  uint32_t hk[kRsGather / 2];
#pragma unroll
  for (int u = 0; u < kRsGather / 2; ++u) hk[u] = 0u;
  for (int r0 = 0; r0 < nw; r0 += 32 * kRsGather) {
    float x[kRsGather];
#pragma unroll
    for (int u = 0; u < kRsGather; ++u) {
      const int i = r0 + lane + 32 * u;
      x[u] = i < nw ? __ldcg(q + wids[i]) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kRsGather; ++u) {
      if (r0 + lane + 32 * u < nw) {
        const uint32_t k = rs_key(x[u]);
        rs_add2(myh, (k >> 15) & 255u, rs_addend(k, ex));
        if (r0 == 0) hk[u / 2] |= (k >> 15) << (16 * (u & 1));
      }
    }
  }
  __syncthreads();

  int p = 1;  // the next digit
  if (rs_xsum<C>(sm, xi, sm.ovf ? 1ull : 0ull, nullptr) == 0ull) {  // every part's ids listed
    rs_reduce(sm, tid, wsh);
    __syncthreads();
    rs_pick<C>(sm, tid, above, T, false, xi);
    prefix = (prefix << 8) | static_cast<uint32_t>(sm.digit);  // key >> 15 of tau
    above = sm.above;
    p = 2;
    // ---- filter: keys above the 16-bit prefix into the bitmap, keys at it
    // (with their ids) into the small list
    for (int r0 = 0; r0 < nw; r0 += 32 * kRsGather) {
      uint32_t hv[kRsGather];
      if (r0 == 0) {
#pragma unroll
        for (int u = 0; u < kRsGather; ++u) hv[u] = (hk[u / 2] >> (16 * (u & 1))) & 0xffffu;
      } else {
#pragma unroll
        for (int u = 0; u < kRsGather; ++u) {
          const int i = r0 + lane + 32 * u;
          hv[u] = i < nw ? __float_as_uint(__ldcg(q + wids[i])) : 0u;
        }
#pragma unroll
        for (int u = 0; u < kRsGather; ++u) hv[u] = rs_key(__uint_as_float(hv[u])) >> 15;
      }
#pragma unroll
      for (int u = 0; u < kRsGather; ++u) {
        const int i = r0 + lane + 32 * u;
        if (i < nw) {
          const uint32_t id = wids[i];
          if (hv[u] > prefix) {
            atomicOr(bits + (id >> 5), 1u << (id & 31u));
          } else if (hv[u] == prefix) {
            const int s = atomicAdd(&sm.nsmall, 1);
            if (s < kRsSmallCap) {
              skeys[s] = rs_key(__ldcg(q + id));
              sids[s] = id;
            }
          }
        }
      }
    }
    __syncthreads();  // also: sm.digit / sm.above are rewritten by the next pick
    const int nsmall = sm.nsmall;
    if (rs_xsum<C>(sm, xi, nsmall > kRsSmallCap ? 1ull : 0ull, nullptr) == 0ull) {
      if (C == 1 && nsmall <= kRsDirect) {
        // ---- tau directly: the key of the small list (all keys at the
        // 16-bit prefix) whose mass above, plus the mass above the prefix,
        // is < T while that plus its own ties' mass is >= T; exactly one
        // distinct key qualifies, and its entries all write the same values
        for (int i = tid; i < nsmall; i += kRsThreads) {
          const uint32_t ki = skeys[i];
          unsigned long long gt = 0, eq = 0;
          for (int k = 0; k < nsmall; ++k) {
            const uint32_t kj = skeys[k];
            const unsigned long long w = static_cast<unsigned long long>(rs_addend(kj, ex)) << wsh;
            gt += kj > ki ? w : 0ull;
            eq += kj == ki ? w : 0ull;
          }
          if (above + gt < T && above + gt + eq >= T) {
            sm.digit = static_cast<int>(ki);
            sm.above = above + gt;
          }
        }
        __syncthreads();
        prefix = static_cast<uint32_t>(sm.digit);
        above = sm.above;
        p = 4;
      }
      // ---- digits 2 and 3 over the small list
      for (; p < 4; ++p) {
        const int sh = rs_shift(p), shp = rs_shift(p - 1);
        const uint32_t dm = (1u << (shp - sh)) - 1u;
        for (int i = tid; i < kRsHistWords; i += kRsThreads) whist[i] = 0u;
        __syncthreads();
        for (int i = tid; i < nsmall; i += kRsThreads) {
          const uint32_t k = skeys[i];
          if ((k >> shp) == prefix) rs_add2(myh, (k >> sh) & dm, rs_addend(k, ex));
        }
        __syncthreads();
        rs_reduce(sm, tid, wsh);
        __syncthreads();
        rs_pick<C>(sm, tid, above, T, false, xi);
        prefix = (prefix << (shp - sh)) | static_cast<uint32_t>(sm.digit);
        above = sm.above;
        __syncthreads();
      }
      // ---- the mask: the bitmap, the small list's keys above tau, its ties
      const uint32_t tau = prefix;
      const unsigned long long wt = static_cast<unsigned long long>(rs_addend(tau, ex)) << wsh;  // > 0
      const unsigned long long need = (T - above + wt - 1) / wt;  // ties to keep (<= the ties)
      for (int i = tid; i < nsmall; i += kRsThreads) {
        const uint32_t k = skeys[i], id = sids[i];
        if (k > tau) {
          atomicOr(bits + (id >> 5), 1u << (id & 31u));
        } else if (k == tau) {
          atomicAdd(&sm.nties, 1);
        }
      }
      __syncthreads();
      unsigned long long lower_ties = 0;  // ties in the parts of lower id
      const unsigned long long nties =
          rs_xsum<C>(sm, xi, static_cast<unsigned long long>(sm.nties), &lower_ties);
      for (int i = tid; i < nsmall; i += kRsThreads) {
        if (skeys[i] != tau) continue;
        const uint32_t id = sids[i];
        bool keep = nties <= need;  // all of them
        if (!keep) {                // else the need of lowest id
          unsigned long long r = 0;
          for (int j = 0; j < nsmall; ++j) r += (skeys[j] == tau && sids[j] < id) ? 1ull : 0ull;
          keep = lower_ties + r < need;
        }
        if (keep) atomicOr(bits + (id >> 5), 1u << (id & 31u));
      }
      __syncthreads();
      int cnt = 0;
      for (int w = tid; w < words; w += kRsThreads) {
        const uint32_t v = bits[w];
        mrow[w] = v;
        cnt += __popc(v);
      }
      for (int o = 16; o; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      if (lane == 0) sm.iscan[warp] = cnt;
      __syncthreads();
      unsigned long long kept = 0;
      for (int w = 0; w < kRsWarps; ++w) kept += static_cast<unsigned long long>(sm.iscan[w]);
      kept = rs_xsum<C>(sm, xi, kept, nullptr);
      if (tid == 0 && h == 0) {
        const unsigned long long Z = above + need * wt;
        if (a.z_fixed) a.z_fixed[row] = Z;
        if (a.z) a.z[row] = __fmul_rn(__ull2float_rn(Z), kTwoM40);
        if (a.kept) a.kept[row] = static_cast<int>(kept);
      }
      rs_done<C>();
      return;
    }
  }

  // ---- the remaining digits by passes over the row (from L2)
  for (; p < 4; ++p) {
    const int sh = rs_shift(p), shp = rs_shift(p - 1);
    const uint32_t dm = (1u << (shp - sh)) - 1u;
    for (int i = tid; i < kRsHistWords; i += kRsThreads) whist[i] = 0u;
    __syncthreads();
    auto add = [&](float x) {
      const uint32_t k = rs_key(x);
      if ((k >> shp) == prefix) rs_add2(myh, (k >> sh) & dm, rs_addend(k, ex));
    };
    if (vec) {
      for (int g0 = warp; g0 * 32 < nf; g0 += kRsWarps * kRsUnroll) {
        float4 x[kRsUnroll];
#pragma unroll
        for (int u = 0; u < kRsUnroll; ++u) x[u] = rs_load4(q, nf, (g0 + u * kRsWarps) * 32 + lane);
#pragma unroll
        for (int u = 0; u < kRsUnroll; ++u) {
          add(x[u].x);
          add(x[u].y);
          add(x[u].z);
          add(x[u].w);
        }
      }
    } else {
      for (int w0 = warp; w0 < words; w0 += kRsWarps * kRsUnroll) {
        float x[kRsUnroll];
#pragma unroll
        for (int u = 0; u < kRsUnroll; ++u) {
          const int word = w0 + u * kRsWarps;
          x[u] = word < words ? rs_load(q, V, word * 32 + lane) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kRsUnroll; ++u) add(x[u]);
      }
    }
    __syncthreads();
    rs_reduce(sm, tid, wsh);
    __syncthreads();
    rs_pick<C>(sm, tid, above, T, false, xi);
    prefix = (prefix << (shp - sh)) | static_cast<uint32_t>(sm.digit);
    above = sm.above;
    __syncthreads();  // sm.digit / sm.above are rewritten by the next pick
  }
  const uint32_t tau = prefix;
  const unsigned long long wt = static_cast<unsigned long long>(rs_addend(tau, ex)) << wsh;  // > 0
  const unsigned long long need = (T - above + wt - 1) / wt;  // ties to keep

  // ---- the mask by a pass over the row, in rounds of 1024 consecutive
  // words: warp w reads words base + 32w + j (j = 0..31, lane L holding id
  // 32 word + L), so a word's keep and tie bits are two ballots, and lane L
  // keeps those of word base + 32w + L.  The ties' ranks in id order are the
  // ties of the parts of lower id and of the earlier rounds plus a block scan
  // of the per-word counts of this round.
  unsigned long long ties_before = 0;  // ties in the lower parts and the earlier rounds
  if constexpr (C > 1) {
    int t = 0;
    for (int w = warp; w < words; w += kRsWarps) t += rs_key(rs_load(q, V, w * 32 + lane)) == tau ? 1 : 0;
    for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) sm.iscan[warp] = t;
    __syncthreads();
    unsigned long long own = 0;
    for (int w = 0; w < kRsWarps; ++w) own += static_cast<unsigned long long>(sm.iscan[w]);
    rs_xsum<C>(sm, xi, own, &ties_before);  // its barrier also orders sm.iscan
  }
  int n_gt = 0;                        // kept keys above tau in this thread's words
  for (int base = 0; base < words; base += kRsThreads) {
    const int wb = base + 32 * warp;
    uint32_t gtb = 0, tieb = 0;
    {
      float x[32];  // the warp's 32 words of the round, all loads in flight
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        const int word = wb + u;
        x[u] = word < words ? rs_load(q, V, word * 32 + lane) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        const uint32_t k = rs_key(x[u]);
        const uint32_t g = __ballot_sync(0xffffffffu, k > tau);
        const uint32_t t = __ballot_sync(0xffffffffu, k == tau);
        if (lane == u) {
          gtb = g;
          tieb = t;
        }
      }
    }
    const int word = wb + lane;  // this thread's word (masks 0 past the row)
    const int c = __popc(tieb);
    n_gt += __popc(gtb);
    int incl_t = c;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl_t, o);
      if (lane >= o) incl_t += y;
    }
    if (lane == 31) sm.iscan[warp] = incl_t;
    __syncthreads();
    int before = incl_t - c;
    int round_ties = 0;
    for (int w = 0; w < kRsWarps; ++w) {
      const int y = sm.iscan[w];
      if (w < warp) before += y;
      round_ties += y;
    }
    if (word < words) {
      // keep this word's ties of rank < need, lowest ids first
      const unsigned long long r0 = ties_before + static_cast<unsigned long long>(before);
      uint32_t keep = 0;
      if (r0 < need) {
        const unsigned long long m = need - r0;
        uint32_t t = tieb;
        for (unsigned long long i = 0; i < m && t; ++i) {
          keep |= t & (0u - t);
          t &= t - 1u;
        }
      }
      mrow[word] = gtb | keep;
    }
    ties_before += static_cast<unsigned long long>(round_ties);
    __syncthreads();  // sm.iscan is rewritten next round
  }
  // keys above tau over the row
  for (int o = 16; o; o >>= 1) n_gt += __shfl_xor_sync(0xffffffffu, n_gt, o);
  if (lane == 0) sm.iscan[warp] = n_gt;
  __syncthreads();
  unsigned long long g = 0;
  for (int w = 0; w < kRsWarps; ++w) g += static_cast<unsigned long long>(sm.iscan[w]);
  g = rs_xsum<C>(sm, xi, g, nullptr);
  if (tid == 0 && h == 0) {
    const unsigned long long Z = above + need * wt;
    if (a.z_fixed) a.z_fixed[row] = Z;
    if (a.z) a.z[row] = __fmul_rn(__ull2float_rn(Z), kTwoM40);
    if (a.kept) a.kept[row] = static_cast<int>(g + need);
  }
  rs_done<C>();
}
}  // namespace

int accept_chunks(int vocab) { return (vocab + kChunk - 1) / kChunk; }

// CTAs per tree: 1, 2, 4, 8 or 16, about one per kMinChunk entries of the
// vocabulary; halved while the trees' clusters would not fit one wave of
// `sms` SMs, but never below what keeps a CTA's chunk within 16384 entries
// (the shared-memory size the kernel is set up for).
int accept_cluster_size(int vocab, int batch, int sms) {
  const int want = (vocab + kMinChunk - 1) / kMinChunk;
  int c = 1;
  while (c < want && c < kMaxCluster) c *= 2;
  int c_min = 1;
  while (c_min < kMaxCluster && static_cast<long>(c_min) * 16384 < vocab) c_min *= 2;
  while (c > c_min && static_cast<long>(batch) * c > sms) c /= 2;
  return c;
}

int launch_accept(const AcceptArgs& a, void* workspace, cudaStream_t stream) {
  const int nchunk = accept_chunks(a.vocab);
  static thread_local int sms_dev = -1, sms = 148;
  {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev != sms_dev &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0) {
      sms = n;
      sms_dev = dev;
    }
  }
  const int C = accept_cluster_size(a.vocab, a.batch, sms);
  float2* ws_ms = static_cast<float2*>(workspace);
  unsigned long long* ws_z = reinterpret_cast<unsigned long long*>(
      static_cast<char*>(workspace) + sizeof(float2) * static_cast<size_t>(a.total_nodes) * nchunk);
  const bool stats = a.kind == 1 || a.mask != nullptr;
  // CTAs per row: enough for about four CTAs per SM over all rows (most of
  // which are leaves and exit at once), twelve when draft rows and a mask
  // are read too (rows of twice the bytes, six CTAs per SM); each takes
  // every nparts-th chunk.  At most one per workspace chunk.
  const bool masked = a.mask != nullptr;
  const long per_sm = masked ? 12l : 4l;
  const int nparts = max(1, min(nchunk, static_cast<int>((per_sm * sms + a.total_nodes - 1) / a.total_nodes)));
  if (stats) {
    const unsigned items = static_cast<unsigned>(static_cast<long>(a.total_nodes) * nparts);
    if (masked) {
      constexpr int kCh4 = kRowThreads * 4 * 4;
      accept_rowstats_kernel<4><<<items, kRowThreads, 0, stream>>>(a, (a.vocab + kCh4 - 1) / kCh4, nparts,
                                                                   ws_ms, ws_z);
    } else {
      accept_rowstats_kernel<kRowVec><<<items, kRowThreads, 0, stream>>>(a, nchunk, nparts, ws_ms, ws_z);
    }
    if (cudaGetLastError() != cudaSuccess) return -1;
  }
  static thread_local int attr_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev != dev) {
    cudaFuncSetAttribute(accept_tree_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaFuncSetAttribute(accept_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         tree_smem_bytes(16384, true));
    attr_dev = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, a.batch, 1);
  cfg.blockDim = dim3(kTreeThreads, 1, 1);
  cfg.dynamicSmemBytes = tree_smem_bytes(bonus_chunk(a.vocab, C), a.test == 2);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = stats ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, accept_tree_kernel, a, nparts,
                            static_cast<const float2*>(ws_ms),
                            static_cast<const unsigned long long*>(ws_z)) == cudaSuccess
             ? 0
             : -1;
}

size_t accept_workspace_bytes(int vocab, int total_nodes) {
  return static_cast<size_t>(total_nodes) * accept_chunks(vocab) *
         (sizeof(float2) + sizeof(unsigned long long));
}

int accept_max_nodes() { return kMaxN; }

// One CTA per row, or two (a cluster of two, half the row each) when the
// rows fill at most half of the SMs.
int launch_retained_set(const RetainArgs& a, cudaStream_t stream) {
  static thread_local int attr_dev = -1, sms = 148;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev != dev) {
    cudaFuncSetAttribute(retained_set_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(sizeof(RsSmem)));
    cudaFuncSetAttribute(retained_set_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(sizeof(RsSmem)));
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0) sms = n;
    attr_dev = dev;
  }
  const int split = 2 * a.rows <= sms ? a.rows : 0;  // rows of two CTAs
  const int whole = a.rows - split;
  if (whole > 0) {
    retained_set_kernel<1><<<static_cast<unsigned>(whole), kRsThreads, sizeof(RsSmem), stream>>>(a, 0);
    if (cudaGetLastError() != cudaSuccess) return -1;
  }
  if (split > 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * split, 1, 1);
    cfg.blockDim = dim3(kRsThreads, 1, 1);
    cfg.dynamicSmemBytes = sizeof(RsSmem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, retained_set_kernel<2>, a, whole) != cudaSuccess) return -1;
  }
  return 0;
}


}  // namespace tv
