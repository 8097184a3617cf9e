// accept_kernel.cu -- the fused accept pass: one thread-block cluster per tree.
//
// Sources (titles abbreviated):
//   [EC]  "端云协同推测解码中草稿模型动态生成与验证并行化：探究树形注意力机制与显存碎片整理联合加速",
//         §2.2.3 batch verification: p_accept = min(1, p_target/p_draft) per
//         node, parallel uniforms -> accept mask, root-first search cut at the
//         first rejection, longest accepted path, all inside a GPU kernel with
//         no host round trip.
//   [LLM] "端侧大模型推测解码草稿模型动态剪枝策略：详解基于重要性采样的树形验证并行加速机制",
//         §2.2.1-§2.2.2 importance correction q~ = q 1_R / Z and the ScaleMask
//         step (add log(1/Z) on retained tokens, -inf elsewhere); §7.1 the
//         log-space chain (log w = -LSE of the kept draft mass); §1.2 step 3
//         resampling at the rejection.
//
// Design (GB300): grid (C, B) with cluster (C,1,1): the C CTAs of a cluster
// share one tree and talk through distributed shared memory.
//   phase 1  rows with children: log-sum-exp of the target logits row (fp32,
//            online max/sum, 128-bit loads) and/or the retained draft mass Z
//            (exact 2^-40 fixed point, 64-bit integer sums), rows spread over
//            the cluster; then p~, q~ of the children.
//   phase 2  every CTA gathers p~, q~ of all nodes over DSMEM, takes the tests
//            with warp ballots, and walks each node's parent chain over the
//            ballot bits; a block max over (depth, -index) picks the cut node.
//   phase 3  the bonus draw: the cut node's row is split across the cluster,
//            each CTA sums its fixed-point quanta, the partial sums are
//            combined in rank order over DSMEM, and the CTA whose range holds
//            t = floor(u0 * S) finds the token with a block scan.
// Every decision-carrying sum is an exact integer, so the result does not
// depend on the reduction order.
#include <cooperative_groups.h>

#include "tv_device.cuh"
#include "tv_launch.h"

namespace cg = cooperative_groups;

namespace tv {
namespace {

constexpr int kThreads = 512;
constexpr int kMaxN = 512;
constexpr int kWarps = kThreads / 32;

struct AccSmem {
  int32_t parent[kMaxN];
  int32_t token[kMaxN];
  float u[kMaxN];
  float pq[kMaxN][2];     // p~, q~ of node i (written by the CTA owning parent(i))
  float row_lse[kMaxN];   // logits mode: LSE of rows owned by this CTA
  float row_z[kMaxN];     // mask mode: Z of rows owned by this CTA
  uint8_t has_child[kMaxN];
  uint32_t acc_bits[kMaxN / 32];
  // block reductions
  float red_f0[kWarps], red_f1[kWarps];
  unsigned long long red_u64[kWarps];
  uint32_t red_u32[kWarps];
  int red_i32[kWarps];
  // cluster exchange slots (read by the other CTAs)
  float x_m, x_s;            // partial (max, sum) of exp
  unsigned long long x_u64;  // partial fixed-point sum
  float x_maxv;
  int x_maxi;
  int bad;
  int cut;                   // j*
  int cut_len;
};

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
  return __float2ull_rz(__fmul_rn(r, 1099511627776.0f));
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

__device__ __forceinline__ bool mask_bit(const uint32_t* mrow, int v) {
  return (__ldg(mrow + (v >> 5)) >> (v & 31)) & 1u;
}

// ---- block reductions (all threads call; result valid in every thread)
__device__ unsigned long long block_sum_u64(AccSmem& sm, unsigned long long x) {
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sm.red_u64[w] = x;
  __syncthreads();
  unsigned long long t = 0;
  for (int i = 0; i < kWarps; ++i) t += sm.red_u64[i];
  return t;
}
__device__ uint32_t block_max_u32(AccSmem& sm, uint32_t x) {
  x = __reduce_max_sync(0xffffffffu, x);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sm.red_u32[w] = x;
  __syncthreads();
  uint32_t t = 0;
  for (int i = 0; i < kWarps; ++i) t = max(t, sm.red_u32[i]);
  return t;
}
__device__ void block_lse(AccSmem& sm, float& m, float& s) {
  for (int o = 16; o; o >>= 1) {
    float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_combine(m, s, m2, s2);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) {
    sm.red_f0[w] = m;
    sm.red_f1[w] = s;
  }
  __syncthreads();
  m = -INFINITY;
  s = 0.0f;
  for (int i = 0; i < kWarps; ++i) lse_combine(m, s, sm.red_f0[i], sm.red_f1[i]);
}
// max value, smallest index among equal maxima (NaN ignored)
__device__ void block_argmax(AccSmem& sm, float& v, int& idx) {
  for (int o = 16; o; o >>= 1) {
    float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    if (v2 > v || (v2 == v && i2 < idx)) {
      v = v2;
      idx = i2;
    }
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) {
    sm.red_f0[w] = v;
    sm.red_i32[w] = idx;
  }
  __syncthreads();
  v = -INFINITY;
  idx = 0x7fffffff;
  for (int i = 0; i < kWarps; ++i) {
    if (sm.red_f0[i] > v || (sm.red_f0[i] == v && sm.red_i32[i] < idx)) {
      v = sm.red_f0[i];
      idx = sm.red_i32[i];
    }
  }
}

// Visits every element v in [lo, hi) of a row of floats whose first element
// sits at float index `rowbase` of a 16-byte aligned buffer; 128-bit loads on
// the aligned body, threads strided.  f(v, value_target, value_draft).
template <bool kTwo, typename F>
__device__ __forceinline__ void for_row(const float* t, const float* d, size_t rowbase, int lo,
                                        int hi, F&& f) {
  int a0 = lo + static_cast<int>((4 - ((rowbase + lo) & 3)) & 3);
  if (a0 > hi) a0 = hi;
  const int a1 = a0 + ((hi - a0) & ~3);
  for (int v = lo + threadIdx.x; v < a0; v += kThreads) f(v, t[v], kTwo ? d[v] : 0.0f);
  for (int v = a0 + 4 * threadIdx.x; v < a1; v += 4 * kThreads) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(t + v));
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
    if (kTwo) y = __ldg(reinterpret_cast<const float4*>(d + v));
    f(v, x.x, y.x);
    f(v + 1, x.y, y.y);
    f(v + 2, x.z, y.z);
    f(v + 3, x.w, y.w);
  }
  for (int v = a1 + threadIdx.x; v < hi; v += kThreads) f(v, t[v], kTwo ? d[v] : 0.0f);
}

__global__ void __launch_bounds__(kThreads, 1) accept_kernel(const AcceptArgs a) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int b = blockIdx.y;
  const int tid = threadIdx.x;
  __shared__ AccSmem sm;

  const int n0 = a.node_offsets[b];
  const int N = a.node_offsets[b + 1] - n0;
  const int V = a.vocab;
  const int W = (V + 31) >> 5;
  const bool logits = a.kind == 1;
  const bool masked = a.mask != nullptr;

  // ---------------------------------------------------------------- phase 0
  if (tid == 0)
    sm.bad = (N < 1 || N > a.max_nodes || N > kMaxN || n0 < 0 || n0 + N > a.total_nodes) ? 1 : 0;
  __syncthreads();
  if (!sm.bad) {
    for (int i = tid; i < N; i += kThreads) {
      const int p = a.parent[n0 + i];
      const int x = a.tokens[n0 + i];
      sm.parent[i] = p;
      sm.token[i] = x;
      sm.u[i] = a.uniforms[n0 + i];
      sm.has_child[i] = 0;
      const bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i && x >= 0 && x < V);
      if (!ok) atomicExch(&sm.bad, 1);
    }
  }
  __syncthreads();
  if (sm.bad) {  // identical decision in every CTA of the cluster
    if (rank == 0) {
      for (int k = tid; k < a.max_nodes; k += kThreads) a.path[(size_t)b * a.max_nodes + k] = -1;
      if (tid == 0) {
        a.accepted_len[b] = -1;
        a.bonus_token[b] = -1;
        a.status[b] = kBadTree;
      }
      if (a.debug_pq && N >= 1 && N <= kMaxN && n0 >= 0 && n0 + N <= a.total_nodes)
        for (int i = tid; i < N; i += kThreads) {
          a.debug_pq[2 * (size_t)(n0 + i)] = 0.0f;
          a.debug_pq[2 * (size_t)(n0 + i) + 1] = 0.0f;
        }
    }
    return;
  }
  for (int i = tid + 1; i < N; i += kThreads) sm.has_child[sm.parent[i]] = 1;
  __syncthreads();

  // p~, q~ of child i of row j (whose LSE / Z are known)
  auto child_pq = [&](int i, int j, float lse, float z) {
    const size_t row = static_cast<size_t>(n0 + j) * V;
    const int x = sm.token[i];
    float p = __ldg(a.target + row + x);
    if (logits) p = expf(p - lse);
    float q = __ldg(a.draft + row + x);
    if (masked) {
      if (mask_bit(a.mask + static_cast<size_t>(n0 + j) * W, x)) {
        p = __fdiv_rn(p, z);
        q = __fdiv_rn(q, z);
      } else {
        p = 0.0f;
        q = 0.0f;
      }
    }
    sm.pq[i][0] = p;
    sm.pq[i][1] = q;
  };

  // Z of row j over [lo, hi): sum of quanta of retained draft mass
  auto row_z_partial = [&](int j, int lo, int hi) -> unsigned long long {
    const size_t rowbase = static_cast<size_t>(n0 + j) * V;
    const uint32_t* mrow = a.mask + static_cast<size_t>(n0 + j) * W;
    unsigned long long acc = 0;
    for_row<false>(a.draft + rowbase, nullptr, rowbase, lo, hi, [&](int v, float q, float) {
      if (mask_bit(mrow, v)) acc += fix40(q);
    });
    return acc;
  };
  auto row_lse_partial = [&](int j, int lo, int hi, float& m, float& s) {
    const size_t rowbase = static_cast<size_t>(n0 + j) * V;
    m = -INFINITY;
    s = 0.0f;
    for_row<false>(a.target + rowbase, nullptr, rowbase, lo, hi,
                   [&](int, float x, float) { lse_push(m, s, x); });
  };
  auto z_from_sum = [](unsigned long long S) -> float {
    return __fmul_rn(__ull2float_rn(S), 9.094947017729282379150390625e-13f);  // * 2^-40
  };

  // ---------------------------------------------------------------- phase 1
  const bool rows_needed = logits || masked;
  if (rows_needed) {
    for (int j = rank; j < N; j += C) {
      if (!sm.has_child[j]) continue;
      float lse = 0.0f, z = 1.0f;
      if (logits) {
        float m, s;
        row_lse_partial(j, 0, V, m, s);
        block_lse(sm, m, s);
        lse = m + logf(s);
      }
      if (masked) z = z_from_sum(block_sum_u64(sm, row_z_partial(j, 0, V)));
      if (tid == 0) {
        sm.row_lse[j] = lse;
        sm.row_z[j] = z;
      }
      for (int i = tid + 1; i < N; i += kThreads)
        if (sm.parent[i] == j) child_pq(i, j, lse, z);
      __syncthreads();
    }
  } else {
    for (int i = tid + 1; i < N; i += kThreads) child_pq(i, sm.parent[i], 0.0f, 1.0f);
  }
  cluster.sync();

  // ---------------------------------------------------------------- phase 2
  float my_p = 0.0f, my_q = 0.0f;
  bool acc = false;
  {
    const int i = tid;  // kThreads == kMaxN: one node per thread
    if (i >= 1 && i < N) {
      const int owner = rows_needed ? (sm.parent[i] % C) : rank;
      const float* src = (owner == rank) ? &sm.pq[i][0] : cluster.map_shared_rank(&sm.pq[i][0], owner);
      my_p = src[0];
      my_q = src[1];
      acc = __fmul_rn(sm.u[i], my_q) < my_p;
    }
    const uint32_t bal = __ballot_sync(0xffffffffu, acc);
    if ((tid & 31) == 0) sm.acc_bits[tid >> 5] = bal;
  }
  __syncthreads();
  {
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
  const int cut = sm.cut;
  const int len = sm.cut_len;
  if (rank == 0) {
    int32_t* path = a.path + static_cast<size_t>(b) * a.max_nodes;
    for (int k = len + tid; k < a.max_nodes; k += kThreads) path[k] = -1;
    if (tid == 0) {
      for (int d = len - 1, v = cut; d >= 0; --d, v = sm.parent[v]) path[d] = v;
      a.accepted_len[b] = len;
      a.bonus_token[b] = -1;  // overwritten by the draw below (ordered by the cluster barriers)
      a.status[b] = kOk;
    }
    if (a.debug_pq && tid < N) {
      a.debug_pq[2 * static_cast<size_t>(n0 + tid)] = my_p;
      a.debug_pq[2 * static_cast<size_t>(n0 + tid) + 1] = my_q;
    }
  }

  // ---------------------------------------------------------------- phase 3
  // LSE / Z of the cut row: from its owner when it has children, else
  // reduced now across the cluster (chunk per CTA, combined in rank order).
  const int chunk = (((V + C - 1) / C) + 3) & ~3;
  const int lo = min(V, rank * chunk), hi = min(V, lo + chunk);
  const bool cut_has_child = sm.has_child[cut] != 0;
  float lse = 0.0f, z = 1.0f;
  if (rows_needed) {
    if (cut_has_child) {
      const int owner = cut % C;
      const float* l = owner == rank ? &sm.row_lse[cut] : cluster.map_shared_rank(&sm.row_lse[cut], owner);
      const float* zz = owner == rank ? &sm.row_z[cut] : cluster.map_shared_rank(&sm.row_z[cut], owner);
      lse = *l;
      z = *zz;
    } else {
      float m = -INFINITY, s = 0.0f;
      unsigned long long zs = 0;
      if (logits) {
        row_lse_partial(cut, lo, hi, m, s);
        block_lse(sm, m, s);
      }
      if (masked) zs = block_sum_u64(sm, row_z_partial(cut, lo, hi));
      if (tid == 0) {
        sm.x_m = m;
        sm.x_s = s;
        sm.x_u64 = zs;
      }
      cluster.sync();
      float M = -INFINITY, Ssum = 0.0f;
      unsigned long long Z = 0;
      for (int c = 0; c < C; ++c) {
        AccSmem* o = cluster.map_shared_rank(&sm, c);
        lse_combine(M, Ssum, o->x_m, o->x_s);
        Z += o->x_u64;
      }
      lse = M + logf(Ssum);
      z = z_from_sum(Z);
      cluster.sync();  // every CTA has read the slots before they are reused
    }
  }

  const size_t crow = static_cast<size_t>(n0 + cut) * V;
  const uint32_t* cmask = masked ? a.mask + static_cast<size_t>(n0 + cut) * W : nullptr;
  // p~_v and q~_v of the cut row
  auto ptil = [&](int v, float t) -> float {
    float p = logits ? expf(t - lse) : t;
    if (masked) p = mask_bit(cmask, v) ? __fdiv_rn(p, z) : 0.0f;
    return p;
  };
  auto qtil = [&](int v, float d) -> float {
    if (masked) return mask_bit(cmask, v) ? __fdiv_rn(d, z) : 0.0f;
    return d;
  };
  auto quanta = [&](int pass, int v, float t, float d) -> unsigned long long {
    const float p = ptil(v, t);
    return fix40(pass == 0 ? __fsub_rn(p, qtil(v, d)) : p);
  };

  const float u0 = sm.u[0];
  int token = -1;
  for (int pass = cut_has_child ? 0 : 1; pass < 2; ++pass) {
    unsigned long long part = 0;
    for_row<true>(a.target + crow, a.draft + crow, crow, lo, hi,
                  [&](int v, float t, float d) { part += quanta(pass, v, t, d); });
    part = block_sum_u64(sm, part);
    if (tid == 0) sm.x_u64 = part;
    cluster.sync();
    unsigned long long S = 0, before = 0;
    for (int c = 0; c < C; ++c) {
      const unsigned long long sc = cluster.map_shared_rank(&sm, c)->x_u64;
      if (c < rank) before += sc;
      S += sc;
    }
    cluster.sync();
    if (S == 0) continue;  // the same decision in every CTA
    const unsigned long long t = scaled_draw(u0, S);
    if (t >= before && t - before < part) {
      // this CTA holds the token: contiguous sub-ranges per thread, block scan
      const unsigned long long tl = t - before;
      const int n = hi - lo;
      const int sub = (n + kThreads - 1) / kThreads;
      const int s0 = lo + min(n, tid * sub), s1 = lo + min(n, (tid + 1) * sub);
      unsigned long long mine = 0;
      for (int v = s0; v < s1; ++v) mine += quanta(pass, v, a.target[crow + v], a.draft[crow + v]);
      // exclusive scan over threads (warp shuffles + per-warp totals)
      unsigned long long inc = mine;
      const int l = tid & 31, w = tid >> 5;
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
        if (l >= o) inc += y;
      }
      __syncthreads();
      if (l == 31) sm.red_u64[w] = inc;
      __syncthreads();
      unsigned long long excl = inc - mine;
      for (int k = 0; k < w; ++k) excl += sm.red_u64[k];
      if (mine > 0 && tl >= excl && tl - excl < mine) {
        unsigned long long cum = excl;
        for (int v = s0; v < s1; ++v) {
          cum += quanta(pass, v, a.target[crow + v], a.draft[crow + v]);
          if (cum > tl) {
            a.bonus_token[b] = v;
            break;
          }
        }
      }
    }
    token = 0;  // found (written by the owning thread)
    break;
  }
  if (token < 0) {
    // no mass at all: smallest index of the largest p~ (NaN ignored)
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for_row<false>(a.target + crow, nullptr, crow, lo, hi, [&](int v, float t, float) {
      const float p = ptil(v, t);
      if (p > bv || (p == bv && v < bi)) {
        bv = p;
        bi = v;
      }
    });
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
        const AccSmem* o = cluster.map_shared_rank(&sm, c);
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

}  // namespace

int launch_accept(const AcceptArgs& a, int cluster_size, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster_size, a.batch, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, accept_kernel, a) == cudaSuccess ? 0 : -1;
}

int accept_max_nodes() { return kMaxN; }

}  // namespace tv
