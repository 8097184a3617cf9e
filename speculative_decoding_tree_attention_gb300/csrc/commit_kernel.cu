// commit_kernel.cu -- commit of the accepted path into the paged KV pool.
//
// Sources (titles abbreviated):
//   [MM]  "端侧多模态大模型推测解码草稿模型动态剪枝：详解基于重要性采样的树形验证并行加速策略":
//         §9.1 item 2, the target KV cache is preallocated and the KV of tree
//         nodes is written into it by a scatter kernel.
//   [LLM] "端侧大模型推测解码草稿模型动态剪枝策略：详解基于重要性采样的树形验证并行加速机制":
//         §2.3.2, pool slots are taken only for the unique accepted path.
//   [EC]  "端云协同推测解码中草稿模型动态生成与验证并行化：探究树形注意力机制与显存碎片整理联合加速":
//         §5.2, the prefix cache grows incrementally by the accepted path.
//
// One CTA per (sequence, KV head).  The root (the token committed by the
// previous step, whose K/V this step computed) and the accepted path become
// positions L .. L+a of the sequence: every CTA of the sequence checks the
// path against the parent array and the pages of those positions (the same
// decision everywhere), then copies its head's rows in 16-byte pieces.  The
// head-0 CTA writes the status and the new prefix length, so no output needs
// initialising.
#include "tv_device.cuh"
#include "tv_launch.h"

namespace tv {
namespace {

constexpr int kCommitThreads = 128;
constexpr int kNoPage = 7;

__global__ void __launch_bounds__(kCommitThreads) commit_kernel(const CommitArgs a) {
  const int b = blockIdx.x, kvh = blockIdx.y, tid = threadIdx.x;
  __shared__ int s_bad, s_nopage;
  const int n0 = a.node_offsets[b];
  const int N = a.node_offsets[b + 1] - n0;
  const int acc = a.accepted_len[b];
  const int L = a.prefix_lens[b];
  if (tid == 0) {
    s_bad = (N < 1 || N > a.max_nodes || n0 < 0 || n0 + N > a.total_nodes || acc < 0 ||
             acc >= N || L < 0) ? 1 : 0;
    s_nopage = 0;
  }
  __syncthreads();
  const int32_t* path = a.path + static_cast<size_t>(b) * a.max_nodes;
  const int32_t* btab = a.block_table + static_cast<size_t>(b) * a.max_blocks_per_seq;
  if (!s_bad) {
    // the path runs down from the root: path[d] is a child of path[d-1]
    for (int d = tid; d < acc; d += kCommitThreads) {
      const int v = path[d];
      const int prev = d == 0 ? 0 : path[d - 1];
      if (v < 1 || v >= N || a.parent[n0 + v] != prev) atomicOr(&s_bad, 1);
    }
    // every position L .. L+acc has a page
    const long long last = static_cast<long long>(L) + acc;
    for (long long pg = L / 16 + tid; pg <= last / 16; pg += kCommitThreads) {
      const int blk = pg < a.max_blocks_per_seq ? btab[pg] : -1;
      if (blk < 0 || blk >= a.num_blocks) atomicOr(&s_nopage, 1);
    }
  }
  __syncthreads();
  const int code = s_bad ? kBadTree : (s_nopage ? kNoPage : kOk);
  if (kvh == 0 && tid == 0) {
    a.status[b] = code;
    a.new_prefix_lens[b] = code == kOk ? L + acc + 1 : L;
  }
  if (code != kOk) return;
  // (acc + 1) tokens x {K, V} x D/8 pieces of 16 bytes
  const int pieces = a.head_dim / 8;
  const int items = (acc + 1) * 2 * pieces;
  for (int it = tid; it < items; it += kCommitThreads) {
    const int c = it % pieces;
    const int kv = (it / pieces) & 1;
    const int t = it / (2 * pieces);
    const int v = t == 0 ? 0 : path[t - 1];
    const int pos = L + t;
    const int blk = btab[pos / 16];
    const uint4* src = reinterpret_cast<const uint4*>(
        (kv ? a.v_nodes : a.k_nodes) + (static_cast<size_t>(n0 + v) * a.hkv + kvh) * a.head_dim) + c;
    uint4* dst = reinterpret_cast<uint4*>(
        (kv ? a.v_pool : a.k_pool) +
        ((static_cast<size_t>(blk) * a.hkv + kvh) * 16 + pos % 16) * a.head_dim) + c;
    *dst = __ldg(src);
  }
}

}  // namespace

int launch_commit(const CommitArgs& a, cudaStream_t stream) {
  commit_kernel<<<dim3(a.batch, a.hkv), kCommitThreads, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace tv
