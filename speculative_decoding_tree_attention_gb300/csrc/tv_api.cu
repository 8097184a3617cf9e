// tv_api.cu -- the C ABI of libtv (include/tv.h): argument checks on the host,
// launch configuration, TMA tensor maps, and launches on the caller's stream.
// The library allocates nothing and never synchronises.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/tv.h"
#include "tv_device.cuh"
#include "tv_launch.h"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int sm_count() {
  static thread_local int cached_dev = -1, cached_n = 148;
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cached_n;
  if (dev == cached_dev) return cached_n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return cached_n;
  cached_dev = dev;
  cached_n = n;
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct AttnPlan {
  int group;        // query heads per KV head
  int lanes;        // CTAs per virtual CTA (m-tile pairs of one layer)
  int vctas;        // virtual CTAs
  int min_tiles;    // fewest key tiles per virtual CTA
  size_t workspace; // counters + partial-result slots
};

// Fewest 128-key tiles a virtual CTA is given: below this a unit is not split
// further, since a split piece costs about this much in fixed work (its Q
// load, the pipeline fill and its partial-result write).  Timed at 2, 3, 4,
// 5, 6 and 9: only the short-prefix MHA line (32 heads x 9 tiles) moved, and
// 3 was fastest there (each unit then splits into three whole ranges).
constexpr int kMinTiles = 3;

// Launch plan for `sms` SMs (one persistent CTA per SM).  A layer of `lanes`
// CTAs takes the m-tile pairs (256 packed rows) of a (sequence, KV head): as
// many lanes as the largest tree has pairs, so that the CTAs reading the
// same K/V tiles run together.  The virtual CTAs (sms / lanes of them, fewer
// when the host hints bound the work below kMinTiles tiles each) share the
// line of key tiles equally on the device.  Workspace: two arrival counters
// per CTA, then two partial-result slots per CTA.
bool plan_attention(const tv_attn_params* p, int sms, AttnPlan* out) {
  if (!p || sms < 1) return false;
  if (p->batch < 1 || p->num_q_heads < 1 || p->num_kv_heads < 1) return false;
  if (p->num_q_heads % p->num_kv_heads) return false;
  if (p->head_dim != 64 && p->head_dim != 128) return false;
  if (p->block_size != TV_BLOCK_SIZE) return false;
  if (p->max_nodes < 1 || p->max_nodes > TV_MAX_NODES) return false;
  if (p->total_nodes < p->batch || p->num_blocks < 1 || p->max_blocks_per_seq < 1) return false;
  if (p->max_prefix_len < 0) return false;
  if ((p->max_prefix_len + 15) / 16 > p->max_blocks_per_seq) return false;
  if (p->out_dtype != TV_OUT_BF16 && p->out_dtype != TV_OUT_FP32) return false;
  if (static_cast<int64_t>(p->num_blocks) * p->num_kv_heads * 16 >= (1ll << 31)) return false;
  if (static_cast<int64_t>(p->total_nodes) * p->num_q_heads >= (1ll << 31)) return false;
  AttnPlan pl;
  pl.group = p->num_q_heads / p->num_kv_heads;
  const long long mpairs = (static_cast<long long>(p->max_nodes) * pl.group + 255) / 256;
  pl.lanes = static_cast<int>(std::min<long long>(mpairs, sms));
  const long long layers = (mpairs + pl.lanes - 1) / pl.lanes;
  const long long tiles = (p->max_prefix_len + 127) / 128 + (p->max_nodes + 127) / 128;
  const long long wmax = static_cast<long long>(p->batch) * p->num_kv_heads * layers * tiles;
  if (wmax >= (1ll << 31)) return false;  // the device schedule counts tiles in 32 bits
  pl.min_tiles = kMinTiles;
  // at most 4096 virtual CTAs: the device computes range boundaries with
  // fp32 products of v r < 4096^2 = 2^24 (exact integers)
  pl.vctas = static_cast<int>(
      std::max(1ll, std::min<long long>({sms / pl.lanes, wmax / kMinTiles, 4096ll})));
  const size_t ctas = static_cast<size_t>(pl.vctas) * pl.lanes;
  pl.workspace = (ctas * 8 + 255) / 256 * 256 + 2 * ctas * tv::attn_slot_bytes(p->head_dim);
  *out = pl;
  return true;
}

bool encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides_bytes, const cuuint32_t* box,
            CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, type, rank, const_cast<void*>(base), dims,
            strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

const char* tv_status_string(int s) {
  switch (s) {
    case TV_OK: return "TV_OK";
    case TV_ERR_INVALID_ARG: return "TV_ERR_INVALID_ARG";
    case TV_ERR_UNSUPPORTED: return "TV_ERR_UNSUPPORTED";
    case TV_ERR_WORKSPACE: return "TV_ERR_WORKSPACE";
    case TV_ERR_CUDA: return "TV_ERR_CUDA";
    case TV_ERR_BAD_TREE: return "TV_ERR_BAD_TREE";
    case TV_ERR_DEVICE_TIMEOUT: return "TV_ERR_DEVICE_TIMEOUT";
    case TV_ERR_NO_PAGE: return "TV_ERR_NO_PAGE";
    default: return "TV_ERR_UNKNOWN";
  }
}

int tv_version(void) { return TV_VERSION; }

namespace {
// One thread block waits on an mbarrier that nothing arrives at, through the
// kernels' bounded wait, and reports the outcome.
__global__ void selftest_wait_timeout_kernel(int32_t* status, unsigned long long* waited_ns,
                                             unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tv::mbar_init(&bar, 1);
    tv::fence_mbar_init();
  }
  __syncthreads();
  const unsigned long long t0 = tv::global_ns();
  const bool done = tv::mbar_wait(&bar, 0, nullptr, limit_ns);
  if (threadIdx.x == 0) {
    *status = done ? tv::kOk : tv::kDeviceTimeout;
    *waited_ns = tv::global_ns() - t0;
  }
}
}  // namespace

int tv_selftest_wait_timeout(int32_t* status, unsigned long long* waited_ns,
                             unsigned long long limit_ns, cudaStream_t stream) {
  if (!status || !waited_ns) return TV_ERR_INVALID_ARG;
  if (limit_ns < 1000000ull || limit_ns > 1000000000ull) return TV_ERR_INVALID_ARG;
  selftest_wait_timeout_kernel<<<1, 32, 0, stream>>>(status, waited_ns, limit_ns);
  return cudaGetLastError() == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

size_t tv_tree_attention_workspace_size(const tv_attn_params* p) {
  AttnPlan pl;
  if (!plan_attention(p, sm_count(), &pl)) return 0;
  return pl.workspace;
}

int tv_tree_attention_plan(const tv_attn_params* p, int32_t sms, tv_attn_plan* out) {
  if (!out) return TV_ERR_INVALID_ARG;
  AttnPlan pl;
  if (!plan_attention(p, sms > 0 ? sms : sm_count(), &pl)) return TV_ERR_INVALID_ARG;
  out->ctas = pl.vctas * pl.lanes;
  out->lanes = pl.lanes;
  out->virtual_ctas = pl.vctas;
  out->min_tiles = pl.min_tiles;
  out->workspace_bytes = pl.workspace;
  return TV_OK;
}

}  // extern "C"

namespace {

struct Fp8Scales {
  const float *q, *kp, *vp, *kn, *vn;
};

// The shared path of tv_tree_attention and tv_tree_attention_fp8: checks,
// tensor maps, arguments, the status and counter memsets and the launch.
int attention_call(const tv_attn_params* p, const Fp8Scales* f8, const void* q_nodes,
                   const void* k_prefix_blocks, const void* v_prefix_blocks,
                   const int32_t* block_table, const void* k_nodes, const void* v_nodes,
                   const int32_t* parent, const int32_t* prefix_lens,
                   const int32_t* node_offsets, void* out, int32_t* status, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
  if (!p) return TV_ERR_INVALID_ARG;
  if (p->head_dim != 64 && p->head_dim != 128) return TV_ERR_UNSUPPORTED;
  if (f8 && p->head_dim != 128) return TV_ERR_UNSUPPORTED;
  AttnPlan pl;
  if (!plan_attention(p, sm_count(), &pl)) return TV_ERR_INVALID_ARG;
  const void* ptrs[] = {q_nodes, k_prefix_blocks, v_prefix_blocks, block_table, k_nodes,
                        v_nodes, parent, prefix_lens, node_offsets, out, status};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return TV_ERR_INVALID_ARG;
  if (f8) {
    const void* sc[] = {f8->q, f8->kp, f8->vp, f8->kn, f8->vn};
    for (const void* q : sc)
      if (!q || !aligned16(q)) return TV_ERR_INVALID_ARG;
  }
  if (!workspace || workspace_bytes < pl.workspace || !aligned16(workspace))
    return TV_ERR_WORKSPACE;

  const int D = p->head_dim, Hkv = p->num_kv_heads;
  tv::AttnMaps maps;
  std::memset(&maps, 0, sizeof maps);
  if (f8) {
    // E4M3 codes, one byte each, 128-byte rows.  Pool: (128 bytes, 16 rows,
    // pages), box = one page (2 KB).  Tree K/V: (128 bytes, nodes, KV heads),
    // box = 8 nodes of one head (1 KB).  128-byte swizzle.
    const cuuint64_t pdims[3] = {128, 16, static_cast<cuuint64_t>(p->num_blocks) * Hkv};
    const cuuint64_t pstr[2] = {128, 2048};
    const cuuint32_t pbox[3] = {128, 16, 1};
    if (!encode(&maps.k_pool, k_prefix_blocks, 3, pdims, pstr, pbox, CU_TENSOR_MAP_DATA_TYPE_UINT8))
      return TV_ERR_CUDA;
    if (!encode(&maps.v_pool, v_prefix_blocks, 3, pdims, pstr, pbox, CU_TENSOR_MAP_DATA_TYPE_UINT8))
      return TV_ERR_CUDA;
    const cuuint64_t ndims[3] = {128, static_cast<cuuint64_t>(p->total_nodes), static_cast<cuuint64_t>(Hkv)};
    const cuuint64_t nstr[2] = {static_cast<cuuint64_t>(Hkv) * 128, 128};
    const cuuint32_t nbox[3] = {128, 8, 1};
    if (!encode(&maps.k_nodes, k_nodes, 3, ndims, nstr, nbox, CU_TENSOR_MAP_DATA_TYPE_UINT8))
      return TV_ERR_CUDA;
    if (!encode(&maps.v_nodes, v_nodes, 3, ndims, nstr, nbox, CU_TENSOR_MAP_DATA_TYPE_UINT8))
      return TV_ERR_CUDA;
  } else {
    // Paged pool as a 5-D tensor so that one box is one 16-token page of one
    // KV head, landing in shared memory as [8-row group][64-column half][8
    // rows][128 B]: dims (64 columns, 8 rows, halves, 2 row groups, pages),
    // box (64, 8, halves, 2, 1).
    const int halves = D / 64;
    {
      const cuuint64_t dims[5] = {64, 8, static_cast<cuuint64_t>(halves), 2,
                                  static_cast<cuuint64_t>(p->num_blocks) * Hkv};
      const cuuint64_t str[4] = {static_cast<cuuint64_t>(D) * 2, 128,
                                 static_cast<cuuint64_t>(D) * 2 * 8, static_cast<cuuint64_t>(D) * 2 * 16};
      const cuuint32_t box[5] = {64, 8, static_cast<cuuint32_t>(halves), 2, 1};
      if (!encode(&maps.k_pool, k_prefix_blocks, 5, dims, str, box)) return TV_ERR_CUDA;
      if (!encode(&maps.v_pool, v_prefix_blocks, 5, dims, str, box)) return TV_ERR_CUDA;
    }
    // Tree K/V as a 4-D tensor (64 columns, nodes, halves, KV heads); a box
    // is 8 consecutive nodes of one head: [half][8 rows][128 B].
    {
      const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(p->total_nodes),
                                  static_cast<cuuint64_t>(halves), static_cast<cuuint64_t>(Hkv)};
      const cuuint64_t str[3] = {static_cast<cuuint64_t>(D) * 2 * Hkv, 128,
                                 static_cast<cuuint64_t>(D) * 2};
      const cuuint32_t box[4] = {64, 8, static_cast<cuuint32_t>(halves), 1};
      if (!encode(&maps.k_nodes, k_nodes, 4, dims, str, box)) return TV_ERR_CUDA;
      if (!encode(&maps.v_nodes, v_nodes, 4, dims, str, box)) return TV_ERR_CUDA;
    }
  }

  const size_t ctas = static_cast<size_t>(pl.vctas) * pl.lanes;
  tv::AttnArgs a;
  std::memset(&a, 0, sizeof a);
  a.q = static_cast<const uint16_t*>(q_nodes);
  a.block_table = block_table;
  a.parent = parent;
  a.prefix_lens = prefix_lens;
  a.node_offsets = node_offsets;
  a.out = out;
  a.status = status;
  a.counters = static_cast<int32_t*>(workspace);
  a.slots = static_cast<uint8_t*>(workspace) + (ctas * 8 + 255) / 256 * 256;
  a.batch = p->batch;
  a.hq = p->num_q_heads;
  a.hkv = Hkv;
  a.group = pl.group;
  a.head_dim = D;
  a.max_blocks_per_seq = p->max_blocks_per_seq;
  a.num_blocks = p->num_blocks;
  a.max_nodes = p->max_nodes;
  a.max_prefix_len = p->max_prefix_len;
  a.total_nodes = p->total_nodes;
  a.lanes = pl.lanes;
  a.vctas = pl.vctas;
  a.min_tiles = pl.min_tiles;
  a.out_fp32 = p->out_dtype == TV_OUT_FP32 ? 1 : 0;
  const float scale = p->softmax_scale > 0.0f ? p->softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  a.scale_log2 = scale * 1.4426950408889634f;
  if (f8) {
    a.fp8 = 1;
    a.q_scale = f8->q;
    a.kp_scale = f8->kp;
    a.vp_scale = f8->vp;
    a.kn_scale = f8->kn;
    a.vn_scale = f8->vn;
  }

  // status and the arrival counters of split units start at zero
  if (cudaMemsetAsync(status, 0, sizeof(int32_t) * p->batch, stream) != cudaSuccess)
    return TV_ERR_CUDA;
  if (cudaMemsetAsync(a.counters, 0, ctas * 8, stream) != cudaSuccess) return TV_ERR_CUDA;
  if (tv::launch_tree_attention(a, maps, stream) != 0) return TV_ERR_CUDA;
  return TV_OK;
}

}  // namespace

extern "C" {

int tv_tree_attention(const tv_attn_params* p, const uint16_t* q_nodes,
                      const uint16_t* k_prefix_blocks, const uint16_t* v_prefix_blocks,
                      const int32_t* block_table, const uint16_t* k_nodes,
                      const uint16_t* v_nodes, const int32_t* parent,
                      const int32_t* prefix_lens, const int32_t* node_offsets, void* out,
                      int32_t* status, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  return attention_call(p, nullptr, q_nodes, k_prefix_blocks, v_prefix_blocks, block_table,
                        k_nodes, v_nodes, parent, prefix_lens, node_offsets, out, status,
                        workspace, workspace_bytes, stream);
}

int tv_tree_attention_fp8(const tv_attn_params* p, const uint8_t* q_nodes, const float* q_scale,
                          const uint8_t* k_prefix_blocks, const float* k_prefix_scale,
                          const uint8_t* v_prefix_blocks, const float* v_prefix_scale,
                          const int32_t* block_table, const uint8_t* k_nodes,
                          const float* k_nodes_scale, const uint8_t* v_nodes,
                          const float* v_nodes_scale, const int32_t* parent,
                          const int32_t* prefix_lens, const int32_t* node_offsets, void* out,
                          int32_t* status, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
  const Fp8Scales sc = {q_scale, k_prefix_scale, v_prefix_scale, k_nodes_scale, v_nodes_scale};
  return attention_call(p, &sc, q_nodes, k_prefix_blocks, v_prefix_blocks, block_table, k_nodes,
                        v_nodes, parent, prefix_lens, node_offsets, out, status, workspace,
                        workspace_bytes, stream);
}

size_t tv_accept_workspace_size(const tv_accept_params* p) {
  if (!p || p->vocab < 1 || p->vocab >= (1 << 18) || p->total_nodes < 1) return 0;
  return tv::accept_workspace_bytes(p->vocab, p->total_nodes);
}

int tv_accept(const tv_accept_params* p, const float* target, const float* draft_probs,
              const int32_t* draft_tokens, const int32_t* parent, const int32_t* node_offsets,
              const float* uniforms, const uint32_t* retained_mask, int32_t* accepted_len,
              int32_t* path, int32_t* bonus_token, int32_t* status, float* debug_pq,
              void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return tv_accept_ex(p, nullptr, target, draft_probs, draft_tokens, parent, node_offsets,
                      uniforms, retained_mask, accepted_len, path, bonus_token, status, debug_pq,
                      workspace, workspace_bytes, stream);
}

int tv_accept_ex(const tv_accept_params* p, const tv_accept_options* opt, const float* target,
                 const float* draft_probs, const int32_t* draft_tokens, const int32_t* parent,
                 const int32_t* node_offsets, const float* uniforms,
                 const uint32_t* retained_mask, int32_t* accepted_len, int32_t* path,
                 int32_t* bonus_token, int32_t* status, float* debug_pq, void* workspace,
                 size_t workspace_bytes, cudaStream_t stream) {
  if (!p) return TV_ERR_INVALID_ARG;
  if (opt && opt->test != TV_TEST_RATIO && opt->test != TV_TEST_LOG_CLAMP &&
      opt->test != TV_TEST_MULTI)
    return TV_ERR_INVALID_ARG;
  if (opt && !(opt->log_clamp >= 0.0f && opt->log_clamp <= 88.0f)) return TV_ERR_INVALID_ARG;
  if (opt && opt->gamma && !aligned16(opt->gamma)) return TV_ERR_INVALID_ARG;
  if (p->batch < 1 || p->vocab < 1 || p->vocab >= (1 << 18)) return TV_ERR_INVALID_ARG;
  if (p->max_nodes < 1 || p->max_nodes > TV_MAX_NODES || p->max_nodes > tv::accept_max_nodes())
    return TV_ERR_INVALID_ARG;
  if (p->kind != TV_INPUT_PROBS && p->kind != TV_INPUT_LOGITS) return TV_ERR_INVALID_ARG;
  if (p->total_nodes < p->batch) return TV_ERR_INVALID_ARG;
  const void* ptrs[] = {target, draft_probs, draft_tokens, parent, node_offsets, uniforms,
                        accepted_len, path, bonus_token, status};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return TV_ERR_INVALID_ARG;
  if ((retained_mask && !aligned16(retained_mask)) || (debug_pq && !aligned16(debug_pq)))
    return TV_ERR_INVALID_ARG;
  tv::AcceptArgs a;
  a.target = target;
  a.draft = draft_probs;
  a.tokens = draft_tokens;
  a.parent = parent;
  a.node_offsets = node_offsets;
  a.uniforms = uniforms;
  a.mask = retained_mask;
  a.accepted_len = accepted_len;
  a.path = path;
  a.bonus_token = bonus_token;
  a.status = status;
  a.debug_pq = debug_pq;
  a.vocab = p->vocab;
  a.max_nodes = p->max_nodes;
  a.kind = p->kind;
  a.batch = p->batch;
  a.total_nodes = p->total_nodes;
  a.test = opt ? opt->test : TV_TEST_RATIO;
  a.log_clamp = (opt && opt->log_clamp > 0.0f) ? opt->log_clamp : 20.0f;
  a.gamma = opt ? opt->gamma : nullptr;
  // per-row statistics (logits input or a retained-set mask) need workspace
  if (p->kind == TV_INPUT_LOGITS || retained_mask) {
    const size_t need = tv::accept_workspace_bytes(p->vocab, p->total_nodes);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return TV_ERR_WORKSPACE;
  }
  if (tv::launch_accept(a, workspace, stream) != 0) return TV_ERR_CUDA;
  return TV_OK;
}

}  // extern "C"

int tv_commit_kv(const tv_commit_params* p, const uint16_t* k_nodes, const uint16_t* v_nodes,
                 const int32_t* parent, const int32_t* node_offsets, const int32_t* accepted_len,
                 const int32_t* path, const int32_t* block_table, const int32_t* prefix_lens,
                 uint16_t* k_prefix_blocks, uint16_t* v_prefix_blocks, int32_t* new_prefix_lens,
                 int32_t* status, cudaStream_t stream) {
  if (!p) return TV_ERR_INVALID_ARG;
  if (p->head_dim != 64 && p->head_dim != 128) return TV_ERR_UNSUPPORTED;
  if (p->batch < 1 || p->num_kv_heads < 1 || p->block_size != TV_BLOCK_SIZE ||
      p->max_blocks_per_seq < 1 || p->num_blocks < 1 || p->max_nodes < 1 ||
      p->max_nodes > TV_MAX_NODES || p->total_nodes < p->batch)
    return TV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(p->num_blocks) * p->num_kv_heads * 16 >= (1ll << 31))
    return TV_ERR_INVALID_ARG;
  const void* ptrs[] = {k_nodes, v_nodes, parent, node_offsets, accepted_len, path,
                        block_table, prefix_lens, k_prefix_blocks, v_prefix_blocks,
                        new_prefix_lens, status};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return TV_ERR_INVALID_ARG;
  if (static_cast<const void*>(new_prefix_lens) == static_cast<const void*>(prefix_lens))
    return TV_ERR_INVALID_ARG;
  tv::CommitArgs a;
  a.k_nodes = k_nodes;
  a.v_nodes = v_nodes;
  a.parent = parent;
  a.node_offsets = node_offsets;
  a.accepted_len = accepted_len;
  a.path = path;
  a.block_table = block_table;
  a.prefix_lens = prefix_lens;
  a.k_pool = k_prefix_blocks;
  a.v_pool = v_prefix_blocks;
  a.new_prefix_lens = new_prefix_lens;
  a.status = status;
  a.batch = p->batch;
  a.hkv = p->num_kv_heads;
  a.head_dim = p->head_dim;
  a.max_blocks_per_seq = p->max_blocks_per_seq;
  a.num_blocks = p->num_blocks;
  a.max_nodes = p->max_nodes;
  a.total_nodes = p->total_nodes;
  return tv::launch_commit(a, stream) == 0 ? TV_OK : TV_ERR_CUDA;
}

int tv_retained_set(const tv_retain_params* p, const float* draft_probs, uint32_t* retained_mask,
                    uint64_t* z_fixed, float* z, int32_t* kept, cudaStream_t stream) {
  if (!p || p->rows < 1 || p->rows > 65535 || p->vocab < 1 || p->vocab > (1 << 18))
    return TV_ERR_INVALID_ARG;
  if (!(p->mass >= 0x1p-40f && p->mass <= 32.0f)) return TV_ERR_INVALID_ARG;  // NaN fails too
  if (!draft_probs || !retained_mask || !aligned16(draft_probs) || !aligned16(retained_mask))
    return TV_ERR_INVALID_ARG;
  if ((z_fixed && !aligned16(z_fixed)) || (z && !aligned16(z)) || (kept && !aligned16(kept)))
    return TV_ERR_INVALID_ARG;
  tv::RetainArgs a;
  a.draft = draft_probs;
  a.mask = retained_mask;
  a.z_fixed = reinterpret_cast<unsigned long long*>(z_fixed);
  a.z = z;
  a.kept = kept;
  a.threshold = static_cast<unsigned long long>(std::floor(static_cast<double>(p->mass) * 0x1p40));
  a.rows = p->rows;
  a.vocab = p->vocab;
  if (a.threshold < 1) return TV_ERR_INVALID_ARG;
  return tv::launch_retained_set(a, stream) == 0 ? TV_OK : TV_ERR_CUDA;
}
