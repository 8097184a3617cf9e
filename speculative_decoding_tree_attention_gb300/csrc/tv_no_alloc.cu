// tv_no_alloc.cu -- tree attention for callers that cannot allocate device
// memory.
//
// Some callers have no way to hand the library a workspace: code that runs
// while a CUDA graph is being captured (where cudaMalloc is not allowed), a
// plugin or custom operator inside an engine that owns all device memory and
// offers no scratch API, or a service that forbids allocation after start-up
// so that latency and memory use stay fixed.  tv_tree_attention_no_alloc
// serves them: it takes the same inputs and outputs as tv_tree_attention, but
// no workspace.  Whatever device scratch a launch plan asks for
// (tv_tree_attention_workspace_size) comes from a fixed array that lives in
// the library itself, so nothing is allocated at call time.
//
// The array below is TV_NO_ALLOC_SCRATCH_BYTES of device memory.  Each GPU on
// which this entry point is used holds it from the first call until the
// process exits.  Calls whose plan needs more than that are rejected with
// TV_ERR_WORKSPACE before anything is enqueued.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/tv.h"

namespace {

// Device scratch of tv_tree_attention_no_alloc, shared by every call.
static __device__ __align__(256) unsigned char tv_no_alloc_scratch[TV_NO_ALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_lock;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  Looked up once
// per device (the host-side name of the array is only a stand-in and must
// never be passed to a kernel).  Returns TV_OK or TV_ERR_CUDA.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TV_ERR_CUDA;
  std::lock_guard<std::mutex> guard(g_setup_lock);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, tv_no_alloc_scratch) != cudaSuccess || !p) return TV_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return TV_OK;
}

}  // namespace

extern "C" int tv_tree_attention_no_alloc(const tv_attn_params* params, const uint16_t* q_nodes,
                                          const uint16_t* k_prefix_blocks,
                                          const uint16_t* v_prefix_blocks,
                                          const int32_t* block_table, const uint16_t* k_nodes,
                                          const uint16_t* v_nodes, const int32_t* parent,
                                          const int32_t* prefix_lens,
                                          const int32_t* node_offsets, void* out,
                                          int32_t* status, cudaStream_t stream) {
  if (!params) return TV_ERR_INVALID_ARG;
  const size_t need = tv_tree_attention_workspace_size(params);
  if (need > static_cast<size_t>(TV_NO_ALLOC_SCRATCH_BYTES)) return TV_ERR_WORKSPACE;
  // The arrival counters at the start of the array must be zero: the call
  // below clears them on the stream before its kernel runs.  The partial
  // results are written by the kernel before any merge reads them.
  void* scratch = nullptr;
  if (need > 0) {
    const int rc = scratch_address(&scratch);
    if (rc != TV_OK) return rc;
  }
  return tv_tree_attention(params, q_nodes, k_prefix_blocks, v_prefix_blocks, block_table,
                           k_nodes, v_nodes, parent, prefix_lens, node_offsets, out, status,
                           scratch, need > 0 ? static_cast<size_t>(TV_NO_ALLOC_SCRATCH_BYTES) : 0,
                           stream);
}
