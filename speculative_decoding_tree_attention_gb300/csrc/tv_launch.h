// tv_launch.h -- argument blocks and launchers shared by the host API and the
// kernels (internal to libtv; not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tv {

struct AcceptArgs {
  const float* target;
  const float* draft;
  const int32_t* tokens;
  const int32_t* parent;
  const int32_t* node_offsets;
  const float* uniforms;
  const uint32_t* mask;
  int32_t* accepted_len;
  int32_t* path;
  int32_t* bonus_token;
  int32_t* status;
  float* debug_pq;
  int32_t vocab;
  int32_t max_nodes;
  int32_t kind;
  int32_t batch;
  int32_t total_nodes;
  int32_t test;          // 0: ratio test, 1: log-space clamped test
  float log_clamp;       // L of the clamped test
  const float* gamma;    // [batch] calibration factors or null (1)
};

// Launches the accept pass; `workspace` holds per-(row, part) statistics (at
// most one part per 8K-entry chunk of the vocabulary) and
// must be accept_workspace_bytes() long when the input is logits or a mask
// is given (it is not touched otherwise).
int launch_accept(const AcceptArgs& a, void* workspace, cudaStream_t stream);

struct RetainArgs {
  const float* draft;          // [rows][vocab]
  uint32_t* mask;              // [rows][ceil(vocab/32)]
  unsigned long long* z_fixed; // [rows] or null
  float* z;                    // [rows] or null
  int32_t* kept;               // [rows] or null
  unsigned long long threshold;// T = floor(mass * 2^40) >= 1
  int32_t rows, vocab;
};

// Retained set of every row (one CTA per row).
int launch_retained_set(const RetainArgs& a, cudaStream_t stream);
size_t accept_workspace_bytes(int vocab, int total_nodes);
int accept_cluster_size(int vocab, int batch, int sms);
int accept_max_nodes();

struct AttnArgs {
  const uint16_t* q;          // [total_nodes][Hq][D]
  const int32_t* block_table; // [batch][max_blocks_per_seq]
  const int32_t* parent;      // [total_nodes]
  const int32_t* prefix_lens; // [batch]
  const int32_t* node_offsets;// [batch+1]
  void* out;                  // [total_nodes][Hq][D], bf16 or fp32 (out_fp32)
  int32_t* status;            // [batch]
  int32_t* counters;          // [ctas][2] ticket and done counters of split units (zeroed per call)
  uint8_t* slots;             // [2 * ctas] partial-result slots of attn_slot_bytes(D)
  int32_t batch, hq, hkv, group, head_dim;
  int32_t max_blocks_per_seq, num_blocks, max_nodes, max_prefix_len, total_nodes;
  int32_t lanes;              // CTAs per virtual CTA: one per m-tile pair of a layer
  int32_t vctas;              // virtual CTAs launched (ctas = vctas * lanes)
  int32_t min_tiles;          // fewest key tiles a virtual CTA is given
  int32_t out_fp32;           // 1: fp32 output, 0: bf16
  float scale_log2;           // softmax scale * log2(e)
  // E4M3 inputs (tv_tree_attention_fp8): q, pools and tree K/V hold codes,
  // each row of D codes with one fp32 scale
  int32_t fp8;
  const float* q_scale;       // [total_nodes][Hq]
  const float* kp_scale;      // [num_blocks][Hkv][16]
  const float* vp_scale;
  const float* kn_scale;      // [total_nodes][Hkv]
  const float* vn_scale;
};

struct AttnMaps {
  CUtensorMap k_pool;   // 5D (64, 8 rows, halves, 2 groups, pages), box = one page, 128B swizzle
  CUtensorMap v_pool;
  CUtensorMap k_nodes;  // 4D (64, nodes, halves, Hkv heads), box = 8 nodes of one head
  CUtensorMap v_nodes;
};

int launch_tree_attention(const AttnArgs& a, const AttnMaps& maps, cudaStream_t stream);
// Bytes of one partial-result slot: 256 rows of fp32 O, (m, l) per row, a flag.
size_t attn_slot_bytes(int head_dim);

struct CommitArgs {
  const uint16_t* k_nodes;    // [total_nodes][Hkv][D]
  const uint16_t* v_nodes;
  const int32_t* parent;      // [total_nodes]
  const int32_t* node_offsets;// [batch+1]
  const int32_t* accepted_len;// [batch]
  const int32_t* path;        // [batch][max_nodes]
  const int32_t* block_table; // [batch][max_blocks_per_seq]
  const int32_t* prefix_lens; // [batch]
  uint16_t* k_pool;           // [num_blocks][Hkv][16][D]
  uint16_t* v_pool;
  int32_t* new_prefix_lens;   // [batch]
  int32_t* status;            // [batch]
  int32_t batch, hkv, head_dim, max_blocks_per_seq, num_blocks, max_nodes, total_nodes;
};

int launch_commit(const CommitArgs& a, cudaStream_t stream);

}  // namespace tv
