/*
 * tv.h -- C ABI of libtv: the target-model tree-verification step of
 * speculative decoding, on one GB300 GPU (sm_103a).
 *
 * Sources (four web pages on speculative decoding; titles abbreviated):
 *   [EC]  "端云协同推测解码中草稿模型动态生成与验证并行化：探究树形注意力机制与显存碎片整理联合加速"
 *         (edge-cloud speculative decoding; tree attention; KV defragmentation)
 *   [LLM] "端侧大模型推测解码草稿模型动态剪枝策略：详解基于重要性采样的树形验证并行加速机制"
 *         (on-device LLM draft pruning; importance-sampling correction)
 *   [MM]  "端侧多模态大模型推测解码草稿模型动态剪枝：详解基于重要性采样的树形验证并行加速策略"
 *         (on-device multimodal draft pruning; importance-sampled tree verification)
 *
 * General rules for every entry point
 *   - The caller owns every buffer.  The library allocates nothing, frees
 *     nothing and never synchronises the device or the stream; all work is
 *     enqueued on the caller's stream in order.
 *   - Pointers are DEVICE pointers unless a comment says "host".
 *   - Inputs are read only.  Outputs are fully written when the call returns
 *     TV_OK and the enqueued work completes.
 *   - Argument errors are found on the host and returned before anything is
 *     enqueued.  Data errors found on the device (a bad parent index, an
 *     out-of-range block id or token) are reported per sequence in the
 *     device-side `status` array; the kernels never trap.
 *   - Stateless and re-entrant: concurrent calls on different streams are
 *     safe when their workspaces differ.
 *
 * Tree convention (shared by both entry points)
 *   Sequence b owns tree nodes node_offsets[b] .. node_offsets[b+1]-1 of the
 *   flattened node arrays ([EC] appendix B: cumulative lengths over the
 *   flattened tree).  parent[] holds LOCAL indices (0 .. N_b-1): parent of
 *   the root (local node 0) is -1 and 0 <= parent[i] < i for i >= 1
 *   ([EC] appendix B, Tree_Parent_Idx, -1 at the root).  Node 0 is the last
 *   committed token; nodes >= 1 are draft tokens.
 */
#ifndef TV_H_
#define TV_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

#define TV_VERSION 100     /* 1.0.0 */
#define TV_MAX_NODES 512   /* largest tree (nodes per sequence) */
#define TV_BLOCK_SIZE 16   /* tokens per page of the paged prefix KV pool */

typedef enum {
  TV_OK = 0,
  TV_ERR_INVALID_ARG = 1,    /* null pointer, bad size or layout (host) */
  TV_ERR_UNSUPPORTED = 2,    /* valid but not implemented (e.g. head_dim) */
  TV_ERR_WORKSPACE = 3,      /* workspace missing or smaller than required */
  TV_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed */
  TV_ERR_BAD_TREE = 5,       /* device: malformed tree, block id or token */
  TV_ERR_DEVICE_TIMEOUT = 6, /* device: a bounded wait ran out */
  TV_ERR_NO_PAGE = 7         /* device: no pool page for a position to commit */
} tv_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* tv_status_string(int status);
/* TV_VERSION of the loaded library. */
int tv_version(void);

/* Self-test of the device-timeout path.  Every wait of the library's kernels
 * on an mbarrier is bounded (2 s); when one runs out the kernel records
 * TV_ERR_DEVICE_TIMEOUT in the sequence's status, releases what it holds and
 * returns, so the context stays usable.  This entry point enqueues one
 * kernel that waits on an mbarrier nothing ever arrives at, through the same
 * bounded wait, with the limit `limit_ns` (1 ms .. 1 s), then writes the
 * outcome: status[0] = TV_ERR_DEVICE_TIMEOUT (or TV_OK had the wait ended)
 * and waited_ns[0] = the nanoseconds it waited.  status, waited_ns: device
 * pointers (int32, uint64), 4- and 8-byte aligned.  Returns
 * TV_ERR_INVALID_ARG (nothing enqueued) for a NULL pointer or a limit out of
 * range, TV_ERR_CUDA if the launch fails, else TV_OK. */
int tv_selftest_wait_timeout(int32_t* status, unsigned long long* waited_ns,
                             unsigned long long limit_ns, cudaStream_t stream);

/* ========================================================================
 * Tree attention
 *
 * For every sequence b, tree node i (local) and query head h, with KV head
 * kvh = floor(h / (Hq/Hkv)):
 *
 *   out[n0+i][h] = sum_k softmax_k(scale * q.k_k) * v_k
 *
 * over the key list [prefix tokens 0 .. L_b-1 ; tree nodes j of sequence b]
 * where every prefix token is visible and tree node j is visible iff j is an
 * ancestor of i or j == i: the tree mask M_tree[i,j] = 0 iff j is an ancestor
 * of i or j = i, -inf otherwise ([EC] §2.2.2).  The committed prefix KV is
 * stored once in a paged pool and reached through block_table ([MM] §3.2
 * common-prefix merging; [LLM] §2.3.1 cuSeqLens + block_table).  One launch
 * handles every sequence, every head and every node ([MM] §3.2: one kernel
 * for all branches).  Inputs bf16, accumulation and softmax fp32, output bf16
 * (or fp32, out_dtype).
 * ====================================================================== */
typedef enum { TV_OUT_BF16 = 0, TV_OUT_FP32 = 1 } tv_out_dtype;

typedef struct {
  int32_t batch;              /* B >= 1                                        */
  int32_t num_q_heads;        /* Hq                                            */
  int32_t num_kv_heads;       /* Hkv; Hq % Hkv == 0                            */
  int32_t head_dim;           /* D: 64 or 128                                  */
  int32_t block_size;         /* tokens per page: must be TV_BLOCK_SIZE (16)   */
  int32_t max_blocks_per_seq; /* row stride of block_table                     */
  int32_t num_blocks;         /* pages in the pool                             */
  int32_t max_nodes;          /* upper bound of N_b (<= TV_MAX_NODES)          */
  int32_t total_nodes;        /* node_offsets[batch] (host copy)               */
  int32_t max_prefix_len;     /* upper bound of L_b (host hint for the grid)   */
  float softmax_scale;        /* 0 => 1/sqrt(D)                                */
  int32_t out_dtype;          /* tv_out_dtype of `out`: bf16 (0) or fp32 (1).
                                 The bf16 output is the fp32 result rounded
                                 once to nearest even.                         */
} tv_attn_params;             /* host struct */

/* Bytes of device workspace tv_tree_attention needs for these parameters on
 * the current device (0 if the parameters are invalid).  The workspace holds
 * two arrival counters per CTA (zeroed by every call, on the stream) and two
 * partial-result slots per CTA: when the line of key tiles is cut inside a
 * unit (256 packed rows of one sequence and KV head), every piece but the
 * last to finish leaves its unnormalised output and (max, sum) per row there,
 * and the last merges them in a fixed order.  About 2 * SMs * (256 * D * 4 + 2 KB) bytes: 40.5 MB at
 * D = 128 on 152 SMs. */
size_t tv_tree_attention_workspace_size(const tv_attn_params* params);

/* Launch plan of tv_tree_attention (host only; nothing is enqueued):
 * persistent CTAs (at most one per SM) in virtual CTAs of `lanes` CTAs, one
 * lane per m-tile pair of a layer of a (sequence, KV head); the virtual CTAs
 * share the line of key tiles (sequence, KV head, layer, tile) in equal
 * contiguous ranges of at least min_tiles tiles, computed on the device from
 * prefix_lens and node_offsets. */
typedef struct {
  int32_t ctas;            /* CTAs launched = virtual_ctas * lanes          */
  int32_t lanes;           /* CTAs per virtual CTA                          */
  int32_t virtual_ctas;    /* at most SMs / lanes                           */
  int32_t min_tiles;       /* fewest 128-key tiles per virtual CTA          */
  size_t workspace_bytes;  /* = tv_tree_attention_workspace_size on `sms`   */
} tv_attn_plan;

/* The plan for `sms` SMs (sms <= 0: the current device's count, 148 when no
 * device is visible).  Returns TV_OK, or TV_ERR_INVALID_ARG for invalid
 * parameters or a NULL `plan`. */
int tv_tree_attention_plan(const tv_attn_params* params, int32_t sms, tv_attn_plan* plan);

/* Layouts (all row-major, contiguous):
 *   q_nodes          bf16 [total_nodes][Hq][D]
 *   k_prefix_blocks  bf16 [num_blocks][Hkv][block_size][D]   (paged pool)
 *   v_prefix_blocks  bf16 [num_blocks][Hkv][block_size][D]
 *   block_table      int32 [batch][max_blocks_per_seq]: page of logical block
 *                    t/16 of sequence b; entries past ceil(L_b/16) unused
 *   k_nodes, v_nodes bf16 [total_nodes][Hkv][D]   (K/V of the tree tokens)
 *   parent           int32 [total_nodes]  local parent, -1 at each root
 *   prefix_lens      int32 [batch]        L_b >= 0 (<= max_prefix_len)
 *   node_offsets     int32 [batch+1]      cumulative node counts, N_b >= 1
 *   out              bf16 or fp32 (out_dtype) [total_nodes][Hq][D]
 *   status           int32 [batch]        per-sequence TV_OK / TV_ERR_BAD_TREE /
 *                                         TV_ERR_DEVICE_TIMEOUT (device)
 *   workspace        device bytes >= tv_tree_attention_workspace_size()
 *                    (TV_ERR_WORKSPACE otherwise); contents need no
 *                    initialisation; calls that overlap on the GPU need
 *                    distinct workspaces
 * bf16 pointers are passed as uint16_t (bf16 bit patterns).  All device
 * pointers must be 16-byte aligned.  A sequence whose tree or block ids are
 * malformed gets status TV_ERR_BAD_TREE and an all-zero output. */
int tv_tree_attention(const tv_attn_params* params, const uint16_t* q_nodes,
                      const uint16_t* k_prefix_blocks, const uint16_t* v_prefix_blocks,
                      const int32_t* block_table, const uint16_t* k_nodes,
                      const uint16_t* v_nodes, const int32_t* parent,
                      const int32_t* prefix_lens, const int32_t* node_offsets, void* out,
                      int32_t* status, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream);

/* ------------------------------------------------------------------------
 * FP8 tree attention ([EC] §9.2: FP8 mixed-precision tree verification,
 * E4M3 values with fp32 accumulation and one scale per 128-element block).
 *
 * The same attention as tv_tree_attention (same mask, key list, layouts of
 * the index arrays, output, status and workspace), on E4M3 inputs: q_nodes,
 * the pools and the tree K/V hold one-byte E4M3 codes (OCP layout: bias 7,
 * subnormals, NaN at S.1111.111, no infinities), and every row of D codes
 * (a token of one head: the 128-element block at D = 128) carries one fp32
 * scale; the value is code x scale.  head_dim must be 128
 * (TV_ERR_UNSUPPORTED otherwise).
 *   q_nodes          u8 [total_nodes][Hq][128],        q_scale fp32 [total_nodes][Hq]
 *   k_prefix_blocks  u8 [num_blocks][Hkv][16][128],    k_prefix_scale fp32 [num_blocks][Hkv][16]
 *   v_prefix_blocks  u8 [num_blocks][Hkv][16][128],    v_prefix_scale fp32 [num_blocks][Hkv][16]
 *   k_nodes, v_nodes u8 [total_nodes][Hkv][128],       k_nodes_scale, v_nodes_scale fp32 [total_nodes][Hkv]
 * Arithmetic: S = Q K^T on the tensor cores over the codes (E4M3 x E4M3,
 * fp32 accumulation), each score times its query row's and key row's scale;
 * fp32 online softmax; each V row converted to fp16 as code x scale (the
 * exact product rounded once), P rounded to fp16 (the row sum adds the
 * rounded values), P V in fp16 with fp32 accumulation.  The dequantised V
 * values must lie in the fp16 range (|code x scale| <= 65504, i.e. a V scale
 * of at most 146 for codes up to 448); larger ones become infinite.  All
 * device pointers 16-byte aligned (the scale arrays 4-byte). */
int tv_tree_attention_fp8(const tv_attn_params* params, const uint8_t* q_nodes,
                          const float* q_scale, const uint8_t* k_prefix_blocks,
                          const float* k_prefix_scale, const uint8_t* v_prefix_blocks,
                          const float* v_prefix_scale, const int32_t* block_table,
                          const uint8_t* k_nodes, const float* k_nodes_scale,
                          const uint8_t* v_nodes, const float* v_nodes_scale,
                          const int32_t* parent, const int32_t* prefix_lens,
                          const int32_t* node_offsets, void* out, int32_t* status,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Tree attention for callers that cannot allocate (no counterpart on the
 * pages: an engineering addition of this library).
 *
 * Same inputs, outputs, layouts, semantics and status codes as
 * tv_tree_attention, but no workspace argument: the device scratch the plan
 * needs (tv_tree_attention_workspace_size: arrival counters and
 * partial-result slots) comes from a fixed device array inside the library,
 * so a caller that may not call cudaMalloc (code running under stream
 * capture, an operator inside an engine that owns all device memory, a
 * service that forbids allocation after start-up) can still use it.  This
 * entry point allocates nothing and calls no allocating routine.
 *   - The array is TV_NO_ALLOC_SCRATCH_BYTES (64 MiB) of device memory; every
 *     GPU on which this entry point runs holds it until the process exits.
 *   - A call whose scratch would not fit
 *     (tv_tree_attention_workspace_size(params) > TV_NO_ALLOC_SCRATCH_BYTES)
 *     returns TV_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and keeps it for the
 *     life of the process; make that first call before any stream capture on
 *     the device, and do not reset the device's primary context afterwards.
 *   - Every call uses the same array and it keeps the last call's contents;
 *     the arrival counters that must start at zero are cleared by each call
 *     on its stream.  Calls that overlap on the GPU (other streams, other host
 *     threads) race on the array: serialise them. */
#define TV_NO_ALLOC_SCRATCH_BYTES (64u << 20)
int tv_tree_attention_no_alloc(const tv_attn_params* params, const uint16_t* q_nodes,
                               const uint16_t* k_prefix_blocks, const uint16_t* v_prefix_blocks,
                               const int32_t* block_table, const uint16_t* k_nodes,
                               const uint16_t* v_nodes, const int32_t* parent,
                               const int32_t* prefix_lens, const int32_t* node_offsets,
                               void* out, int32_t* status, cudaStream_t stream);

/* ========================================================================
 * Fused accept pass ([EC] §2.2.3; [LLM] §2.2.1-§2.2.2, §7.1)
 *
 * Per tree b, for every draft node i >= 1 with parent j:
 *   p = target probability of token x_i in row j (probs given, or softmax of
 *       the logits row, fp32), q = draft probability of x_i in row j.
 *   Pruning renormalisation when retained_mask is given: on the retained set
 *   R_j, p~ = p / Z_j and q~ = q / Z_j (log space: add log(1/Z_j)); off R_j
 *   p~ = q~ = 0 (log space: -inf).  Z_j = the retained draft mass, summed
 *   exactly in 2^-40 fixed point and rounded once to fp32.  Without a mask
 *   p~ = p, q~ = q.
 *   Test: a_i = fl32(u_i * q~) < p~  (u < min(1, p~/q~), strict, NaN rejects).
 * Walk: the deepest node whose whole root path is accepted (cut at the first
 *   rejection), ties to the smallest index; accepted_len = its depth.
 * Bonus token: from the cut node j*: if j* has children, the residual
 *   max(0, p~ - q~) of row j*; if it is a leaf or the residual is all zero,
 *   p~ of row j*; if that is all zero too, the smallest index of max p~.
 *   The draw is an exact inverse CDF in 2^-40 fixed point: quanta
 *   f_v = floor(min(r_v, 32) * 2^40), S = sum f_v (uint64),
 *   t = floor(u_0 * S), token = min v with f_0 + .. + f_v > t.
 * ====================================================================== */
typedef enum { TV_INPUT_PROBS = 0, TV_INPUT_LOGITS = 1 } tv_input_kind;

typedef struct {
  int32_t batch;        /* B >= 1                                           */
  int32_t vocab;        /* V, 1 <= V < 2^18                                 */
  int32_t max_nodes;    /* row stride of `path`; >= every N_b, <= TV_MAX_NODES */
  int32_t total_nodes;  /* node_offsets[batch] (host copy)                  */
  int32_t kind;         /* tv_input_kind: the form of `target`              */
} tv_accept_params;     /* host struct */

/* Bytes of device workspace tv_accept needs when the target rows are logits
 * or a retained_mask is given (per-row partial statistics); with
 * probabilities and no mask the workspace may be NULL. */
size_t tv_accept_workspace_size(const tv_accept_params* params);

/* Layouts:
 *   target        fp32 [total_nodes][V]  row j = target next-token
 *                 probabilities (or logits) after node j
 *   draft_probs   fp32 [total_nodes][V]  row j = draft probabilities after node j
 *   draft_tokens  int32 [total_nodes]    token of node i (node 0 unused)
 *   parent, node_offsets                 as for tree attention
 *   uniforms      fp32 [total_nodes]     u_i in [0,1) tests node i >= 1;
 *                                        u at each root is the bonus draw u_0
 *   retained_mask uint32 [total_nodes][ceil(V/32)] or NULL: bit v%32 of word
 *                 v/32 of row j set iff v is in R_j
 *   accepted_len  int32 [batch]          accepted draft tokens (-1 on error)
 *   path          int32 [batch][max_nodes]: local ids of the accepted path at
 *                 depths 1..accepted_len, then -1
 *   bonus_token   int32 [batch]          (-1 on error)
 *   status        int32 [batch]
 *   debug_pq      fp32 [total_nodes][2] or NULL: (p~, q~) used by the test of
 *                 each node (0, 0 at roots)
 *   workspace     device bytes >= tv_accept_workspace_size() for logits input
 *                 or with a mask (else may be NULL)
 * All device pointers 16-byte aligned; V * 4 a multiple of 16 is not required. */
int tv_accept(const tv_accept_params* params, const float* target, const float* draft_probs,
              const int32_t* draft_tokens, const int32_t* parent, const int32_t* node_offsets,
              const float* uniforms, const uint32_t* retained_mask, int32_t* accepted_len,
              int32_t* path, int32_t* bonus_token, int32_t* status, float* debug_pq,
              void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Accept-test variants (tv_accept_ex; tv_accept is tv_accept_ex with NULL
 * options, i.e. TV_TEST_RATIO and no calibration factor):
 *   TV_TEST_RATIO      a_i = fl32(u_i * q~) < fl32(gamma_b * p~): the test
 *                      u < min(1, gamma * p/q) with the calibration factor of
 *                      [MM] §3.3 (gamma = exp(-lambda KL) computed by the
 *                      caller, one per sequence; gamma = 1 is the plain test).
 *   TV_TEST_LOG_CLAMP  the log-space test of [LLM] §10.2:
 *                      r = clamp(log p~ - log q~ + log gamma_b, -L, L) in fp32,
 *                      a_i = u_i < (r >= 0 ? 1 : exp(r)); p~ = 0 or a NaN r
 *                      rejects (a pruned token never passes).
 * For these two the walk and the bonus draw are unchanged (the residual
 * max(0, p~ - q~)).
 *   TV_TEST_MULTI      multi-candidate verification with residual updates
 *                      (multi-step speculative sampling of SpecInfer, which
 *                      the pages cite; the pages only say "resample at the
 *                      rejection"): from the root, the children c of the
 *                      current node j are tried in increasing index order
 *                      against the current target distribution cur (at first
 *                      p~_j): accept iff fl32(u_c * q~_j(x_c)) <
 *                      fl32(gamma_b * cur(x_c)), and the first accepted child
 *                      becomes the current node.  A rejection replaces cur by
 *                      fl32(r / N) with r = max(0, fl32(cur - q~_j)) and N the
 *                      fp32 of the exact 2^-40 fixed-point sum of r (cur is
 *                      kept when that sum is 0).  When every child of the
 *                      final node is rejected, the bonus is drawn from the
 *                      last r (from cur when its sum is 0); at a leaf from p~.
 *                      On a chain it decides exactly as TV_TEST_RATIO.
 *                      debug_pq holds (cur(x_c), q~(x_c)) of the tested
 *                      children and zeros for untested nodes.
 * gamma: device fp32 [batch] or NULL (1); a gamma_b that is not a positive
 * finite number gives that sequence TV_ERR_BAD_TREE.  log_clamp: L, 0 => 20. */
typedef enum { TV_TEST_RATIO = 0, TV_TEST_LOG_CLAMP = 1, TV_TEST_MULTI = 2 } tv_accept_test;

typedef struct {
  int32_t test;        /* tv_accept_test                                 */
  float log_clamp;     /* L for TV_TEST_LOG_CLAMP, 0 => 20; at most 88    */
  const float* gamma;  /* device fp32 [batch] calibration factors, or NULL */
} tv_accept_options;   /* host struct */

int tv_accept_ex(const tv_accept_params* params, const tv_accept_options* options,
                 const float* target, const float* draft_probs, const int32_t* draft_tokens,
                 const int32_t* parent, const int32_t* node_offsets, const float* uniforms,
                 const uint32_t* retained_mask, int32_t* accepted_len, int32_t* path,
                 int32_t* bonus_token, int32_t* status, float* debug_pq, void* workspace,
                 size_t workspace_bytes, cudaStream_t stream);

/* ========================================================================
 * Retained set of the draft rows (the step before the accept pass's pruning
 * renormalisation; [LLM] §2.1.2 soft truncation by cumulative probability
 * mass, [LLM] §7.1 the same decision in log space).
 *
 * For every row r of draft_probs, with key_v = q_v if q_v > 0 else 0 (NaN
 * and negatives count as 0) and the fixed-point quantum
 * f_v = floor(min(key_v, 32) * 2^40) used by tv_accept:
 *   order the tokens by key desc, id asc; R_r = the shortest prefix of that
 *   order whose sum of f_v reaches T = floor(mass * 2^40), or every token if
 *   no prefix does (the crossing token is kept; ties go to the lower id).
 * Outputs: retained_mask bit v%32 of word v/32 of row r set iff v in R_r
 * (the layout tv_accept takes), and optionally z_fixed[r] = sum of f_v over
 * R_r (exact, uint64), z[r] = z_fixed[r] * 2^-40 rounded once to fp32 (the
 * Z that tv_accept divides by), kept[r] = |R_r|.  Every sum is an exact
 * integer: the result does not depend on the reduction order.
 * ====================================================================== */
typedef struct {
  int32_t rows;   /* R >= 1                                                */
  int32_t vocab;  /* V, 1 <= V <= 2^18                                     */
  float mass;     /* retained mass, 1 - Prune_Ratio: 2^-40 <= mass <= 32   */
} tv_retain_params; /* host struct */

/* Layouts: draft_probs fp32 [rows][V]; retained_mask uint32 [rows][ceil(V/32)];
 * z_fixed uint64 [rows], z fp32 [rows], kept int32 [rows] (each optional,
 * NULL to skip).  Device pointers 16-byte aligned. */
int tv_retained_set(const tv_retain_params* params, const float* draft_probs,
                    uint32_t* retained_mask, uint64_t* z_fixed, float* z, int32_t* kept,
                    cudaStream_t stream);

/* ========================================================================
 * Commit of the accepted path ([MM] §9.1 item 2: the target KV cache is
 * preallocated and tree-node KV is written into it by a scatter kernel;
 * [LLM] §2.3.2: pool slots only for the unique accepted path; [EC] §5.2:
 * the prefix cache grows incrementally by the accepted path).
 *
 * For every sequence b with accepted_len a = accepted_len[b] >= 0 and
 * prefix length L = prefix_lens[b]: the root (local node 0, the token
 * committed by the previous step, whose K/V this step computed) and the
 * accepted nodes path[b][0..a-1] become committed tokens at positions
 * L, L+1, .., L+a.  For every KV head, the K and V rows of node v
 * (k_nodes/v_nodes row n0 + v) are copied to row pos % 16 of pool page
 * block_table[b][pos / 16] (layouts as for tree attention), and
 * new_prefix_lens[b] = L + a + 1; status[b] = TV_OK.
 * A sequence is left untouched (new_prefix_lens[b] = L, nothing written) with
 *   TV_ERR_BAD_TREE if a < 0 (its accept pass failed), a >= N_b, its tree
 *     extent is malformed, or path[b][d] is not a child of path[b][d-1]
 *     (path[b][-1] = the root);
 *   TV_ERR_NO_PAGE if a position L..L+a has no page (block id < 0 or >=
 *     num_blocks, or past max_blocks_per_seq): the caller's allocator
 *     provides the pages before the call.
 * Every output is written by the call: status and new_prefix_lens need no
 * initialisation.  new_prefix_lens must not alias prefix_lens.  Positions
 * L..L+a of every listed page must not be read by other work in flight.
 * ====================================================================== */
typedef struct {
  int32_t batch;              /* B >= 1                                      */
  int32_t num_kv_heads;       /* Hkv                                         */
  int32_t head_dim;           /* D: 64 or 128                                */
  int32_t block_size;         /* must be TV_BLOCK_SIZE (16)                  */
  int32_t max_blocks_per_seq; /* row stride of block_table                   */
  int32_t num_blocks;         /* pages in the pool                           */
  int32_t max_nodes;          /* row stride of path; >= every N_b            */
  int32_t total_nodes;        /* node_offsets[batch] (host copy)             */
} tv_commit_params;           /* host struct */

/* Layouts: k_nodes, v_nodes bf16 [total_nodes][Hkv][D]; parent, node_offsets,
 * accepted_len, path as produced for / by tv_accept; block_table int32
 * [batch][max_blocks_per_seq]; prefix_lens, new_prefix_lens, status int32
 * [batch]; k_prefix_blocks, v_prefix_blocks bf16 [num_blocks][Hkv][16][D]
 * (written).  All device pointers 16-byte aligned. */
int tv_commit_kv(const tv_commit_params* params, const uint16_t* k_nodes,
                 const uint16_t* v_nodes, const int32_t* parent, const int32_t* node_offsets,
                 const int32_t* accepted_len, const int32_t* path, const int32_t* block_table,
                 const int32_t* prefix_lens, uint16_t* k_prefix_blocks, uint16_t* v_prefix_blocks,
                 int32_t* new_prefix_lens, int32_t* status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* TV_H_ */
