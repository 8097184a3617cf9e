"""Tree verification for speculative decoding on GB300 (sm_103a).

Thin Python binding over the C-ABI library ``libtv.so`` (declared in
``include/tv.h``): argument marshalling only.  Every step of the computation
runs in the library's CUDA kernels; there is no CPU or PyTorch fallback, and
the functions raise if the library cannot be loaded.

PyTorch is used for device memory and the current CUDA stream only.

    tree_attention(...)  -> out, status      (tv_tree_attention)
    tree_attention_fp8(...) -> out, status   (tv_tree_attention_fp8, E4M3 inputs)
    accept(...)          -> dict of outputs  (tv_accept)
    commit_kv(...)       -> new_prefix_lens, status (tv_commit_kv)
    retained_set(...)    -> mask, z_fixed, z, kept (tv_retained_set)
"""
from __future__ import annotations

import ctypes as C
import os

__all__ = ["TVError", "load", "tree_attention", "tree_attention_fp8", "accept", "commit_kv", "retained_set",
           "attention_workspace_size", "attention_plan", "attention_params",
           "TV_MAX_NODES", "TV_OK", "TV_ERR_BAD_TREE", "TV_ERR_DEVICE_TIMEOUT", "TV_ERR_NO_PAGE",
           "status_string"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libtv.so")

TV_OK = 0
TV_ERR_INVALID_ARG = 1
TV_ERR_UNSUPPORTED = 2
TV_ERR_WORKSPACE = 3
TV_ERR_CUDA = 4
TV_ERR_BAD_TREE = 5
TV_ERR_DEVICE_TIMEOUT = 6
TV_ERR_NO_PAGE = 7
TV_MAX_NODES = 512
TV_BLOCK_SIZE = 16
EXPORTS = ("tv_status_string", "tv_version", "tv_tree_attention_workspace_size",
           "tv_tree_attention", "tv_accept_workspace_size", "tv_accept", "tv_accept_ex",
           "tv_commit_kv",
           "tv_retained_set", "tv_selftest_wait_timeout", "tv_tree_attention_plan",
           "tv_tree_attention_no_alloc", "tv_tree_attention_fp8")


class TVError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


class AttnParams(C.Structure):
    _fields_ = [("batch", C.c_int32), ("num_q_heads", C.c_int32), ("num_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("block_size", C.c_int32),
                ("max_blocks_per_seq", C.c_int32), ("num_blocks", C.c_int32),
                ("max_nodes", C.c_int32), ("total_nodes", C.c_int32),
                ("max_prefix_len", C.c_int32), ("softmax_scale", C.c_float),
                ("out_dtype", C.c_int32)]


class AttnPlan(C.Structure):
    _fields_ = [("ctas", C.c_int32), ("lanes", C.c_int32), ("virtual_ctas", C.c_int32),
                ("min_tiles", C.c_int32), ("workspace_bytes", C.c_size_t)]


class AcceptParams(C.Structure):
    _fields_ = [("batch", C.c_int32), ("vocab", C.c_int32), ("max_nodes", C.c_int32),
                ("total_nodes", C.c_int32), ("kind", C.c_int32)]


class AcceptOptions(C.Structure):
    _fields_ = [("test", C.c_int32), ("log_clamp", C.c_float), ("gamma", C.c_void_p)]


class RetainParams(C.Structure):
    _fields_ = [("rows", C.c_int32), ("vocab", C.c_int32), ("mass", C.c_float)]


class CommitParams(C.Structure):
    _fields_ = [("batch", C.c_int32), ("num_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("block_size", C.c_int32), ("max_blocks_per_seq", C.c_int32),
                ("num_blocks", C.c_int32), ("max_nodes", C.c_int32), ("total_nodes", C.c_int32)]


_lib = None


def load(path: str | None = None) -> C.CDLL:
    """Loads libtv.so (built in-tree by ``_build.build()``); raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise OSError(f"libtv.so not found at {p}: build it with "
                      "speculative_decoding_tree_attention_gb300._build.build()")
    lib = C.CDLL(p)
    vp, sz = C.c_void_p, C.c_size_t
    lib.tv_status_string.argtypes = [C.c_int]
    lib.tv_status_string.restype = C.c_char_p
    lib.tv_version.restype = C.c_int
    lib.tv_tree_attention_workspace_size.argtypes = [C.POINTER(AttnParams)]
    lib.tv_tree_attention_workspace_size.restype = sz
    lib.tv_tree_attention.argtypes = [C.POINTER(AttnParams)] + [vp] * 11 + [vp, sz, vp]
    lib.tv_tree_attention.restype = C.c_int
    lib.tv_tree_attention_fp8.argtypes = [C.POINTER(AttnParams)] + [vp] * 16 + [vp, sz, vp]
    lib.tv_tree_attention_fp8.restype = C.c_int
    lib.tv_accept_workspace_size.argtypes = [C.POINTER(AcceptParams)]
    lib.tv_accept_workspace_size.restype = sz
    lib.tv_accept.argtypes = [C.POINTER(AcceptParams)] + [vp] * 12 + [vp, sz, vp]
    lib.tv_accept.restype = C.c_int
    lib.tv_accept_ex.argtypes = [C.POINTER(AcceptParams), C.c_void_p] + [vp] * 12 + [vp, sz, vp]
    lib.tv_accept_ex.restype = C.c_int
    lib.tv_tree_attention_no_alloc.argtypes = [C.POINTER(AttnParams)] + [vp] * 11 + [vp]
    lib.tv_tree_attention_no_alloc.restype = C.c_int
    lib.tv_selftest_wait_timeout.argtypes = [vp, vp, C.c_ulonglong, vp]
    lib.tv_selftest_wait_timeout.restype = C.c_int
    lib.tv_tree_attention_plan.argtypes = [C.POINTER(AttnParams), C.c_int32, C.POINTER(AttnPlan)]
    lib.tv_tree_attention_plan.restype = C.c_int
    lib.tv_commit_kv.argtypes = [C.POINTER(CommitParams)] + [vp] * 12 + [vp]
    lib.tv_commit_kv.restype = C.c_int
    lib.tv_retained_set.argtypes = [C.POINTER(RetainParams)] + [vp] * 5 + [vp]
    lib.tv_retained_set.restype = C.c_int
    if path is None:
        _lib = lib
    return lib


def status_string(code: int) -> str:
    try:
        return load().tv_status_string(int(code)).decode()
    except OSError:
        return {0: "TV_OK", 1: "TV_ERR_INVALID_ARG", 2: "TV_ERR_UNSUPPORTED",
                3: "TV_ERR_WORKSPACE", 4: "TV_ERR_CUDA", 5: "TV_ERR_BAD_TREE",
                6: "TV_ERR_DEVICE_TIMEOUT", 7: "TV_ERR_NO_PAGE"}.get(int(code), "TV_ERR_UNKNOWN")


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _check_dev(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


OUT_DTYPES = {"bf16": 0, "fp32": 1}


def attention_params(q_nodes, k_prefix_blocks, block_table, prefix_lens, *, num_kv_heads,
                     max_nodes, max_prefix_len, softmax_scale=0.0, out_dtype="bf16") -> AttnParams:
    total, hq, d = q_nodes.shape
    nb = k_prefix_blocks.shape[0]
    return AttnParams(int(prefix_lens.shape[0]), int(hq), int(num_kv_heads), int(d),
                      int(k_prefix_blocks.shape[2]), int(block_table.shape[1]), int(nb),
                      int(max_nodes), int(total), int(max_prefix_len), float(softmax_scale),
                      OUT_DTYPES[out_dtype])


def attention_workspace_size(params: AttnParams) -> int:
    return int(load().tv_tree_attention_workspace_size(C.byref(params)))


def attention_plan(params: AttnParams, sms: int = 0) -> dict:
    """tv_tree_attention_plan: the launch plan for `sms` SMs (0: the current
    device).  Raises TVError for invalid parameters."""
    plan = AttnPlan()
    rc = load().tv_tree_attention_plan(C.byref(params), int(sms), C.byref(plan))
    if rc != TV_OK:
        raise TVError(rc, "tv_tree_attention_plan")
    return {k: int(getattr(plan, k)) for k, _ in AttnPlan._fields_}


def tree_attention(q_nodes, k_prefix_blocks, v_prefix_blocks, block_table, k_nodes, v_nodes,
                   parent, prefix_lens, node_offsets, *, max_nodes: int, max_prefix_len: int,
                   softmax_scale: float = 0.0, out=None, status=None, workspace=None,
                   stream=None, out_dtype: str = "bf16"):
    """tv_tree_attention on the current stream.  Shapes as in include/tv.h:
    q_nodes [total, Hq, D] bf16; k/v_prefix_blocks [num_blocks, Hkv, 16, D] bf16;
    block_table [B, max_blocks] int32; k/v_nodes [total, Hkv, D] bf16;
    parent [total] int32; prefix_lens [B] int32; node_offsets [B+1] int32.
    out_dtype "bf16" or "fp32" (the output tensor's type).
    Returns (out, status); nothing is synchronised."""
    import torch
    lib = load()
    _check_dev(q_nodes, k_prefix_blocks, v_prefix_blocks, block_table, k_nodes, v_nodes,
               parent, prefix_lens, node_offsets)
    prm = attention_params(q_nodes, k_prefix_blocks, block_table, prefix_lens,
                           num_kv_heads=k_prefix_blocks.shape[1], max_nodes=max_nodes,
                           max_prefix_len=max_prefix_len, softmax_scale=softmax_scale,
                           out_dtype=out_dtype)
    if out is None:
        out = torch.empty(q_nodes.shape, device=q_nodes.device,
                          dtype=torch.float32 if out_dtype == "fp32" else torch.bfloat16)
    if status is None:
        status = torch.empty(prm.batch, dtype=torch.int32, device=q_nodes.device)
    need = int(lib.tv_tree_attention_workspace_size(C.byref(prm)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_nodes.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.tv_tree_attention(C.byref(prm), _ptr(q_nodes), _ptr(k_prefix_blocks),
                               _ptr(v_prefix_blocks), _ptr(block_table), _ptr(k_nodes),
                               _ptr(v_nodes), _ptr(parent), _ptr(prefix_lens),
                               _ptr(node_offsets), _ptr(out), _ptr(status), _ptr(workspace),
                               C.c_size_t(ws_bytes), _stream(stream))
    if rc != TV_OK:
        raise TVError(rc, "tv_tree_attention")
    return out, status


def tree_attention_fp8(q_codes, q_scale, k_prefix_blocks, k_prefix_scale, v_prefix_blocks,
                       v_prefix_scale, block_table, k_nodes, k_nodes_scale, v_nodes,
                       v_nodes_scale, parent, prefix_lens, node_offsets, *, max_nodes: int,
                       max_prefix_len: int, softmax_scale: float = 0.0, out=None, status=None,
                       workspace=None, stream=None, out_dtype: str = "bf16"):
    """tv_tree_attention_fp8 on the current stream: E4M3 codes (uint8) with one
    fp32 scale per row of D = 128 codes.  q_codes [total, Hq, 128],
    q_scale [total, Hq]; k/v_prefix_blocks [num_blocks, Hkv, 16, 128],
    k/v_prefix_scale [num_blocks, Hkv, 16]; k/v_nodes [total, Hkv, 128],
    k/v_nodes_scale [total, Hkv]; the index arrays as for tree_attention.
    Returns (out, status); nothing is synchronised."""
    import torch
    lib = load()
    _check_dev(q_codes, q_scale, k_prefix_blocks, k_prefix_scale, v_prefix_blocks,
               v_prefix_scale, block_table, k_nodes, k_nodes_scale, v_nodes, v_nodes_scale,
               parent, prefix_lens, node_offsets)
    prm = attention_params(q_codes, k_prefix_blocks, block_table, prefix_lens,
                           num_kv_heads=k_prefix_blocks.shape[1], max_nodes=max_nodes,
                           max_prefix_len=max_prefix_len, softmax_scale=softmax_scale,
                           out_dtype=out_dtype)
    if out is None:
        out = torch.empty(q_codes.shape, device=q_codes.device,
                          dtype=torch.float32 if out_dtype == "fp32" else torch.bfloat16)
    if status is None:
        status = torch.empty(prm.batch, dtype=torch.int32, device=q_codes.device)
    need = int(lib.tv_tree_attention_workspace_size(C.byref(prm)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_codes.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.tv_tree_attention_fp8(C.byref(prm), _ptr(q_codes), _ptr(q_scale),
                                   _ptr(k_prefix_blocks), _ptr(k_prefix_scale),
                                   _ptr(v_prefix_blocks), _ptr(v_prefix_scale), _ptr(block_table),
                                   _ptr(k_nodes), _ptr(k_nodes_scale), _ptr(v_nodes),
                                   _ptr(v_nodes_scale), _ptr(parent), _ptr(prefix_lens),
                                   _ptr(node_offsets), _ptr(out), _ptr(status), _ptr(workspace),
                                   C.c_size_t(ws_bytes), _stream(stream))
    if rc != TV_OK:
        raise TVError(rc, "tv_tree_attention_fp8")
    return out, status


def tree_attention_no_alloc(q_nodes, k_prefix_blocks, v_prefix_blocks, block_table, k_nodes,
                            v_nodes, parent, prefix_lens, node_offsets, *, max_nodes: int,
                            max_prefix_len: int, softmax_scale: float = 0.0, out=None,
                            status=None, stream=None):
    """tv_tree_attention_no_alloc: as tree_attention, for callers that cannot
    allocate device memory; any device scratch the launch plan needs comes
    from a fixed device array owned by the library (see include/tv.h).  Output
    tensors must be supplied by a caller that cannot allocate; they are
    created here only for convenience."""
    import torch
    lib = load()
    _check_dev(q_nodes, k_prefix_blocks, v_prefix_blocks, block_table, k_nodes, v_nodes,
               parent, prefix_lens, node_offsets)
    prm = attention_params(q_nodes, k_prefix_blocks, block_table, prefix_lens,
                           num_kv_heads=k_prefix_blocks.shape[1], max_nodes=max_nodes,
                           max_prefix_len=max_prefix_len, softmax_scale=softmax_scale)
    if out is None:
        out = torch.empty_like(q_nodes)
    if status is None:
        status = torch.empty(prm.batch, dtype=torch.int32, device=q_nodes.device)
    rc = lib.tv_tree_attention_no_alloc(C.byref(prm), _ptr(q_nodes), _ptr(k_prefix_blocks),
                                        _ptr(v_prefix_blocks), _ptr(block_table), _ptr(k_nodes),
                                        _ptr(v_nodes), _ptr(parent), _ptr(prefix_lens),
                                        _ptr(node_offsets), _ptr(out), _ptr(status),
                                        _stream(stream))
    if rc != TV_OK:
        raise TVError(rc, "tv_tree_attention_no_alloc")
    return out, status


def accept(target, draft_probs, draft_tokens, parent, node_offsets, uniforms,
           retained_mask=None, *, max_nodes: int, kind: str = "probs", debug_pq: bool = False,
           outputs: dict | None = None, stream=None, test: str = "ratio", log_clamp: float = 0.0,
           gamma=None) -> dict:
    """tv_accept_ex on the current stream.  target/draft_probs [total, V] fp32,
    draft_tokens/parent [total] int32, node_offsets [B+1] int32, uniforms
    [total] fp32, retained_mask [total, ceil(V/32)] int32/uint32 or None.
    test: "ratio" (fl32(u q~) < fl32(gamma p~)), "log_clamp" (the clamped
    log-space test, bound log_clamp, 0 => 20) or "multi" (siblings tried in
    order with residual updates); gamma: [B] fp32 CUDA tensor of calibration
    factors or None (1).
    Returns dict(accepted_len, path, bonus_token, status, debug_pq)."""
    import torch
    lib = load()
    _check_dev(target, draft_probs, draft_tokens, parent, node_offsets, uniforms, retained_mask)
    total, V = target.shape
    B = node_offsets.shape[0] - 1
    dev = target.device
    prm = AcceptParams(int(B), int(V), int(max_nodes), int(total),
                       1 if kind == "logits" else 0)
    o = outputs or {}
    acc = o.get("accepted_len")
    if acc is None:
        acc = torch.empty(B, dtype=torch.int32, device=dev)
    path = o.get("path")
    if path is None:
        path = torch.empty(B, max_nodes, dtype=torch.int32, device=dev)
    bonus = o.get("bonus_token")
    if bonus is None:
        bonus = torch.empty(B, dtype=torch.int32, device=dev)
    status = o.get("status")
    if status is None:
        status = torch.empty(B, dtype=torch.int32, device=dev)
    dpq = o.get("debug_pq")
    if dpq is None and debug_pq:
        dpq = torch.empty(total, 2, dtype=torch.float32, device=dev)
    ws = o.get("workspace")
    if ws is None and (kind == "logits" or retained_mask is not None):
        need = int(lib.tv_accept_workspace_size(C.byref(prm)))
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check_dev(gamma)
    tests = {"ratio": 0, "log_clamp": 1, "multi": 2}
    if test not in tests:
        raise ValueError("test must be 'ratio', 'log_clamp' or 'multi'")
    opts = AcceptOptions(tests[test], float(log_clamp), None if gamma is None else gamma.data_ptr())
    rc = lib.tv_accept_ex(C.byref(prm), C.byref(opts), _ptr(target), _ptr(draft_probs), _ptr(draft_tokens),
                       _ptr(parent), _ptr(node_offsets), _ptr(uniforms), _ptr(retained_mask),
                       _ptr(acc), _ptr(path), _ptr(bonus), _ptr(status), _ptr(dpq), _ptr(ws),
                       C.c_size_t(ws_bytes), _stream(stream))
    if rc != TV_OK:
        raise TVError(rc, "tv_accept")
    return dict(accepted_len=acc, path=path, bonus_token=bonus, status=status, debug_pq=dpq)


def selftest_wait_timeout(limit_ms: float = 10.0, stream=None):
    """tv_selftest_wait_timeout: a device wait that nothing ends, bounded by
    limit_ms.  Returns (status, waited_ns) after synchronising."""
    import torch
    lib = load()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    rc = lib.tv_selftest_wait_timeout(_ptr(status), _ptr(waited), C.c_ulonglong(int(limit_ms * 1e6)),
                                      _stream(stream))
    if rc != TV_OK:
        raise TVError(rc, "tv_selftest_wait_timeout")
    torch.cuda.synchronize()
    return int(status.item()), int(waited.item())


def commit_kv(k_nodes, v_nodes, parent, node_offsets, accepted_len, path, block_table,
              prefix_lens, k_prefix_blocks, v_prefix_blocks, *, max_nodes: int,
              new_prefix_lens=None, status=None, stream=None):
    """tv_commit_kv on the current stream: writes the root and the accepted
    path of every sequence into the paged pool (k/v_prefix_blocks, in place).
    Shapes as in include/tv.h; path [B, max_nodes] from accept().
    Returns (new_prefix_lens, status); nothing is synchronised."""
    import torch
    lib = load()
    _check_dev(k_nodes, v_nodes, parent, node_offsets, accepted_len, path, block_table,
               prefix_lens, k_prefix_blocks, v_prefix_blocks)
    total, hkv, d = k_nodes.shape
    B = int(node_offsets.shape[0] - 1)
    prm = CommitParams(B, int(hkv), int(d), int(k_prefix_blocks.shape[2]),
                       int(block_table.shape[1]), int(k_prefix_blocks.shape[0]), int(max_nodes),
                       int(total))
    dev = k_nodes.device
    if new_prefix_lens is None:
        new_prefix_lens = torch.empty(B, dtype=torch.int32, device=dev)
    if status is None:
        status = torch.empty(B, dtype=torch.int32, device=dev)
    rc = lib.tv_commit_kv(C.byref(prm), _ptr(k_nodes), _ptr(v_nodes), _ptr(parent),
                          _ptr(node_offsets), _ptr(accepted_len), _ptr(path), _ptr(block_table),
                          _ptr(prefix_lens), _ptr(k_prefix_blocks), _ptr(v_prefix_blocks),
                          _ptr(new_prefix_lens), _ptr(status), _stream(stream))
    if rc != TV_OK:
        raise TVError(rc, "tv_commit_kv")
    return new_prefix_lens, status


def retained_set(draft_probs, mass: float, *, mask=None, z_fixed=None, z=None, kept=None,
                 stream=None):
    """tv_retained_set on the current stream: draft_probs [R, V] fp32.
    Returns (mask [R, ceil(V/32)] int32 bit patterns, z_fixed [R] int64
    (uint64 bits), z [R] fp32, kept [R] int32); nothing is synchronised."""
    import torch
    lib = load()
    _check_dev(draft_probs)
    R, V = draft_probs.shape
    dev = draft_probs.device
    if mask is None:
        mask = torch.empty(R, (V + 31) // 32, dtype=torch.int32, device=dev)
    if z_fixed is None:
        z_fixed = torch.empty(R, dtype=torch.int64, device=dev)
    if z is None:
        z = torch.empty(R, dtype=torch.float32, device=dev)
    if kept is None:
        kept = torch.empty(R, dtype=torch.int32, device=dev)
    prm = RetainParams(int(R), int(V), float(mass))
    rc = lib.tv_retained_set(C.byref(prm), _ptr(draft_probs), _ptr(mask), _ptr(z_fixed), _ptr(z),
                             _ptr(kept), _stream(stream))
    if rc != TV_OK:
        raise TVError(rc, "tv_retained_set")
    return mask, z_fixed, z, kept
