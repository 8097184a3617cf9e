"""fp64 CPU oracle for tree verification -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the package smoke check and the benchmark's CPU-baseline
leg import this module.  The product path (the C-ABI library and its binding)
never imports, links or calls it, and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, pthreads); this file
compiles it with gcc and marshals numpy arrays through ctypes.  See the header
of ``oracle.c`` for what is computed and which passage of the pages each step
follows.  The one step without arithmetic, the commit of the accepted path
(a copy by definition), is written out here with numpy: ``commit_kv``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (no fast math, no fp contraction)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(
                ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                 "-shared", "-pthread", _SRC, "-o", tmp, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


class _AttnArgs(C.Structure):
    _fields_ = [
        ("batch", C.c_int), ("num_q_heads", C.c_int), ("num_kv_heads", C.c_int),
        ("head_dim", C.c_int), ("block_size", C.c_int), ("max_blocks_per_seq", C.c_int),
        ("scale", C.c_double),
        ("q", C.c_void_p), ("k_prefix", C.c_void_p), ("v_prefix", C.c_void_p),
        ("block_table", C.c_void_p), ("k_nodes", C.c_void_p), ("v_nodes", C.c_void_p),
        ("parent", C.c_void_p), ("prefix_lens", C.c_void_p), ("node_offsets", C.c_void_p),
        ("dtype", C.c_int),
        ("q_scale", C.c_void_p), ("k_prefix_scale", C.c_void_p), ("v_prefix_scale", C.c_void_p),
        ("k_nodes_scale", C.c_void_p), ("v_nodes_scale", C.c_void_p),
    ]


class _AcceptArgs(C.Structure):
    _fields_ = [
        ("batch", C.c_int), ("vocab", C.c_int), ("kind", C.c_int), ("max_nodes", C.c_int),
        ("target", C.c_void_p), ("draft_probs", C.c_void_p), ("draft_tokens", C.c_void_p),
        ("parent", C.c_void_p), ("node_offsets", C.c_void_p), ("uniforms", C.c_void_p),
        ("retained_mask", C.c_void_p),
        ("accepted_len", C.c_void_p), ("path", C.c_void_p), ("bonus_token", C.c_void_p),
        ("status", C.c_void_p), ("pq_out", C.c_void_p),
        ("test", C.c_int), ("log_clamp", C.c_float), ("gamma", C.c_void_p),
    ]


def _load():
    global _lib
    if _lib is None:
        lib = C.CDLL(build())
        lib.oracle_tree_attention_rows.argtypes = [C.POINTER(_AttnArgs), C.c_int, C.c_void_p,
                                                   C.c_void_p, C.c_int]
        lib.oracle_tree_attention_rows.restype = C.c_int
        lib.oracle_accept.argtypes = [C.POINTER(_AcceptArgs), C.c_int]
        lib.oracle_accept.restype = C.c_int
        lib.oracle_quantise.argtypes = [C.c_float]
        lib.oracle_quantise.restype = C.c_uint64
        lib.oracle_scaled_draw.argtypes = [C.c_float, C.c_uint64]
        lib.oracle_scaled_draw.restype = C.c_uint64
        lib.oracle_retained_mass_row.argtypes = [C.c_void_p, C.c_void_p, C.c_int]
        lib.oracle_retained_mass_row.restype = C.c_float
        lib.oracle_retained_set_row.argtypes = [C.c_void_p, C.c_int, C.c_uint64, C.c_void_p,
                                                C.POINTER(C.c_uint64), C.POINTER(C.c_float),
                                                C.POINTER(C.c_int)]
        lib.oracle_retained_set_row.restype = C.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def tree_attention_rows(case: dict, rows, nthreads: int | None = None) -> np.ndarray:
    """fp64 outputs for the listed (b, local node, q head) rows -> [len(rows), D].
    Inputs are bf16 bit patterns, or, when case["dtype"] == "e4m3", E4M3 codes
    (uint8) with fp32 row scales case["<name>_scale"] (one per row of D)."""
    lib = _load()
    e4m3 = case.get("dtype", "bf16") == "e4m3"
    names = ("q", "k_prefix", "v_prefix", "k_nodes", "v_nodes")
    keep = {k: _c(case[k], np.uint8 if e4m3 else np.uint16) for k in names}
    scales = {k: (_c(case[k + "_scale"], np.float32) if e4m3 else None) for k in names}
    for k in ("block_table", "parent", "prefix_lens", "node_offsets"):
        keep[k] = _c(case[k], np.int32)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    hq, hkv, d = case["num_q_heads"], case["num_kv_heads"], case["head_dim"]
    scale = case.get("softmax_scale") or 1.0 / np.sqrt(d)
    args = _AttnArgs(int(case["batch"]), int(hq), int(hkv), int(d), int(case["block_size"]),
                     int(keep["block_table"].shape[1]), float(scale),
                     *[_ptr(keep[k]) for k in ("q", "k_prefix", "v_prefix", "block_table",
                                               "k_nodes", "v_nodes", "parent", "prefix_lens",
                                               "node_offsets")],
                     1 if e4m3 else 0, *[_ptr(scales[k]) for k in names])
    out = np.zeros((rows.shape[0], d), dtype=np.float64)
    rc = lib.oracle_tree_attention_rows(C.byref(args), rows.shape[0], _ptr(rows), _ptr(out),
                                        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_tree_attention_rows: unsupported arguments")
    return out


def all_rows(case: dict) -> np.ndarray:
    """Every (b, i, h) row in output order ([total_nodes][Hq])."""
    off = np.asarray(case["node_offsets"])
    hq = case["num_q_heads"]
    rows = []
    for b in range(case["batch"]):
        for i in range(off[b + 1] - off[b]):
            for h in range(hq):
                rows.append((b, i, h))
    return np.asarray(rows, dtype=np.int32).reshape(-1, 3)


def tree_attention(case: dict, nthreads: int | None = None) -> np.ndarray:
    """Full fp64 output [total_nodes][Hq][D]."""
    rows = all_rows(case)
    out = tree_attention_rows(case, rows, nthreads)
    tot = int(np.asarray(case["node_offsets"])[-1])
    return out.reshape(tot, case["num_q_heads"], case["head_dim"])


def accept(case: dict, nthreads: int | None = None, want_pq: bool = True, test: int = 0,
           log_clamp: float = 20.0, gamma=None) -> dict:
    """Oracle accept pass.  Returns accepted_len, path, bonus_token, status, pq.
    test 0: ratio test with calibration factors `gamma` ([batch] fp32, None = 1);
    test 1: the log-space clamped test with bound `log_clamp`;
    test 2: the multi-candidate walk (siblings in order, residual updates)."""
    lib = _load()
    off = _c(case["node_offsets"], np.int32)
    batch = off.shape[0] - 1
    tot = int(off[-1])
    max_nodes = int(case["max_nodes"])
    keep = {
        "target": _c(case["target"], np.float32),
        "draft_probs": _c(case["draft_probs"], np.float32),
        "draft_tokens": _c(case["draft_tokens"], np.int32),
        "parent": _c(case["parent"], np.int32),
        "uniforms": _c(case["uniforms"], np.float32),
        "retained_mask": _c(case.get("retained_mask"), np.uint32),
        "gamma": None if gamma is None else _c(gamma, np.float32),
    }
    out = {
        "accepted_len": np.zeros(batch, np.int32),
        "path": np.zeros((batch, max_nodes), np.int32),
        "bonus_token": np.zeros(batch, np.int32),
        "status": np.zeros(batch, np.int32),
        "pq": np.zeros((max(tot, 1), 2), np.float32) if want_pq else None,
    }
    kind = 1 if case.get("kind", "probs") == "logits" else 0
    args = _AcceptArgs(batch, int(case["vocab"]), kind, max_nodes,
                       _ptr(keep["target"]), _ptr(keep["draft_probs"]), _ptr(keep["draft_tokens"]),
                       _ptr(keep["parent"]), _ptr(off), _ptr(keep["uniforms"]),
                       _ptr(keep["retained_mask"]),
                       _ptr(out["accepted_len"]), _ptr(out["path"]), _ptr(out["bonus_token"]),
                       _ptr(out["status"]), _ptr(out["pq"]), int(test), float(log_clamp),
                       _ptr(keep["gamma"]))
    rc = lib.oracle_accept(C.byref(args), int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_accept: unsupported arguments")
    return out


def e4m3_value(code: int) -> float:
    """The oracle's decoding of one E4M3 code."""
    lib = _load()
    lib.oracle_e4m3_to_f64.restype = C.c_double
    lib.oracle_e4m3_to_f64.argtypes = [C.c_uint8]
    return float(lib.oracle_e4m3_to_f64(code))


def quantise(r: float) -> int:
    return int(_load().oracle_quantise(C.c_float(r)))


def scaled_draw(u: float, S: int) -> int:
    return int(_load().oracle_scaled_draw(C.c_float(u), C.c_uint64(S)))


def retained_mass(q_row, mask_row) -> float:
    q = _c(q_row, np.float32)
    m = None if mask_row is None else _c(mask_row, np.uint32)
    return float(_load().oracle_retained_mass_row(_ptr(q), _ptr(m), int(q.shape[0])))


def commit_kv(k_nodes, v_nodes, parent, node_offsets, accepted_len, path, block_table,
              prefix_lens, k_pool, v_pool, max_nodes):
    """Commit of the accepted path, by definition (multimodal page §9.1 item 2:
    tree-node KV scattered into the preallocated target KV cache; on-device
    LLM page §2.3.2: slots only for the unique accepted path; edge-cloud page
    §5.2: the prefix cache grows by the accepted path).

    For each sequence b with a = accepted_len[b] and L = prefix_lens[b]: the
    root (local node 0) and path[b][0..a-1] become positions L .. L+a; the K
    and V rows of those nodes (every KV head) go to row pos % 16 of page
    block_table[b][pos // 16].  Status 5 (malformed: a < 0, a >= N, a bad
    extent, or a path step that is not a child of the previous node) or 7 (a
    position without a page) leaves the sequence untouched.  Arrays are numpy
    (bf16 as uint16 bit patterns).  Returns (k_pool, v_pool, new_prefix_lens,
    status) as new arrays."""
    k_pool = np.array(k_pool, copy=True)
    v_pool = np.array(v_pool, copy=True)
    off = np.asarray(node_offsets, np.int64)
    B = off.shape[0] - 1
    total = int(np.asarray(k_nodes).shape[0])
    num_blocks = k_pool.shape[0]
    table = np.asarray(block_table)
    new_lens = np.array(prefix_lens, np.int32, copy=True)
    status = np.zeros(B, np.int32)
    for b in range(B):
        n0, N = int(off[b]), int(off[b + 1] - off[b])
        a, L = int(accepted_len[b]), int(prefix_lens[b])
        ok = 1 <= N <= max_nodes and n0 >= 0 and n0 + N <= total and 0 <= a < N and L >= 0
        nodes = [0]
        if ok:
            for d in range(a):
                v = int(path[b][d])
                if not (1 <= v < N and int(parent[n0 + v]) == nodes[-1]):
                    ok = False
                    break
                nodes.append(v)
        if not ok:
            status[b] = 5
            continue
        pages = []
        for t in range(a + 1):
            pg = (L + t) // 16
            blk = int(table[b][pg]) if pg < table.shape[1] else -1
            if not 0 <= blk < num_blocks:
                break
            pages.append(blk)
        if len(pages) < a + 1:
            status[b] = 7
            continue
        for t, (v, blk) in enumerate(zip(nodes, pages)):
            k_pool[blk, :, (L + t) % 16, :] = k_nodes[n0 + v]
            v_pool[blk, :, (L + t) % 16, :] = v_nodes[n0 + v]
        new_lens[b] = L + a + 1
    return k_pool, v_pool, new_lens, status


def retained_threshold(mass: float) -> int:
    """T = floor(mass * 2^40) for an fp32 mass (exact in fp64)."""
    return int(np.floor(float(np.float32(mass)) * 2.0 ** 40))


def retained_set(q_rows, mass: float):
    """Retained set of every row of q_rows [R][V] fp32 (see oracle.c,
    oracle_retained_set_row).  Returns (mask [R][ceil(V/32)] uint32,
    z_fixed [R] uint64, z [R] fp32 = z_fixed * 2^-40 rounded once, kept [R])."""
    q = _c(np.atleast_2d(q_rows), np.float32)
    R, V = q.shape
    T = retained_threshold(mass)
    masks = np.zeros((R, (V + 31) // 32), np.uint32)
    zf = np.zeros(R, np.uint64)
    z32 = np.zeros(R, np.float32)
    kept = np.zeros(R, np.int32)
    lib = _load()
    for r in range(R):
        z = C.c_uint64(0)
        zs = C.c_float(0.0)
        k = C.c_int(0)
        row = np.ascontiguousarray(q[r])
        mrow = np.zeros((V + 31) // 32, np.uint32)
        if lib.oracle_retained_set_row(_ptr(row), int(V), C.c_uint64(T), _ptr(mrow), C.byref(z),
                                       C.byref(zs), C.byref(k)) != 0:
            raise ValueError("oracle_retained_set_row: bad arguments")
        masks[r] = mrow
        zf[r] = z.value
        z32[r] = zs.value
        kept[r] = k.value
    return masks, zf, z32, kept
