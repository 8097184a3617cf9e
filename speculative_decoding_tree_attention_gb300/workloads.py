"""Seeded synthetic inputs for tree verification (input generation only).

This module builds the inputs that both the CUDA path and the CPU oracle
consume: random bf16 Q/K/V, paged prefix pools with block tables, draft trees,
target/draft distributions, uniforms and retained-set masks.  It contains none
of the verification arithmetic (no attention, no acceptance test, no walk, no
sampling): it only draws numbers and shapes them.

Every tensor comes from its own NumPy Philox stream,
``Generator(Philox(SeedSequence([config_seed, stream, ...])))``, so a case is a
pure function of (config, seed, overrides).

The five workloads follow the shapes the pages' workloads imply (see the
``CONFIGS`` table).  Notation: ``normal(0, var)`` below means variance ``var``.

Tree shapes
  * ``binary``: the full binary tree of depth 3 (15 nodes), parent(i) = (i-1)//2.
  * ``topk``: breadth-first growth; every node shallower than ``depth`` gets
    k ~ U{1..kmax} children, the k most probable tokens of its draft row, until
    ``n`` nodes exist; if every branch reaches the depth limit first, nodes in
    discovery order get their next most probable tokens (up to kmax children)
    until ``n`` nodes exist.
  * ``importance``: the importance-sampled tree of the on-device multimodal
    pruning page (§3.1): each node offers the top-8 draft tokens of its retained
    set, weighted w_i = p_i^beta / sum_j p_j^beta with beta = 0.6; nodes are
    added best-first by Gumbel-perturbed path log-weight (sampling without
    replacement), up to ``n`` nodes and depth 8.
  Nodes are then numbered breadth-first with siblings in descending draft
  probability, so parent(i) < i and node 0 is the root (the last committed
  token, never tested).
"""
from __future__ import annotations

import heapq

import numpy as np

# stream ids (one per tensor family)
_S_TREE, _S_Q, _S_KP, _S_VP, _S_KN, _S_VN, _S_TABLE, _S_LEN, _S_ROWS, _S_UNI, _S_GUMBEL, _S_EXT = range(12)

CONFIGS = {
    1: dict(name="tiny", batch=1, hq=4, hkv=4, d=64, prefix=(128, 128), tree="binary", n=(15, 15),
            depth=3, kmax=2, vocab=1000, target_var=2.0, draft="independent", draft_var=2.0,
            shuffle=False, mask_mass=None),
    2: dict(name="7b_like", batch=1, hq=32, hkv=32, d=128, prefix=(1024, 1024), tree="topk",
            n=(64, 64), depth=6, kmax=4, vocab=32000, target_var=2.0, draft="noise",
            draft_var=0.5, shuffle=False, mask_mass=None),
    3: dict(name="serving", batch=16, hq=32, hkv=8, d=128, prefix=(512, 4096), tree="topk",
            n=(26, 64), depth=5, kmax=4, vocab=32000, target_var=2.0, draft="noise",
            draft_var=0.5, shuffle=True, mask_mass=None),
    4: dict(name="multimodal", batch=4, hq=28, hkv=4, d=128, prefix=(1600, 1600),
            image_tokens=576, image_std=2.0, tree="importance", n=(128, 128), depth=8, topk=8,
            beta=0.6, vocab=151936, target_var=2.0, draft="noise", draft_var=0.5,
            shuffle=False, mask_mass=0.7),
    5: dict(name="long", batch=4, hq=64, hkv=8, d=128, prefix=(32768, 32768), tree="topk",
            n=(256, 256), depth=10, kmax=4, vocab=128256, target_var=3.0, draft="noise",
            draft_var=1.0, shuffle=False, mask_mass=None),
}
BLOCK_SIZE = 16


def config(num: int, **overrides) -> dict:
    c = dict(CONFIGS[num])
    c["num"] = num
    c["seed"] = 20260 + num
    c.update(overrides)
    return c


def rng(*key) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([int(k) for k in key])))


def to_bf16_bits(x) -> np.ndarray:
    """fp64/fp32 array -> bf16 bit patterns (uint16), round to nearest even via fp32."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32)  # finite inputs only: the rounding add cannot overflow
    u = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ E4M3 inputs
# The FP8 form of the attention inputs (the caller's FP8 KV cache): E4M3 codes
# with one fp32 scale per row of D elements (a token of one head).  Only input
# preparation lives here; decoding belongs to the consumers.
E4M3_MAX = 448.0


def _e4m3_magnitudes() -> np.ndarray:
    """Values of the non-negative finite codes 0..126, ascending (the code order)."""
    e, m = np.arange(127) >> 3, np.arange(127) & 7
    return np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))


def e4m3_encode(x) -> np.ndarray:
    """E4M3 codes (uint8) of real values: round to nearest, ties to the even
    code, magnitudes above 448 saturate to 448, NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    mags = _e4m3_magnitudes()
    ax = np.abs(x)
    hi = np.clip(np.searchsorted(mags, np.minimum(ax, E4M3_MAX), side="left"), 1, 126)
    lo = hi - 1
    d_lo, d_hi = ax - mags[lo], mags[hi] - ax
    code = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(ax >= E4M3_MAX, 126, code)
    code = np.where(ax == 0.0, 0, code).astype(np.uint8)
    code = np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def quantize_e4m3_rows(values) -> tuple[np.ndarray, np.ndarray]:
    """Per-row (last axis) scales s = max|row| / 448 in fp32 (1 for an all-zero
    row) and the codes of row / s."""
    v = np.asarray(values, dtype=np.float64)
    amax = np.abs(v).max(axis=-1)
    scale = np.where(amax > 0, amax / E4M3_MAX, 1.0).astype(np.float32)
    codes = e4m3_encode(v / scale.astype(np.float64)[..., None])
    return codes, scale


def e4m3_case(case: dict) -> dict:
    """The E4M3 form of an attention case: every bf16 input re-quantised per row."""
    out = dict(case, dtype="e4m3")
    for k in ("q", "k_prefix", "v_prefix", "k_nodes", "v_nodes"):
        codes, scale = quantize_e4m3_rows(bf16_bits_to_f32(case[k]))
        out[k] = codes
        out[k + "_scale"] = scale
    return out


def _softmax32(x: np.ndarray, out: np.ndarray | None = None) -> np.ndarray:
    """Input preparation: probabilities from logits in fp64 (row blocks), rounded to fp32."""
    x = np.atleast_2d(x)
    out = np.empty(x.shape, np.float32) if out is None else out
    for r0 in range(0, x.shape[0], 32):
        x64 = x[r0:r0 + 32].astype(np.float64)
        x64 -= x64.max(axis=-1, keepdims=True)
        np.exp(x64, out=x64)
        x64 /= x64.sum(axis=-1, keepdims=True)
        out[r0:r0 + 32] = x64
    return out


def _desc_order(row: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries, descending, ties to the lower index."""
    k = min(k, row.shape[0])
    if k <= 0:
        return np.zeros(0, np.int64)
    part = np.argpartition(-row, k - 1)[:k] if k < row.shape[0] else np.arange(row.shape[0])
    # exact descending order with index tie-break among the candidates
    cand = part[np.lexsort((part, -row[part]))]
    return cand[:k]


def retained_mask_row(q_row: np.ndarray, mass: float) -> np.ndarray:
    """Cumulative-mass soft truncation of a draft row (input preparation):
    tokens by descending draft probability (ties to the lower id) are kept
    until the cumulative mass reaches ``mass``, the crossing token included.
    Returns the packed bitmask, uint32 [ceil(V/32)], bit v%32 of word v//32."""
    V = q_row.shape[0]
    order = np.argsort(-q_row.astype(np.float64), kind="stable")  # ties: lower id first
    cum = np.cumsum(q_row[order].astype(np.float64))
    nkeep = int(np.searchsorted(cum, mass, side="left")) + 1
    nkeep = min(nkeep, V)
    bits = np.zeros(((V + 31) // 32) * 32, dtype=np.uint8)
    bits[order[:nkeep]] = 1
    return np.packbits(bits.reshape(-1, 32)[:, ::-1], axis=1).view(">u4").astype(np.uint32).ravel()


def unpack_mask(words, vocab: int) -> np.ndarray:
    """Packed uint32 bitmask (bit v%32 of word v//32) -> bool [vocab]."""
    w = np.ascontiguousarray(words, dtype="<u4")
    return np.unpackbits(w.view(np.uint8), bitorder="little")[:vocab].astype(bool)


class _Rows:
    """Target/draft logits rows of one tree (fp32), drawn per discovery index
    into preallocated storage."""

    def __init__(self, cfg, b, vocab, nmax):
        self.cfg, self.b, self.V = cfg, b, vocab
        self.t = np.empty((nmax, vocab), np.float32)
        self.d = np.empty((nmax, vocab), np.float32)
        self.have = np.zeros(nmax, bool)

    def get(self, r):
        if not self.have[r]:
            g = rng(self.cfg["seed"], _S_ROWS, self.b, r)
            t = self.t[r]
            g.standard_normal(out=t, dtype=np.float32)
            t *= np.float32(np.sqrt(self.cfg["target_var"]))
            d = self.d[r]
            g.standard_normal(out=d, dtype=np.float32)
            d *= np.float32(np.sqrt(self.cfg["draft_var"]))
            if self.cfg["draft"] != "independent":
                d += t
            self.have[r] = True
        return self.t[r], self.d[r]


def _grow_tree(cfg, b, n_target, rows: _Rows):
    """Returns (parent_discovery[list], token[list]) in discovery order."""
    g = rng(cfg["seed"], _S_TREE, b)
    kind = cfg["tree"]
    parent, token, depth = [-1], [-1], [0]
    if kind in ("binary", "topk"):
        head = 0
        while len(parent) < n_target and head < len(parent):
            j = head
            head += 1
            if depth[j] >= cfg["depth"]:
                continue
            k = 2 if kind == "binary" else int(g.integers(1, cfg["kmax"] + 1))
            q = rows.get(j)[1]
            for tok in _desc_order(q, k):
                if len(parent) >= n_target:
                    break
                parent.append(j)
                token.append(int(tok))
                depth.append(depth[j] + 1)
        if kind == "topk":
            # the growth can stop short of n nodes (every branch at the depth
            # limit); top up: nodes in discovery order get their next most
            # probable tokens, up to kmax children each, until n nodes exist
            j = 0
            while len(parent) < n_target and j < len(parent):
                if depth[j] < cfg["depth"]:
                    have = {token[i] for i in range(1, len(parent)) if parent[i] == j}
                    for tok in _desc_order(rows.get(j)[1], cfg["kmax"]):
                        if len(parent) >= n_target or len(have) >= cfg["kmax"]:
                            break
                        if int(tok) in have:
                            continue
                        have.add(int(tok))
                        parent.append(j)
                        token.append(int(tok))
                        depth.append(depth[j] + 1)
                j += 1
        return parent, token
    if kind == "importance":
        gg = rng(cfg["seed"], _S_GUMBEL, b)
        heap = []
        logw_path = [0.0]
        counter = 0

        def offer(j):
            nonlocal counter
            if depth[j] >= cfg["depth"]:
                return
            q = _softmax32(rows.get(j)[1])[0]
            kept = unpack_mask(retained_mask_row(q, cfg["mask_mass"]), q.shape[0])
            cand = _desc_order(np.where(kept, q, -1.0), cfg["topk"])
            cand = cand[kept[cand]]
            pw = q[cand].astype(np.float64) ** cfg["beta"]
            w = pw / pw.sum()
            gum = gg.gumbel(size=cand.shape[0])
            for c, wc, gc in zip(cand, w, gum):
                key = logw_path[j] + np.log(wc)
                heapq.heappush(heap, (-(key + gc), counter, j, int(c), key))
                counter += 1

        offer(0)
        while len(parent) < n_target and heap:
            _, _, j, tok, key = heapq.heappop(heap)
            parent.append(j)
            token.append(tok)
            depth.append(depth[j] + 1)
            logw_path.append(key)
            offer(len(parent) - 1)
        return parent, token
    raise ValueError(kind)


def _bfs_renumber(parent, token, qprob_of):
    """Breadth-first numbering, siblings by descending draft probability of
    their token in the parent's row (ties to the lower token id)."""
    n = len(parent)
    children = [[] for _ in range(n)]
    for i in range(1, n):
        children[parent[i]].append(i)
    order = [0]
    head = 0
    while head < len(order):
        j = order[head]
        head += 1
        ch = children[j]
        if ch:
            q = qprob_of(j)
            ch = sorted(ch, key=lambda c: (-float(q[token[c]]), token[c]))
            order.extend(ch)
    new_of = {old: new for new, old in enumerate(order)}
    new_parent = np.array([-1] + [new_of[parent[o]] for o in order[1:]], dtype=np.int32)
    new_token = np.array([token[o] for o in order], dtype=np.int32)
    return np.array(order, dtype=np.int64), new_parent, new_token


def make_case(cfg: dict, parts=("attn", "accept"), kind: str = "probs") -> dict:
    """Build one synthetic case.  ``cfg`` from :func:`config` (overrides allowed:
    batch, prefix, n, vocab, hq, hkv, d, ...).  ``kind`` is "probs" or "logits"
    (the form of the target rows handed to the accept pass)."""
    B, V = cfg["batch"], cfg["vocab"]
    seed = cfg["seed"]
    glen = rng(seed, _S_LEN)
    n_lo, n_hi = cfg["n"]
    p_lo, p_hi = cfg["prefix"]
    ns = [int(glen.integers(n_lo, n_hi + 1)) for _ in range(B)]
    ls = [int(glen.integers(p_lo, p_hi + 1)) for _ in range(B)]
    if "prefix_lens" in cfg:
        ls = list(cfg["prefix_lens"])
    if "nodes" in cfg:
        ns = list(cfg["nodes"])

    parents, tokens, tgt_rows, dr_rows = [], [], [], []
    need_rows = "accept" in parts
    for b in range(B):
        rows = _Rows(cfg, b, V, max(n_hi, ns[b], len(cfg["parent"][b]) if "parent" in cfg else 0))
        if "parent" in cfg:  # explicit tree shape supplied by a test
            par = list(np.asarray(cfg["parent"][b]).tolist())
            tok = [-1] + [int(rng(seed, _S_TREE, b, i).integers(0, V)) for i in range(1, len(par))]
            order = np.arange(len(par))
            new_par, new_tok = np.asarray(par, np.int32), np.asarray(tok, np.int32)
        else:
            par, tok = _grow_tree(cfg, b, ns[b], rows)
            order, new_par, new_tok = _bfs_renumber(
                par, tok, lambda j: _softmax32(rows.get(j)[1])[0])
        ns[b] = len(new_par)
        parents.append(new_par)
        tokens.append(new_tok)
        if need_rows:
            for o in order:
                rows.get(int(o))
            tgt_rows.append(rows.t[order])
            dr_rows.append(rows.d[order])
        del rows

    node_offsets = np.zeros(B + 1, np.int32)
    node_offsets[1:] = np.cumsum(ns)
    tot = int(node_offsets[-1])
    case = dict(cfg=cfg, batch=B, node_offsets=node_offsets, parent=np.concatenate(parents),
                max_nodes=int(cfg.get("max_nodes", max(n_hi, max(ns)))), total_nodes=tot)

    if "attn" in parts:
        hq, hkv, D = cfg["hq"], cfg["hkv"], cfg["d"]
        nblk = [(l + BLOCK_SIZE - 1) // BLOCK_SIZE for l in ls]
        num_blocks = max(1, sum(nblk))
        max_bps = max(1, max(nblk))
        perm = np.arange(num_blocks, dtype=np.int32)
        if cfg.get("shuffle"):
            perm = rng(seed, _S_TABLE).permutation(num_blocks).astype(np.int32)
        table = np.zeros((B, max_bps), np.int32)
        pos = 0
        for b in range(B):
            table[b, : nblk[b]] = perm[pos: pos + nblk[b]]
            pos += nblk[b]

        def draw(stream, shape):
            return rng(seed, stream).standard_normal(size=shape, dtype=np.float32)

        q = draw(_S_Q, (tot, hq, D))
        kp = draw(_S_KP, (num_blocks, hkv, BLOCK_SIZE, D))
        vp = draw(_S_VP, (num_blocks, hkv, BLOCK_SIZE, D))
        if cfg.get("image_tokens"):
            # image-token prefix positions get a larger spread (std image_std)
            s = np.float32(cfg["image_std"])
            for b in range(B):
                for t0 in range(0, min(cfg["image_tokens"], ls[b]), BLOCK_SIZE):
                    pg = table[b, t0 // BLOCK_SIZE]
                    hi = min(BLOCK_SIZE, cfg["image_tokens"] - t0)
                    kp[pg, :, :hi] *= s
                    vp[pg, :, :hi] *= s
        kn = draw(_S_KN, (tot, hkv, D))
        vn = draw(_S_VN, (tot, hkv, D))
        case.update(num_q_heads=hq, num_kv_heads=hkv, head_dim=D, block_size=BLOCK_SIZE,
                    num_blocks=num_blocks, block_table=table,
                    prefix_lens=np.asarray(ls, np.int32),
                    q=to_bf16_bits(q), k_prefix=to_bf16_bits(kp), v_prefix=to_bf16_bits(vp),
                    k_nodes=to_bf16_bits(kn), v_nodes=to_bf16_bits(vn),
                    softmax_scale=float(cfg.get("softmax_scale", 0.0)))

    if need_rows:
        tgt = np.concatenate(tgt_rows)
        del tgt_rows
        draft_probs = np.concatenate(dr_rows)
        del dr_rows
        _softmax32(draft_probs, out=draft_probs)
        target = _softmax32(tgt, out=tgt) if kind == "probs" else tgt
        gu = rng(seed, _S_UNI)
        uniforms = (gu.integers(0, 1 << 24, size=tot).astype(np.float64) * 2.0 ** -24).astype(
            np.float32)
        case.update(vocab=V, kind=kind, target=target, draft_probs=draft_probs,
                    draft_tokens=np.concatenate(tokens), uniforms=uniforms)
        if cfg.get("mask_mass"):
            case["retained_mask"] = np.stack(
                [retained_mask_row(draft_probs[r], cfg["mask_mass"]) for r in range(tot)])
        else:
            case["retained_mask"] = None
    return case


def extend_pool(case: dict, extra_tokens: int):
    """Input preparation for committing an accepted path: a copy of the case's
    paged pool with fresh pages appended (seeded N(0,1) bf16, so that rows a
    commit must not touch are distinguishable) and every sequence's
    block-table row extended so that positions up to L_b + extra_tokens - 1
    have pages; the new pages are handed out in a shuffled order.  Returns
    (k_pool, v_pool, block_table): uint16 bf16 bits and int32."""
    B = case["batch"]
    lens = np.asarray(case["prefix_lens"], np.int64)
    table0 = np.asarray(case["block_table"], np.int32)
    have = (lens + BLOCK_SIZE - 1) // BLOCK_SIZE
    need = (lens + extra_tokens + BLOCK_SIZE - 1) // BLOCK_SIZE
    add = int(np.sum(need - have))
    nb0 = int(case["k_prefix"].shape[0])
    g = rng(case["cfg"]["seed"], _S_EXT)
    fresh = nb0 + g.permutation(add).astype(np.int32)
    shape = (add,) + tuple(case["k_prefix"].shape[1:])
    k_pool = np.concatenate([case["k_prefix"], to_bf16_bits(g.standard_normal(size=shape))])
    v_pool = np.concatenate([case["v_prefix"], to_bf16_bits(g.standard_normal(size=shape))])
    table = np.full((B, max(table0.shape[1], int(need.max()))), -1, np.int32)
    pos = 0
    for b in range(B):
        table[b, : have[b]] = table0[b, : have[b]]
        k = int(need[b] - have[b])
        table[b, have[b]: need[b]] = fresh[pos: pos + k]
        pos += k
    return k_pool, v_pool, table
