"""A CPU model of the tree-attention kernel's work schedule, checked for the
properties the kernel relies on (no GPU needed):

  * the key tiles of every unit (256 packed rows of a sequence and KV head)
    are computed exactly once, by pieces in key order;
  * a unit cut by range boundaries has one piece per virtual CTA it meets,
    its first piece holds tile 0 and the others start their CTA's range;
  * the partial-result slot of each piece is unique, and the slots the
    merging piece reads (from vfirst, npieces and the CTA lane) are exactly
    the slots the pieces wrote;
  * every CTA gets the same number of tiles (within one), and the CTAs of a
    virtual CTA walk the same (sequence, KV head, key tile) ranges.

The model follows the kernel's arithmetic: units ordered (sequence, KV head,
layer, m-tile pair lane), the line cut at floor(v W / V), V = min(launched
virtual CTAs, W / min_tiles)."""
import itertools

import numpy as np
import pytest

BN, UNIT_ROWS = 128, 256


def plan(batch, hq, hkv, max_nodes, max_prefix, sms=152, min_tiles=3):
    g = hq // hkv
    mpairs = -(-max_nodes * g // UNIT_ROWS)
    lanes = min(mpairs, sms)
    layers = -(-mpairs // lanes)
    tiles = -(-max_prefix // BN) + -(-max_nodes // BN)
    wmax = batch * hkv * layers * tiles
    vctas = max(1, min(sms // lanes, wmax // min_tiles, 4096))
    return dict(g=g, lanes=lanes, vctas=vctas, min_tiles=min_tiles)


def vcta_of(p, W, V):
    v = (p * V) // W
    while v + 1 < V and ((v + 1) * W) // V <= p:
        v += 1
    while v > 0 and (v * W) // V > p:
        v -= 1
    return v


def schedule(lens, nodes, hkv, pl):
    """Every CTA's pieces, as the kernel's build_schedule makes them."""
    g, lanes = pl["g"], pl["lanes"]
    seqs = []
    for L, N in zip(lens, nodes):
        P, T = -(-L // BN), -(-L // BN) + -(-N // BN)
        mpairs = -(-N * g // UNIT_ROWS)
        layers = -(-mpairs // lanes)
        seqs.append(dict(P=P, T=T, mpairs=mpairs, layers=layers, W=hkv * layers * T, N=N))
    W = sum(s["W"] for s in seqs)
    V = max(1, min(pl["vctas"], W // max(1, pl["min_tiles"])))
    out = {}
    for cta in range(pl["vctas"] * lanes):
        v, li = cta // lanes, cta % lanes
        pieces = []
        if W > 0 and v < V:
            s_v, e_v = (v * W) // V, ((v + 1) * W) // V
            c0 = 0
            for b, s in enumerate(seqs):
                lo, hi = max(s_v, c0) - c0, min(e_v, c0 + s["W"]) - c0
                if s["W"] > 0 and lo < hi:
                    for ui in range(lo // s["T"], (hi - 1) // s["T"] + 1):
                        kvh, layer = ui // s["layers"], ui % s["layers"]
                        mp = layer * lanes + li
                        if mp >= s["mpairs"]:
                            continue
                        t0 = max(lo, ui * s["T"]) - ui * s["T"]
                        t1 = min(hi, (ui + 1) * s["T"]) - ui * s["T"]
                        pc = dict(b=b, kvh=kvh, mp=mp, t0=t0, t1=t1, T=s["T"])
                        if t0 == 0 and t1 == s["T"]:
                            pc.update(slot=-1, npieces=1, vfirst=v, cnt=-1)
                        else:
                            u0 = c0 + ui * s["T"]
                            vf, vl = vcta_of(u0, W, V), vcta_of(u0 + s["T"] - 1, W, V)
                            pc.update(vfirst=vf, npieces=vl - vf + 1, cnt=vf * lanes + li,
                                      slot=2 * cta + (0 if t0 > 0 else 1))
                        pieces.append(pc)
                c0 += s["W"]
        out[cta] = pieces
    return out, W, V


def check(lens, nodes, hq, hkv, max_nodes=None, max_prefix=None, sms=152):
    pl = plan(len(lens), hq, hkv, max_nodes or max(nodes), max_prefix or max(1, max(lens)), sms)
    sched, W, V = schedule(lens, nodes, hkv, pl)
    lanes, g = pl["lanes"], pl["g"]
    covered = {}
    slots = {}
    for cta, pieces in sched.items():
        for pc in pieces:
            key = (pc["b"], pc["kvh"], pc["mp"])
            covered.setdefault(key, []).append((pc["t0"], pc["t1"], pc))
            if pc["slot"] >= 0:
                assert pc["slot"] not in slots, "slot written twice"
                slots[pc["slot"]] = key
                assert pc["slot"] < 2 * pl["vctas"] * lanes and pc["cnt"] < pl["vctas"] * lanes
    for b, (L, N) in enumerate(zip(lens, nodes)):
        mpairs = -(-N * g // UNIT_ROWS)
        T = -(-L // BN) + -(-N // BN)
        for kvh, mp in itertools.product(range(hkv), range(mpairs)):
            parts = sorted(covered.pop((b, kvh, mp)), key=lambda x: x[0])
            assert parts[0][0] == 0 and parts[-1][1] == T
            for (a0, a1, _), (b0, b1, _) in zip(parts, parts[1:]):
                assert a1 == b0, "tiles of a unit computed twice or skipped"
            if len(parts) == 1:
                assert parts[0][2]["slot"] == -1
                continue
            # the merger's view: slot of piece s from CTA (vfirst + s) * lanes + lane
            pc0 = parts[0][2]
            assert all(p[2]["npieces"] == len(parts) and p[2]["vfirst"] == pc0["vfirst"]
                       and p[2]["cnt"] == pc0["cnt"] for p in parts)
            want = set()
            for s in range(len(parts)):
                cta = (pc0["vfirst"] + s) * lanes + mp % lanes
                want.add(2 * cta + 1 if s == 0 else 2 * cta)
            assert want == {p[2]["slot"] for p in parts}
    assert not covered
    # balance: every active CTA's tile count within one of W / V (idle lanes
    # of short layers aside)
    counts = [sum(p["t1"] - p["t0"] for p in pcs) for pcs in sched.values()]
    if lanes == 1:
        active = [c for c in counts if c]
        assert max(active) - min(active) <= 1
    return sched, W, V


@pytest.mark.parametrize("num", [1, 2, 3, 4, 5])
def test_workload_schedules(num):
    from speculative_decoding_tree_attention_gb300 import workloads as wl
    cfg = wl.config(num)
    rng = wl.rng(cfg["seed"], 7)
    B = cfg["batch"]
    lens = [int(x) for x in rng.integers(cfg["prefix"][0], cfg["prefix"][1] + 1, B)]
    nodes = [int(x) for x in rng.integers(cfg["n"][0], cfg["n"][1] + 1, B)]
    check(lens, nodes, cfg["hq"], cfg["hkv"], max_nodes=cfg["n"][1], max_prefix=cfg["prefix"][1])


def test_long_context_lanes_share_key_ranges():
    """8 m-tile pairs per KV head: the 8 CTAs of a virtual CTA compute the
    same (sequence, KV head, tiles) pieces, one pair each."""
    sched, W, V = check([32768] * 4, [256] * 4, 64, 8)
    for v in range(V):
        ranges = [[(p["b"], p["kvh"], p["t0"], p["t1"]) for p in sched[v * 8 + i]] for i in range(8)]
        assert all(r == ranges[0] for r in ranges)
        assert [p["mp"] for p in sched[v * 8 + 3]] == [3] * len(sched[v * 8 + 3])


@pytest.mark.parametrize("seed", range(40))
def test_random_batches(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 3, 4, 7, 8, 16]))
    lens = [int(x) for x in rng.integers(0, 3000, B)]
    nodes = [int(x) for x in rng.integers(1, 300, B)]
    sms = int(rng.choice([1, 7, 64, 152]))
    check(lens, nodes, g * hkv, hkv, sms=sms)


def test_many_tiny_sequences_need_several_rounds():
    sched, W, V = check([0] * 2048, [1 + (i % 3) for i in range(2048)], 4, 4)
    assert max(len(p) for p in sched.values()) > 32   # more than one round of 32 pieces


def start_fp32(v, W, V):
    """The kernel's range boundary: v q + k, k = int(fp32(v r) * fp32(1 / V))
    corrected once each way (W = q V + r)."""
    q, r = divmod(W, V)
    n = v * r
    rV = np.float32(1.0) / np.float32(V)
    k = int(np.float32(n) * rV)
    if k * V > n:
        k -= 1
    elif (k + 1) * V <= n:
        k += 1
    return v * q + k


@pytest.mark.parametrize("V", [1, 2, 3, 7, 19, 38, 76, 151, 152, 1000, 4095, 4096])
def test_division_free_range_starts_are_exact(V):
    rng = np.random.default_rng(V)
    Ws = {V, V + 1, 2 * V - 1, 4 * V + 3, 2**31 - 1, 2**31 - 2}
    Ws.update(int(x) for x in rng.integers(V, 2**31 - 1, 40))
    for W in sorted(Ws):
        vs = range(V + 1) if V <= 200 else sorted({0, 1, V - 1, V, *rng.integers(0, V + 1, 300).tolist()})
        for v in vs:
            assert start_fp32(v, W, V) == (v * W) // V, (v, W, V)


def owner_fp32(p, W, V):
    """The kernel's owner of line position p: int(fp32(p) * fp32(V / W)),
    clamped to [0, V), then up to four exact steps each way."""
    VW = np.float32(V) / np.float32(W)
    o = min(V - 1, max(0, int(np.float32(p) * VW)))
    for _ in range(4):
        if o > 0 and start_fp32(o, W, V) > p:
            o -= 1
    for _ in range(4):
        if o + 1 < V and start_fp32(o + 1, W, V) <= p:
            o += 1
    return o


@pytest.mark.parametrize("V", [1, 2, 3, 19, 38, 152, 1000, 4096])
def test_owner_estimate_finds_the_range(V):
    rng = np.random.default_rng(100 + V)
    for W in [V, V + 1, 2 * V + 1, 2**31 - 1] + [int(x) for x in rng.integers(V, 2**31 - 1, 25)]:
        bounds = [(v * W) // V for v in range(V + 1)]
        ps = {0, W - 1}
        for v in range(0, V, max(1, V // 64)):
            ps.update({bounds[v], max(0, bounds[v] - 1), min(W - 1, bounds[v + 1] - 1)})
        ps.update(int(x) for x in rng.integers(0, W, 200))
        for p in ps:
            o = owner_fp32(p, W, V)
            assert bounds[o] <= p < bounds[o + 1], (p, W, V, o)
