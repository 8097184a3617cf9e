"""A host-side model of the tree-attention kernel's mbarrier protocol (CPU only).

The kernel's warps (TMA producer, S = Q K^T issuer, P.V issuer, two softmax
lanes of warps that take alternating 128-key tiles, and the in-order tensor
pipe) are modelled as generators that advance one step at a time under random
interleavings.  Every mbarrier keeps its phase count and answers a parity wait
the way the hardware does (a wait on parity P passes while the last completed
phase has parity P).  The model asserts, at each step, the ordering each wait
is meant to guarantee: S(t) is written only after the softmax has read S(t-2)
from that buffer, the softmax reads the S it expects, the running max of tile
t-1 is there when tile t needs it, P(t) is written only after P(t-1).V has
read the single P buffer, P.V reads the P it expects, and the epilogue runs
after the last P.V.  A run that stops making progress is a deadlock.

As a negative control the same model with a single P.V-completion barrier
(instead of one per tile parity) must fail: there a lane waiting for
P(t-1).V can match the parity of P(t-3).V while P(t-2).V is still pending."""
import random

import pytest


class _Bar:
    def __init__(self, count, name):
        self.count, self.pending, self.done, self.name = count, 0, 0, name

    def arrive(self, n=1):
        self.pending += n
        assert self.pending <= self.count, self.name
        if self.pending == self.count:
            self.pending = 0
            self.done += 1

    def ready(self, parity):
        return (self.done & 1) != parity


class _Violation(AssertionError):
    pass


def _check(cond, what):
    if not cond:
        raise _Violation(what)


def run_model(T, stages, seed, warps=2, split_o_done=True):
    rng = random.Random(seed)
    kfull = [_Bar(1, "kfull") for _ in range(stages)]
    kempty = [_Bar(1, "kempty") for _ in range(stages)]
    vfull = [_Bar(1, "vfull") for _ in range(stages)]
    vempty = [_Bar(1, "vempty") for _ in range(stages)]
    s_full = [_Bar(1, "s_full") for _ in range(2)]
    s_free = [_Bar(32 * warps, "s_free") for _ in range(2)]
    p_full = _Bar(32 * warps, "p_full")
    o_done = [_Bar(1, "o_done") for _ in range(2 if split_o_done else 1)]
    chain = [[_Bar(32, "chain") for _ in range(warps)] for _ in range(2)]
    st = dict(k=set(), v=set(), s=[None, None], s_read=set(), p=None, pv_done=set(), m=set())
    pipe = []

    def od(t):  # the P.V-completion barrier of tile t
        return o_done[t & 1] if split_o_done else o_done[0]

    def od_parity(t):
        return ((t >> 1) & 1) if split_o_done else (t & 1)

    def wait(bar, parity):
        while not bar.ready(parity):
            yield False

    def tma():
        tk = tv = 0
        while tv < T:
            moved = False
            if tk < T and kempty[tk % stages].ready(((tk // stages) & 1) ^ 1):
                st["k"].add(tk)
                kfull[tk % stages].arrive()
                tk += 1
                moved = True
            if tv < tk and vempty[tv % stages].ready(((tv // stages) & 1) ^ 1):
                st["v"].add(tv)
                vfull[tv % stages].arrive()
                tv += 1
                moved = True
            yield moved

    def s_issuer():
        for t in range(T):
            yield from wait(kfull[t % stages], (t // stages) & 1)
            if t >= 2:
                yield from wait(s_free[t & 1], ((t - 2) >> 1) & 1)
            _check(t in st["k"], "S before K landed")
            pipe.append(("S", t))
            yield True

    def pv_issuer():
        for t in range(T):
            yield from wait(p_full, t & 1)
            yield from wait(vfull[t % stages], (t // stages) & 1)
            _check(st["p"] == t and t in st["v"], f"P.V({t}) reads P {st['p']}")
            pipe.append(("PV", t))
            yield True

    def tensor_pipe():  # executes the issued MMAs in order
        while True:
            if not pipe:
                yield False
                continue
            kind, t = pipe.pop(0)
            if kind == "S":
                b = t & 1
                prev = st["s"][b]
                _check(prev is None or all((prev, (prev & 1) * warps + q) in st["s_read"]
                                           for q in range(warps)),
                       f"S({t}) overwrites an unread S({prev})")
                st["s"][b] = t
                s_full[b].arrive()
                kempty[t % stages].arrive()
            else:
                st["pv_done"].add(t)
                od(t).arrive()
                vempty[t % stages].arrive()
            yield True

    def softmax_warp(lane, q):
        for t in range(lane, T, 2):
            yield from wait(s_full[t & 1], (t >> 1) & 1)
            _check(st["s"][t & 1] == t, f"lane reads S {st['s'][t & 1]} for tile {t}")
            st["s_read"].add((t, lane * warps + q))
            s_free[t & 1].arrive(32)
            yield True
            if t >= 1:
                yield from wait(chain[1 - lane][q], ((t - 1) >> 1) & 1)
                _check((t - 1, q) in st["m"], f"running max of tile {t - 1} missing")
            st["m"].add((t, q))
            chain[lane][q].arrive(32)
            yield True
            if t >= 1:
                yield from wait(od(t - 1), od_parity(t - 1))
                _check(t - 1 in st["pv_done"], f"P({t}) written before P({t - 1}).V completed")
            st["p"] = t
            yield True
            p_full.arrive(32)
            yield True
        if T > 0:
            yield from wait(od(T - 1), od_parity(T - 1))
            _check(T - 1 in st["pv_done"], "epilogue before the last P.V")

    actors = [tma(), s_issuer(), pv_issuer(), tensor_pipe()]
    actors += [softmax_warp(lane, q) for lane in range(2) for q in range(warps)]
    finished, idle = set(), 0
    while len(finished) < len(actors) - 1:  # the tensor pipe never finishes
        i = rng.randrange(len(actors))
        if i in finished:
            continue
        try:
            moved = next(actors[i])
        except StopIteration:
            finished.add(i)
            moved = True
        idle = 0 if moved else idle + 1
        _check(idle < 20000, "deadlock")


@pytest.mark.parametrize("stages", [2, 3])
@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 7, 10, 17])
def test_protocol_orderings_hold(T, stages):
    for seed in range(40):
        run_model(T, stages, seed)


def test_a_single_completion_barrier_is_caught():
    caught = 0
    for seed in range(60):
        try:
            run_model(9, 3, seed, split_o_done=False)
        except _Violation:
            caught += 1
    assert caught > 0
