#!/usr/bin/env python
"""Benchmark of one tree-verification step on GB300.

A step is one pass of the whole hot path over one batch of a synthetic
workload: tv_tree_attention (tree attention over the paged prefix plus the
tree mask) followed by tv_accept (logits mode: log-sum-exp, pruning
renormalisation when the workload has a retained-set mask, per-node tests,
the longest accepted path and the bonus draw).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 5] [--impl ours|reference]

Prints ONE JSON line on rank 0.  `value` is tree-tokens/s (tree nodes
verified per second, all ranks) with inputs resident in HBM; L2 is flushed
between timed steps (a 512 MiB write, outside the timed events).  Under
torchrun each rank runs an independent replica (no collective on the data
path: sequences are independent), timing is max over ranks.
The headline is the 32K long-context workload (config 5); the multimodal,
serving and 7B-like workloads (configs 4, 3 and 2) are timed in the same run
and reported under "workloads", each call on its own.
`--impl reference` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from speculative_decoding_tree_attention_gb300 import workloads as wl  # noqa: E402

METRIC = "tree-verify tree-tokens/s"
UNIT = "tree-tokens/s"
FLUSH_BYTES = 512 << 20
ATTN_SRC = os.path.join(ROOT, "speculative_decoding_tree_attention_gb300", "csrc",
                        "tree_attn_kernel.cu")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=5,
                    help="workload 1..5 (default: 5, the 32K long-context batch)")
    ap.add_argument("--mode", choices=["logits", "probs"], default="logits")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of a CUDA graph")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline sample budget")
    ap.add_argument("--no-side", dest="side", action="store_false",
                    help="skip the serving and 7B-like figures reported beside the headline")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (smaller cases for profiler captures)")
    ap.add_argument("--profile", choices=["attention", "attention_fp8", "accept", "retained"],
                    default=None,
                    help="profiler-capture mode: launch only this call of the workload "
                         "--warmup + --steps times, eagerly, then exit (no JSON line)")
    return ap.parse_args()


def workload_desc(cfg, case):
    ns = np.diff(case["node_offsets"])
    return {"workload": f"{cfg['name']} (config {cfg['num']})", "batch": int(cfg["batch"]),
            "q_heads": int(cfg["hq"]), "kv_heads": int(cfg["hkv"]), "head_dim": int(cfg["d"]),
            "prefix_lens": [int(x) for x in case["prefix_lens"]] if cfg["batch"] <= 4 else
            [int(min(case["prefix_lens"])), int(max(case["prefix_lens"]))],
            "tree_nodes": int(ns.sum()), "vocab": int(cfg["vocab"]),
            "retained_mask": bool(cfg.get("mask_mass")), "block_size": wl.BLOCK_SIZE,
            "paged_shuffled": bool(cfg.get("shuffle"))}


def attention_bytes(case):
    """Algorithmic bytes of one tree-attention launch: prefix K+V once per
    (sequence, KV head), Q, tree K/V and the output, all bf16."""
    hq, hkv, D = case["num_q_heads"], case["num_kv_heads"], case["head_dim"]
    L = np.asarray(case["prefix_lens"], np.int64)
    tot = int(case["node_offsets"][-1])
    return int(4 * L.sum() * hkv * D + 2 * tot * hq * D * 2 + 4 * tot * hkv * D)


def attention_flops(case):
    hq, D = case["num_q_heads"], case["head_dim"]
    off = case["node_offsets"]
    f = 0
    for b in range(case["batch"]):
        N = int(off[b + 1] - off[b])
        par = case["parent"][off[b]:off[b + 1]]
        depth = np.zeros(N, np.int64)
        for i in range(1, N):
            depth[i] = depth[par[i]] + 1
        f += 4 * N * int(case["prefix_lens"][b]) * D * hq + 4 * D * hq * int((depth + 1).sum())
    return int(f)


def attention_bytes_fp8(case):
    """Algorithmic bytes of one FP8 tree-attention launch: prefix K+V codes and
    their row scales once per (sequence, KV head), Q codes and scales, tree K/V
    codes and scales, and the bf16 output."""
    hq, hkv, D = case["num_q_heads"], case["num_kv_heads"], case["head_dim"]
    L = np.asarray(case["prefix_lens"], np.int64)
    tot = int(case["node_offsets"][-1])
    return int(L.sum() * hkv * (2 * D + 8) + tot * hq * (D + 4) + tot * hkv * (2 * D + 8)
               + tot * hq * D * 2)


def fp8_inputs(d):
    """E4M3 codes and per-row scales of a resident bf16 workload (the input
    recipe's quantiser: scale = max |row| / 448, 1 for an all-zero row; codes
    rounded to nearest even), made on the device with torch."""
    import torch
    out = {}
    for k in ("q", "kp", "vp", "kn", "vn"):
        x = d[k].float()
        amax = x.abs().amax(dim=-1)
        scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        out[k] = (x / scale.unsqueeze(-1)).to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
        out[k + "_scale"] = scale.contiguous()
    return out


def accept_bytes(case):
    """Algorithmic bytes of one accept launch (logits mode): the target row of
    every node with children (LSE), the draft rows of those nodes and the mask
    rows when a retained set is given (Z), the two rows of one cut node, and
    the per-node vectors."""
    V = case["vocab"]
    off = case["node_offsets"]
    internal = 0
    for b in range(len(off) - 1):
        internal += len(set(case["parent"][off[b] + 1:off[b + 1]].tolist()))
    B = len(off) - 1
    masked = case.get("retained_mask") is not None
    row = 4 * V
    mrow = 4 * ((V + 31) // 32)
    per_node = 4 * 4 * int(off[-1])
    return int(internal * row + (internal * (row + mrow) if masked else 0)
               + B * (2 * row + (mrow if masked else 0)) + per_node)


def load_peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, source).  The attention kernel is timed
    alone in its own graph, so the burst GEMM figure is its tensor peak."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def ncu_traffic(cfg_num):
    """dram bytes per attention launch from a committed ncu summary, only if it
    was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    h = hashlib.sha256(open(ATTN_SRC, "rb").read()).hexdigest()[:16]
    e = d.get(str(cfg_num))
    if not e or e.get("kernel_sha") != h:
        return None
    return e.get("dram_bytes_per_launch")


def max_over_ranks(x: float, device) -> float:
    """The slowest rank's value (replicas: the job ends with its last rank)."""
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def pct(ms):
    """p10 / p50 / p90 of per-rep times given in ms, in microseconds."""
    v = np.sort(np.asarray(ms, np.float64)) * 1e3
    return {k: float(np.percentile(v, q)) for k, q in (("p10", 10), ("p50", 50), ("p90", 90))}


def roofline_entry(nbytes, flops, seconds, peak_bw, peak_tf, peak_kind):
    """The bound is whichever roof is lower for this launch's arithmetic
    intensity: HBM (bytes / peak bandwidth) or the bf16 tensor pipe
    (FLOPs / peak throughput)."""
    src = "of measured (MEASURED_PEAKS.json)" if peak_kind == "measured" else "of fallback"
    if flops / (peak_tf * 1e12) > nbytes / (peak_bw * 1e9):
        a = flops / seconds / 1e12
        return {"bound": "tensor", "achieved": a, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": a / peak_tf, "peak_source": src + " bf16_tflops (burst)"}
    a = nbytes / seconds / 1e9
    return {"bound": "hbm", "achieved": a, "peak": peak_bw, "unit": "GB/s",
            "frac": a / peak_bw, "peak_source": src + " hbm_gbs"}


class Clocks:
    """nvidia-smi samples (every 20 ms) read by a thread, each stamped with the
    host time it arrived.  `load(t0, t1)` marks a window in which the GPU ran
    this benchmark's kernels; the reported median SM clock is over the samples
    inside those windows, the throttle reasons over every sample."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index):
        import threading
        self.p = None
        self.samples = []   # (host time, sm MHz, max MHz, power W, reasons)
        self.windows = []
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(dev_index)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.p.stdout:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm, mx = float(f[1]), float(f[2])
            except ValueError:
                continue
            try:
                pw = float(f[3])
            except ValueError:
                pw = None
            r = [n for n, v in zip(names, f[5:9]) if v.lower().startswith("active")]
            self.samples.append((time.time(), sm, mx, pw, r))

    def load(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.1)
        self.p.terminate()
        try:
            self.p.wait(timeout=10)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.t.join(timeout=5)
        s = list(self.samples)
        under = [x for x in s if any(a <= x[0] <= b + 0.05 for a, b in self.windows)]
        reasons = sorted({n for x in s for n in x[4]})
        pw = [x[3] for x in under if x[3] is not None]
        return {"sm_mhz": statistics.median(x[1] for x in under) if under else None,
                "sm_max_mhz": max(x[2] for x in s) if s else None, "reasons": reasons,
                "samples": len(s), "samples_under_load": len(under),
                "power_w_max": max(pw) if pw else None}


def cpu_baseline(case, budget_s, threads=None):
    """The oracle as it stands, on the host cores, on a bounded sample of the
    same workload: chunks of up to 8 tree nodes (attention for all their query
    heads), and the accept pass of each tree once its last node is done,
    until about `budget_s` seconds of CPU work."""
    import oracle
    oracle.build()
    threads = threads or oracle.default_threads()
    off = case["node_offsets"]
    hq = case["num_q_heads"]
    B = case["batch"]
    done, trees, t0 = 0, 0, time.perf_counter()
    b, i0 = 0, 0
    while True:
        N = int(off[b + 1] - off[b])
        i1 = min(N, i0 + 8)
        rows = np.array([(b, i, h) for i in range(i0, i1) for h in range(hq)], np.int32)
        oracle.tree_attention_rows(case, rows, nthreads=threads)
        done += i1 - i0
        if i1 == N:
            sl = slice(off[b], off[b + 1])
            sub = {k: case[k] for k in ("vocab", "kind", "max_nodes")}
            sub.update(node_offsets=np.array([0, N], np.int32), parent=case["parent"][sl],
                       target=case["target"][sl], draft_probs=case["draft_probs"][sl],
                       draft_tokens=case["draft_tokens"][sl], uniforms=case["uniforms"][sl],
                       retained_mask=None if case.get("retained_mask") is None
                       else case["retained_mask"][sl])
            oracle.accept(sub, nthreads=threads, want_pq=False)
            trees += 1
            b, i0 = (b + 1) % B, 0
        else:
            i0 = i1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": done / el, "unit": UNIT, "cores": int(threads), "kind": "oracle",
            "sample": f"{done} tree nodes (all query heads; attention over the full prefix) and "
                      f"{trees} complete accept pass(es) in {el:.1f} s"}


def run_reference(args):
    cfg = wl.config(args.config, **({"batch": args.batch} if args.batch > 0 else {}))
    case = wl.make_case(cfg, parts=("attn", "accept"), kind=args.mode)
    per_step = min(2.0, 120.0 / max(1, args.steps))
    cpu_baseline(case, min(per_step, 0.5))  # warm-up: builds and pages in the oracle
    t0 = time.perf_counter()
    nodes = 0.0
    last = None
    for _ in range(args.steps):
        r = cpu_baseline(case, per_step)
        nodes += r["value"] * per_step
        last = r
    el = time.perf_counter() - t0
    value = nodes / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_desc(cfg, case), accept_input=args.mode),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": last["cores"],
                             "kind": "oracle",
                             "sample": f"{args.steps} steps of about {per_step:.2f} s each; "
                                       f"last step: {last['sample']}"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def host_arrays(case):
    """The step's inputs as host arrays (bf16 as int16 bit patterns)."""
    host = {
        "q": case["q"].view(np.int16), "kp": case["k_prefix"].view(np.int16),
        "vp": case["v_prefix"].view(np.int16), "table": case["block_table"],
        "kn": case["k_nodes"].view(np.int16), "vn": case["v_nodes"].view(np.int16),
        "parent": case["parent"], "lens": case["prefix_lens"], "off": case["node_offsets"],
        "target": case["target"], "draft": case["draft_probs"], "tokens": case["draft_tokens"],
        "uniforms": case["uniforms"],
    }
    if case.get("retained_mask") is not None:
        host["mask"] = case["retained_mask"].view(np.int32)
    return host


class Step:
    """One workload resident on the device, with its output buffers and the
    two library calls of a step (tree attention, then accept)."""

    def __init__(self, tv, case, cfg, mode, dev):
        import torch
        self.tv, self.case, self.cfg, self.mode = tv, case, cfg, mode
        self.host = host_arrays(case)
        d = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in self.host.items()}
        for k in ("q", "kp", "vp", "kn", "vn"):
            d[k] = d[k].view(torch.bfloat16)
        self.d = d
        B = cfg["batch"]
        self.B = B
        self.tot = int(case["node_offsets"][-1])
        self.max_nodes = int(case["max_nodes"])
        self.mpl = int(max(1, int(np.max(case["prefix_lens"]))))
        self.prm = tv.attention_params(d["q"], d["kp"], d["table"], d["lens"],
                                       num_kv_heads=cfg["hkv"], max_nodes=self.max_nodes,
                                       max_prefix_len=self.mpl)
        ws_bytes = tv.attention_workspace_size(self.prm)
        self.ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        self.out = torch.empty_like(d["q"])
        self.st_attn = torch.empty(B, dtype=torch.int32, device=dev)
        self.acc_out = {"accepted_len": torch.empty(B, dtype=torch.int32, device=dev),
                        "path": torch.empty(B, self.max_nodes, dtype=torch.int32, device=dev),
                        "bonus_token": torch.empty(B, dtype=torch.int32, device=dev),
                        "status": torch.empty(B, dtype=torch.int32, device=dev)}
        acc_prm = tv.AcceptParams(B, int(cfg["vocab"]), self.max_nodes, self.tot,
                                  1 if mode == "logits" else 0)
        acc_ws_bytes = int(tv.load().tv_accept_workspace_size(ctypes.byref(acc_prm)))
        self.acc_ws = torch.empty(max(acc_ws_bytes, 16), dtype=torch.uint8, device=dev)
        acc_stats = mode == "logits" or d.get("mask") is not None
        # kernels of ours per step: tree_attn_kernel, accept_tree_kernel and,
        # for logits or a retained mask, accept_rowstats_kernel (memsets not
        # counted)
        self.launches_per_step = 2 + (1 if acc_stats else 0)

    def attn(self, src=None):
        src = src or self.d
        self.tv.tree_attention(src["q"], src["kp"], src["vp"], src["table"], src["kn"], src["vn"],
                               src["parent"], src["lens"], src["off"], max_nodes=self.max_nodes,
                               max_prefix_len=self.mpl, out=self.out, status=self.st_attn,
                               workspace=self.ws)

    def acc(self, src=None, test="ratio", outputs=None):
        src = src or self.d
        self.tv.accept(src["target"], src["draft"], src["tokens"], src["parent"], src["off"],
                       src["uniforms"], src.get("mask"), max_nodes=self.max_nodes, kind=self.mode,
                       test=test, outputs=dict(outputs or self.acc_out, workspace=self.acc_ws))

    def check(self):
        assert int(self.st_attn.max()) == 0 and int(self.acc_out["status"].max()) == 0, "status"

    def attn_fp8(self, f):
        d = self.d
        self.tv.tree_attention_fp8(f["q"], f["q_scale"], f["kp"], f["kp_scale"], f["vp"],
                                   f["vp_scale"], d["table"], f["kn"], f["kn_scale"], f["vn"],
                                   f["vn_scale"], d["parent"], d["lens"], d["off"],
                                   max_nodes=self.max_nodes, max_prefix_len=self.mpl,
                                   out=self.out, status=self.st_attn, workspace=self.ws)


def timed(fn, n, stream, flush, warm=3):
    """CUDA-event times (ms) of n calls of fn on `stream`, each after an L2
    flush outside its events, after `warm` untimed calls."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    with torch.cuda.stream(stream):
        for k in range(n + warm):
            flush.fill_(k & 0xFF)
            if k >= warm:
                ev[k - warm][0].record(stream)
            fn()
            if k >= warm:
                ev[k - warm][1].record(stream)
    stream.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def graphed(fn, stream):
    """fn captured once into a CUDA graph; returns its replay."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g.replay


def run_profile(tv, step, cfg, args, dev):
    """--profile: the chosen call alone, warmup + steps times on the default
    stream, checked once, for a profiler to capture (say the last launch)."""
    import torch
    f = fp8_inputs(step.d) if args.profile == "attention_fp8" else None
    if args.profile == "retained" and not cfg.get("mask_mass"):
        raise SystemExit(f"--profile retained: workload {cfg['name']} does not prune")
    call = {"attention": step.attn, "attention_fp8": lambda: step.attn_fp8(f), "accept": step.acc,
            "retained": lambda: tv.retained_set(step.d["draft"], float(cfg["mask_mass"]))}[args.profile]
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    if args.profile.startswith("attention"):
        assert int(step.st_attn.max()) == 0, "attention status"
    print(f"profile {args.profile}: {cfg['name']} (config {cfg['num']}, batch {cfg['batch']}), "
          f"{args.warmup + args.steps} launches", flush=True)


def time_retained(tv, d, cfg, rows, nb, stream, flush, peaks):
    """tv_retained_set of every draft row of a workload that prunes, timed on
    its own; the masks must equal the workload's."""
    import torch
    res = {}
    r_ms = timed(lambda: res.__setitem__("m", tv.retained_set(d["draft"], float(cfg["mask_mass"]))),
                 nb, stream, flush)
    assert torch.equal(res["m"][0], d["mask"]), "retained set differs from the workload's masks"
    r_s = statistics.mean(r_ms) / 1e3
    r_bytes = rows * int(cfg["vocab"]) * 4 + res["m"][0].numel() * 4
    return {"workload": f"{cfg['name']} (config {cfg['num']})", "mean_us": r_s * 1e6, "rows": rows,
            "bytes": r_bytes, "achieved_gbs": r_bytes / r_s / 1e9, "frac": r_bytes / r_s / 1e9 / peaks[0],
            "note": "tv_retained_set of every draft row (one CTA per row), timed on its own"}


def kernel_entries(step, attn_ms, acc_ms, peaks, cfg_num):
    """Roofline of the attention call and the HBM fraction of the accept call."""
    peak_bw, peak_tf, peak_kind = peaks
    case = step.case
    a_bytes, a_flops = attention_bytes(case), attention_flops(case)
    attn_s = statistics.mean(attn_ms) / 1e3
    acc_s = statistics.mean(acc_ms) / 1e3
    ab = accept_bytes(case)
    src = "of measured (MEASURED_PEAKS.json)" if peak_kind == "measured" else "of fallback"
    roof = dict({"kernel": "tree_attn_kernel (+ status and counter memsets)"},
                **roofline_entry(a_bytes, a_flops, attn_s, peak_bw, peak_tf, peak_kind),
                traffic=ncu_traffic(cfg_num), algorithmic_bytes=a_bytes, flops=a_flops,
                mean_us=attn_s * 1e6, hbm_gbs=a_bytes / attn_s / 1e9,
                hbm_frac=a_bytes / attn_s / 1e9 / peak_bw,
                tflops=a_flops / attn_s / 1e12, tensor_frac=a_flops / attn_s / 1e12 / peak_tf)
    acc = {"mean_us": acc_s * 1e6, "trees_per_s": step.B / acc_s,
           "accepted_tokens_per_s": float(step.acc_out["accepted_len"].sum().item()) / acc_s,
           "algorithmic_bytes": ab, "achieved_gbs": ab / acc_s / 1e9,
           "peak": peak_bw, "frac": ab / acc_s / 1e9 / peak_bw,
           "peak_source": src + " hbm_gbs", "bound": "hbm"}
    return roof, acc


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return

    import torch
    import speculative_decoding_tree_attention_gb300 as tv
    from speculative_decoding_tree_attention_gb300 import _build

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    _build.build()
    tv.load()
    peaks = load_peaks()

    cfg = wl.config(args.config, **({"batch": args.batch} if args.batch > 0 else {}))
    case = wl.make_case(cfg, parts=("attn", "accept"), kind=args.mode)
    # the other HBM-bound workloads, reported beside the headline (rank 0)
    side_nums = [n for n in (4, 3, 2) if n != cfg["num"]] if (rank == 0 and args.side and not args.profile) else []
    side_cases = {n: wl.make_case(wl.config(n), parts=("attn", "accept"), kind=args.mode)
                  for n in side_nums}
    step = Step(tv, case, cfg, args.mode, dev)
    tot, B = step.tot, step.B
    if args.profile:
        run_profile(tv, step, cfg, args, dev)
        return

    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    clocks = Clocks(vis[local] if local < len(vis) and vis[local].strip().isdigit() else local)
    t_load0 = time.time()

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step.attn()
            step.acc()
        stream.synchronize()
        step.check()
        run_step = run_attn = run_acc = None
        if not args.no_graph:
            # the step (attention then accept) as one graph; and each call as
            # its own graph for the per-kernel breakdown
            run_step = graphed(lambda: (step.attn(), step.acc()), stream)
            run_attn = graphed(step.attn, stream)
            run_acc = graphed(step.acc, stream)
            for _ in range(max(3, args.warmup)):
                run_step()
                run_attn()
                run_acc()
            stream.synchronize()
        else:
            run_step = lambda: (step.attn(), step.acc())
            run_attn, run_acc = step.attn, step.acc

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            flush.fill_(k & 0xFF)  # evicts the inputs from L2 (outside the events)
            e0, e1 = ev[k]
            e0.record(stream)
            run_step()
            e1.record(stream)
    stream.synchronize()
    wall = time.perf_counter() - t_wall0
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_s = sum(step_ms) / 1e3
    # per-call breakdown (same flushing), for the roofline of each kernel
    nb = max(3, min(args.steps, 100))
    attn_ms = timed(run_attn, nb, stream, flush)
    acc_ms = timed(run_acc, nb, stream, flush)
    if world > 1:
        total_s = max_over_ranks(total_s, dev)
    roof, acc_entry = kernel_entries(step, attn_ms, acc_ms, peaks, cfg["num"])

    # ---- the other HBM-bound workloads: each call timed on its own, as above
    side = {}
    for n, c in side_cases.items():
        st = Step(tv, c, wl.config(n), args.mode, dev)
        with torch.cuda.stream(stream):
            st.attn()
            st.acc()
        stream.synchronize()
        st.check()
        ra = graphed(st.attn, stream) if not args.no_graph else st.attn
        rc = graphed(st.acc, stream) if not args.no_graph else st.acc
        a_ms = timed(ra, nb, stream, flush, warm=5)
        c_ms = timed(rc, nb, stream, flush, warm=5)
        r, a = kernel_entries(st, a_ms, c_ms, peaks, n)
        side[f"{wl.config(n)['name']} (config {n})"] = {
            "tree_nodes": st.tot, "attention": r, "accept": a,
            "step_us": (statistics.mean(a_ms) + statistics.mean(c_ms)) * 1e3,
            "plan": tv.attention_plan(st.prm),
            "retained_set": time_retained(tv, st.d, wl.config(n), st.tot, nb, stream, flush, peaks)
            if wl.config(n).get("mask_mass") else None}
        del st, ra, rc
    # ---- FP8 tree attention (E4M3 inputs, [EC] §9.2) on the headline workload
    # and on serving: half the K/V bytes
    fp8 = {}
    fp8_runs = ((("headline", step),) if cfg["d"] == 128 else ()) + \
        (((f"{wl.config(3)['name']} (config 3)", None),) if 3 in side_cases else ())
    for name, st in fp8_runs:
        if st is None:
            st = Step(tv, side_cases[3], wl.config(3), args.mode, dev)
        f = fp8_inputs(st.d)
        with torch.cuda.stream(stream):
            st.attn_fp8(f)
        stream.synchronize()
        assert int(st.st_attn.max()) == 0, "fp8 attention status"
        rf = graphed(lambda: st.attn_fp8(f), stream) if not args.no_graph else (lambda: st.attn_fp8(f))
        f_ms = timed(rf, nb, stream, flush, warm=5)
        f_s = statistics.mean(f_ms) / 1e3
        fb, ff = attention_bytes_fp8(st.case), attention_flops(st.case)
        fp8[name if st is not step else f"{cfg['name']} (config {cfg['num']})"] = {
            "mean_us": f_s * 1e6, "algorithmic_bytes": fb, "hbm_gbs": fb / f_s / 1e9,
            "hbm_frac": fb / f_s / 1e9 / peaks[0], "tflops": ff / f_s / 1e12,
            "note": "tv_tree_attention_fp8: E4M3 Q/K/V, one scale per 128-code row"}
        del f, rf
        if st is not step:
            del st
    torch.cuda.synchronize()
    clocks.load(t_load0, time.time())
    clk = clocks.stop()

    # ---- commit of the accepted path (the step after the walk; reported on its
    # own, not part of the timed step): the root and the accepted nodes of the
    # last step's accept results go into fresh pages of an extended pool
    d, max_nodes = step.d, step.max_nodes
    acc_out = step.acc_out
    kpx, vpx, tabx = wl.extend_pool(case, max_nodes + 1)
    cm = {"kp": torch.from_numpy(kpx.view(np.int16)).to(dev).view(torch.bfloat16),
          "vp": torch.from_numpy(vpx.view(np.int16)).to(dev).view(torch.bfloat16),
          "table": torch.from_numpy(tabx).to(dev)}
    del kpx, vpx
    cm_out = (torch.empty(B, dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev))
    commit_ms = timed(lambda: tv.commit_kv(d["kn"], d["vn"], d["parent"], d["off"],
                                           acc_out["accepted_len"], acc_out["path"], cm["table"],
                                           d["lens"], cm["kp"], cm["vp"], max_nodes=max_nodes,
                                           new_prefix_lens=cm_out[0], status=cm_out[1]),
                      nb, stream, flush)
    assert int(cm_out[1].max()) == 0, "commit status"
    commit_tokens = int(acc_out["accepted_len"].sum().item()) + B
    del cm
    # ---- retained set of the draft rows (the step before the accept pass's
    # renormalisation, for workloads that prune): reported on its own
    retained = time_retained(tv, d, cfg, tot, nb, stream, flush, peaks) if cfg.get("mask_mass") else None
    if retained is None:
        retained = next((w["retained_set"] for w in side.values() if w.get("retained_set")), None)
    # ---- the multi-candidate accept variant (siblings tried in order with
    # residual updates) on the same inputs, reported on its own
    m_out = {k: torch.empty_like(v) for k, v in acc_out.items()}
    m_ms = timed(lambda: step.acc(test="multi", outputs=m_out), nb, stream, flush)
    assert int(m_out["status"].max()) == 0, "multi-candidate accept status"
    m_s = statistics.mean(m_ms) / 1e3
    multi = {"mean_us": m_s * 1e6, "trees_per_s": B / m_s,
             "mean_accepted_len": float(m_out["accepted_len"].float().mean().item()),
             "mean_accepted_len_single": float(acc_out["accepted_len"].float().mean().item()),
             "note": "tv_accept_ex with TV_TEST_MULTI on the step's inputs, timed on its own"}
    del m_out

    # ---- end to end through the public API with host buffers
    host = step.host
    pinned = {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory() for k, v in host.items()}
    e2e_src = {k: torch.empty_like(d[k].view(pinned[k].dtype)) for k in host}
    res_host = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in acc_out.items()}
    h2d = sum(v.numel() * v.element_size() for v in pinned.values())
    d2h = sum(v.numel() * v.element_size() for v in res_host.values())
    e2e_steps = max(3, min(args.steps, 50))
    with torch.cuda.stream(stream):
        src = dict(e2e_src)
        for k in ("q", "kp", "vp", "kn", "vn"):
            src[k] = e2e_src[k].view(torch.bfloat16)
        for _ in range(2):
            for k in host:
                e2e_src[k].copy_(pinned[k], non_blocking=True)
            step.attn(src)
            step.acc(src)
        stream.synchronize()
        e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_a.record(stream)
        for _ in range(e2e_steps):
            for k in host:
                e2e_src[k].copy_(pinned[k], non_blocking=True)
            step.attn(src)
            step.acc(src)
            for k in res_host:
                res_host[k].copy_(acc_out[k], non_blocking=True)
        e_b.record(stream)
    stream.synchronize()
    e2e_s = e_a.elapsed_time(e_b) / 1e3

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    value = world * tot * args.steps / total_s
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes of the pages' workloads, no datasets or weights)",
        "config": dict(workload_desc(cfg, case), accept_input=args.mode,
                       l2="flushed between timed steps (512 MiB write)",
                       launch="one CUDA graph per step" if not args.no_graph else "eager",
                       parallelism="replicas" if world > 1 else "single GPU",
                       attention_plan=tv.attention_plan(step.prm)),
        "roofline": roof,
        "accept": acc_entry,
        "workloads": side,
        "fp8_attention": fp8,
        "e2e": {"value": world * tot * e2e_steps / e2e_s, "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": step.launches_per_step * args.steps,
        "percentiles_us": {"step": pct(step_ms), "attention": pct(attn_ms), "accept": pct(acc_ms)},
        "retained_set": retained,
        "accept_multi": multi,
        "commit": {"mean_us": statistics.mean(commit_ms) * 1e3, "tokens": commit_tokens,
                   "bytes": commit_tokens * 8 * cfg["hkv"] * cfg["d"],  # K+V rows read and written
                   "note": "tv_commit_kv of the root and accepted path, timed on its own"},
        "clocks": clk,
        "wall_s_timed_loop": wall,
    }
    if world == 1 and args.cpu_seconds > 0:
        cb = cpu_baseline(case, args.cpu_seconds)
        one = cpu_baseline(case, max(1.0, args.cpu_seconds / 4), threads=1)
        cb["single_thread"] = {"value": one["value"], "unit": one["unit"], "sample": one["sample"]}
        line["cpu_baseline"] = cb
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
