"""Benchmark of the verify step on the large-batch workload.

Workload (one "step" = one verify round over the whole batch):
  B = 256 sequences, gamma = 8 drafts, V = 128256 (LLaMA-3 vocabulary),
  fp32 logits; target ~ N(0, 3^2), draft = target + N(0, 1); draft tokens
  drawn from softmax(draft / T); T = 1.0; uniforms from splitmix64.
  Geometric fan-out a = 0.8, r = 1, K = 8, budget 64 -> F = [10,9,8,7,6,6,
  5,4,9] on the 9 draft rows, on a second stream beside the verify.

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU
oracle on the same workload instead (the only reference this method has).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from speculative_decoding_verification_temperature_gb300 import synth  # noqa

METRIC = ("verify rounds/s and achieved HBM GB/s over logits vs ~8 TB/s "
          "roofline (1 GB300)")
B, GAMMA, V, T = 256, 8, 128256, 1.0
FAN = dict(K=8, budget=64, a=0.8, r=1.0)
ELT = 4
WORKLOAD = ("large-batch verify + fan-out: B=256, gamma=8, V=128256, fp32, "
            "T=1.0, fan-out a=0.8 r=1 K=8 budget=64")
FALLBACK_HBM = 6800.0


# ------------------------------------------------------------ clocks
class ClockSampler:
    """Samples SM clock and throttle reasons through NVML (ctypes) every
    ~2 ms while running; reading only, no setting is touched."""
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown",
               0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap",
               0x80: "hw_power_brake_slowdown", 0x1: "gpu_idle"}

    def __init__(self, index=0):
        self.ok = False
        self.samples = []
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByIndex_v2(
                    ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
                return
            self.ok = True
            mx = ctypes.c_uint()
            self.nv.nvmlDeviceGetMaxClockInfo(self.h, ctypes.c_uint(1),
                                              ctypes.byref(mx))
            self.max_mhz = mx.value
        except OSError:
            pass

    def _read(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        self.nv.nvmlDeviceGetClockInfo(self.h, ctypes.c_uint(1),
                                       ctypes.byref(c))
        self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h,
                                                       ctypes.byref(r))
        return c.value, r.value

    def start(self):
        self.samples = []
        self._stop = threading.Event()
        if not self.ok:
            return
        def loop():
            while not self._stop.is_set():
                self.samples.append(self._read())
                time.sleep(0.002)
        self.t = threading.Thread(target=loop, daemon=True)
        self.t.start()

    def stop(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "source": "unavailable"}
        self._stop.set()
        self.t.join()
        mhz = [s[0] for s in self.samples] or [0]
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit and name != "gpu_idle":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(self.samples),
                "source": "nvml"}


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch
# from one ncu capture of each kernel on B=128 sequences of this workload
# (profiles/), with the units that launch processed: the fan-out reads every
# row once, so its traffic scales with the rows; the verify's and the fused
# step's with the bytes the method needs (the early exit decides how many
# rows they read).  The verify's includes the rows that clusters helping in
# the tail read ahead.
TRAFFIC = {"fanout": (591.25e6, 128 * 9), "linear": (565.0e6, 343.73e6),
           "fused": (881.2e6, 763.89e6)}


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM, "fallback"


def needed_bytes(n, gamma, V, elt):
    """Logit bytes the method must read for one round: target rows 0..n and
    draft rows 0..min(n, gamma-1) of every sequence."""
    n = np.asarray(n, np.int64)
    rows = (n + 1) + np.minimum(n + 1, gamma)
    return int(rows.sum()) * V * elt


# ---------------------------------------------------------- GPU arm
def workload_name():
    if B == 256:
        return WORKLOAD
    return WORKLOAD.replace("B=256", "B=%d (profiling case)" % B)


def make_sets(nsets, device, rank=0):
    """The rotated input sets of one rank (each rank verifies its own
    batches)."""
    sets = []
    for s in range(nsets):
        c = synth.large(s + 16 * rank, device=device, B=B)
        c.draft_v = c.draft[:, :GAMMA].contiguous()
        sets.append(c)
    return sets


def max_over_ranks(ms, world, dev):
    """The timed region's length as the slowest rank saw it."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(steps, total_ms, world):
    """Rounds per second of the whole job: every rank verifies its own batch
    each step (replicas, weak scaling), so world * steps rounds took
    total_ms (the slowest rank's time)."""
    return world * steps / (total_ms / 1e3)


def gpu_arm(args, rank, world):
    from speculative_decoding_verification_temperature_gb300 import api
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    sets = make_sets(args.sets, dev, rank)
    stream = torch.cuda.current_stream(dev)
    ws = api.Workspace()
    F = api.fanout_schedule(FAN["K"], FAN["budget"], FAN["a"], FAN["r"])

    def verify(c):
        return api.verify_linear(c.target, c.draft_v, c.tokens, c.uniforms,
                                 T, workspace=ws)

    ws_f = api.Workspace()  # the fan-out's own scratch (it runs beside)

    def fanout(c):
        return api.fanout_topk(c.draft, F, workspace=ws_f)

    ws_x = api.Workspace()

    def fused(c):  # the verify and the fan-out in one launch
        return api.verify_linear_fanout(c.target, c.draft, c.tokens,
                                        c.uniforms, T, F, workspace=ws_x)

    # bytes the method needs per set (deterministic outputs): target rows
    # 0..n of every sequence and all K+1 draft rows (the fan-out reads them
    # all; the verify's draft rows are a subset)
    need, need_v = [], []
    for c in sets:
        n = verify(c)["n"].cpu().numpy().astype(np.int64)
        fanout(c)
        need_v.append(needed_bytes(n, GAMMA, V, ELT))
        need.append(int((n + 1).sum()) * V * ELT + B * (FAN["K"] + 1) * V * ELT)
    for i in range(args.warmup):
        verify(sets[i % len(sets)])
        fanout(sets[i % len(sets)])
        fused(sets[i % len(sets)])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    side = torch.cuda.Stream(dev)

    if args.step == "fused":
        # the step: sd_verify_linear_fanout, one launch; CTAs left without a
        # sequence to verify take the fan-out's rows
        def step(c):
            fused(c)
    else:
        # the two calls, the fan-out on a second stream beside the verify
        # (each with its own workspace), joined before the next step
        def step(c):
            fork = torch.cuda.Event()
            fork.record(stream)
            side.wait_event(fork)
            with torch.cuda.stream(side):
                fanout(c)
            verify(c)
            join = torch.cuda.Event()
            join.record(side)
            stream.wait_event(join)

    for i in range(args.warmup):
        step(sets[i % len(sets)])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    # timing events only at the ends of blocks of steps: a timing event
    # between two steps keeps the next step's fan-out from overlapping the
    # verify (measured: 392 instead of 364 us per step)
    blk = 20 if args.steps >= 40 else args.steps
    bounds = list(range(0, args.steps, blk)) + [args.steps]
    ev = [torch.cuda.Event(enable_timing=True) for _ in bounds]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    nb = 0
    for i in range(args.steps):
        if i == bounds[nb]:
            ev[nb].record(stream)
            nb += 1
        step(sets[i % len(sets)])
    ev[-1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(ev[0].elapsed_time(ev[-1]), world, dev)
    ms = total_ms / args.steps
    per = np.array([ev[k].elapsed_time(ev[k + 1]) / (bounds[k + 1] - bounds[k])
                    for k in range(len(bounds) - 1)])  # ms per step, per block
    q1, med, q3 = (float(x) for x in np.percentile(per, [25, 50, 75]))
    # each kernel alone (the same K steps run one call after the other), for
    # the per-kernel roofline
    evk = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
           for _ in range(args.steps)]
    for i in range(args.steps):
        c = sets[i % len(sets)]
        evk[i][0].record(stream)
        verify(c)
        evk[i][1].record(stream)
        fanout(c)
        evk[i][2].record(stream)
    torch.cuda.synchronize()
    ms_v = sum(e[0].elapsed_time(e[1]) for e in evk) / args.steps
    ms_f = sum(e[1].elapsed_time(e[2]) for e in evk) / args.steps
    ms_seq = sum(e[0].elapsed_time(e[2]) for e in evk) / args.steps
    rounds_s = whole_job_rate(args.steps, total_ms, world)
    avg = lambda xs: sum(xs[i % len(sets)] for i in range(args.steps)) / args.steps
    need_avg, need_v_avg = avg(need), avg(need_v)
    fan_bytes = B * (FAN["K"] + 1) * V * ELT
    tensor_bytes = B * (GAMMA + 1) * V * ELT + fan_bytes
    peak, src = hbm_peak()
    # dominant kernel: the fused launch (the whole step), else the larger of
    # the two calls' shares
    if args.step == "fused":
        kern, kb, kms = ("linear_verify_kernel<0,4,false,true,true> (fused "
                         "with the fan-out)", need_avg, ms)
        traffic = (TRAFFIC["fused"][0] / TRAFFIC["fused"][1] * need_avg
                   if TRAFFIC.get("fused") else None)
    elif ms_v >= ms_f:
        kern, kb, kms = "linear_verify_kernel<0,4,false,true>", need_v_avg, ms_v
        traffic = TRAFFIC["linear"][0] / TRAFFIC["linear"][1] * need_v_avg
    else:
        kern, kb, kms = "fanout_kernel<0,4,true>", fan_bytes, ms_f
        traffic = TRAFFIC["fanout"][0] / TRAFFIC["fanout"][1] * B * (FAN["K"] + 1)
    achieved = kb / (kms / 1e3) / 1e9
    res = {
        "metric": METRIC, "value": rounds_s, "unit": "rounds/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_name(), "B": B, "gamma": GAMMA, "V": V,
                   "T": T, "fanout_F": F, "input_sets": len(sets),
                   "step": ("sd_verify_linear_fanout: the verify and the "
                            "fan-out in one launch" if args.step == "fused"
                            else "sd_verify_linear with sd_fanout_topk on a "
                                 "second stream (joined each step)"),
                   "l2": "inputs %.2f GB per set (> 129 MB L2), %d sets "
                         "rotated" % (2 * B * (GAMMA + 1) * V * ELT / 1e9,
                                      len(sets)),
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic,
                     "traffic_source": "ncu capture on B=128 (profiles/), "
                                       "scaled by the units processed",
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (%s)" % src,
                     "kernel": kern, "bytes_per_launch": kb,
                     "ms_per_launch": kms},
        "step_bytes_read": need_avg,
        "step_gbs": need_avg / (ms / 1e3) / 1e9,
        "step_frac": need_avg / (ms / 1e3) / 1e9 / peak,
        "full_tensor_bytes": tensor_bytes,
        "ms_per_step_median": med,
        "ms_per_step_iqr": [q1, q3],
        "ms_per_step_stats": "median and quartiles over blocks of %d steps"
                             % blk,
        "sequential_ms_per_step": ms_seq,
        "verify": {"ms": ms_v, "bytes": need_v_avg,
                   "gbs": need_v_avg / (ms_v / 1e3) / 1e9},
        "fanout": {"ms": ms_f, "bytes": fan_bytes,
                   "gbs": fan_bytes / (ms_f / 1e3) / 1e9},
        "gpu_launches": (1 if args.step == "fused" else 2) * args.steps,
        "tuning": {k: api.tune_get(k) for k in api.TUNE},
        "clocks": clk,
        "wall_s": wall,
    }
    if args.e2e_steps > 0:
        res["e2e"] = e2e_arm(args, sets, dev, ws, world, F)
    checks = [] if rank == 0 and args.oracle_seqs > 0 else None
    if args.aux_steps > 0:
        res["other_workloads"] = other_workloads(args, dev, peak, checks)
    if rank == 0 and args.oracle_seqs > 0:
        c = sets[0]
        if args.step == "fused":
            g = {k: v.cpu().numpy() for k, v in fused(c).items()}
        else:
            g = {k: v.cpu().numpy() for k, v in verify(c).items()}
            g["fan_tokens"] = fanout(c)["tokens"].cpu().numpy()
        res["cpu_baseline"], res["flagged"] = cpu_baseline(
            sets, args.oracle_seqs, F, g)
        res["flagged"]["what"] = (
            "oracle over one round of the step's inputs: accept tests within "
            "1e-5 of their threshold per accept test made, final draws "
            "within 1e-5 of a CDF boundary per draw (and those whose token "
            "differs from the oracle's, inside its admissible range); "
            "mismatches = sequences differing from the oracle elsewhere")
        for name, kind, case, out, Tw, extra in checks or []:
            res["other_workloads"][name]["flagged"] = oracle_check(
                kind, case, out, Tw, extra)
    return res


def e2e_arm(args, sets, dev, ws, world, F):
    """Same metric through the public API with host buffers: per step the
    pinned-host inputs are copied to the device, verified, and the results
    copied back.  The copies run on their own stream into two device input
    sets used in turn, so step i+1's inputs cross the host link while step i
    is verified (the link, not the GPU, bounds this number); every step's
    copies are inside the timed region.  The plain copies alone are timed
    too, as the link's bound."""
    from speculative_decoding_verification_temperature_gb300 import api
    c = sets[0]
    h = {k: getattr(c, k).cpu().pin_memory()
         for k in ("target", "draft", "tokens", "uniforms")}
    d = [{k: torch.empty_like(v, device=dev) for k, v in h.items()}
         for _ in range(2)]
    dv = [torch.empty((B, GAMMA, V), dtype=h["draft"].dtype, device=dev)
          for _ in range(2)]
    out_h = {"n": torch.empty(B, dtype=torch.int32).pin_memory(),
             "tokens": torch.empty((B, GAMMA + 1),
                                   dtype=torch.int32).pin_memory(),
             "prob": torch.empty(B, dtype=torch.float32).pin_memory(),
             "fan_tokens": torch.empty((B, sum(F)),
                                       dtype=torch.int32).pin_memory()}
    stream = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    used = [torch.cuda.Event() for _ in range(2)]
    for e in used:
        e.record(stream)
    steps = max(3, min(args.steps, args.e2e_steps))

    def load(i):
        s = i % 2
        copy.wait_event(used[s])  # step i-2 is done with this set
        with torch.cuda.stream(copy):
            for k in h:
                d[s][k].copy_(h[k], non_blocking=True)
        copied[s].record(copy)

    wsx = api.Workspace()

    def step(i):
        s = i % 2
        stream.wait_event(copied[s])
        if args.step == "fused":
            o = api.verify_linear_fanout(d[s]["target"], d[s]["draft"],
                                         d[s]["tokens"], d[s]["uniforms"], T,
                                         F, workspace=wsx)
        else:
            dv[s].copy_(d[s]["draft"][:, :GAMMA])
            o = api.verify_linear(d[s]["target"], dv[s], d[s]["tokens"],
                                  d[s]["uniforms"], T, workspace=ws)
            o["fan_tokens"] = api.fanout_topk(d[s]["draft"], F,
                                              workspace=ws)["tokens"]
        used[s].record(stream)
        for k in out_h:
            out_h[k].copy_(o[k], non_blocking=True)

    def run(n):
        load(0)
        for i in range(n):
            if i + 1 < n:
                load(i + 1)
            step(i)

    run(max(3, args.warmup))  # first host-to-device copies after pinning
    torch.cuda.synchronize()  # run slower
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(
        enable_timing=True)
    a.record(stream)
    copy.wait_stream(stream)  # no copy starts before the timed region
    run(steps)
    stream.wait_stream(copy)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    # the host-to-device copies alone, same bytes, same stream
    a.record(copy)
    for i in range(steps):
        with torch.cuda.stream(copy):
            for k in h:
                d[i % 2][k].copy_(h[k], non_blocking=True)
    b.record(copy)
    torch.cuda.synchronize()
    ms_copy = a.elapsed_time(b)
    h2d = sum(v.numel() * v.element_size() for v in h.values())
    d2h = sum(v.numel() * v.element_size() for v in out_h.values())
    return {"value": world * steps / (ms / 1e3), "unit": "rounds/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps,
            "h2d_only": {"ms_per_step": ms_copy / steps,
                         "gbs": h2d * steps / (ms_copy / 1e3) / 1e9,
                         "rounds_s": world * steps / (ms_copy / 1e3)},
            "overlap": "inputs double-buffered: step i+1's host-to-device "
                       "copy runs on its own stream beside step i"}


# ------------------------------------------------- the other workloads
def _rows_linear(n, gamma, greedy):
    n = np.asarray(n, np.int64)
    return int(((n + 1) + (0 if greedy else np.minimum(n + 1, gamma))).sum())


def _rows_kcand(npc, n, gamma):
    npc = np.asarray(npc, np.int64)
    n = np.asarray(n, np.int64)
    tgt = np.minimum(npc + 1, gamma).sum(1) + (n == gamma)
    drf = np.minimum(n + 1, gamma)
    return int((tgt + drf).sum())


def _rows_tree(parent, nodes, n, greedy):
    parent = np.asarray(parent)
    rows = 0
    for b in range(parent.shape[0]):
        visited = [0] + [int(v) for v in nodes[b, :n[b]]]
        for u in visited:
            rows += 1
            if not greedy and np.any(parent[b] == u):
                rows += 1
    return rows


def _time_graph(fn, sets, steps, warmup, dev):
    """Device time per round with the `steps` calls captured once in a CUDA
    graph and replayed (a small round is shorter than the host's cost of
    one call).  Falls back to the host loop if capture fails; returns
    (ms, how)."""
    for i in range(warmup):  # also fills the library's per-kernel caches
        fn(sets[i % len(sets)])
    torch.cuda.synchronize()
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(steps):
                fn(sets[i % len(sets)])
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        s = torch.cuda.current_stream(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s)
        g.replay()
        b.record(s)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps, "cuda graph of %d calls" % steps
    except RuntimeError as e:
        torch.cuda.synchronize()
        return _time(fn, sets, steps, 0, dev), "host loop (%s)" % str(e)[:60]


def _time(fn, sets, steps, warmup, dev):
    stream = torch.cuda.current_stream(dev)
    for i in range(warmup):
        fn(sets[i % len(sets)])
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(steps):
        fn(sets[i % len(sets)])
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps  # ms per round


def other_workloads(args, dev, peak, checks=None):
    """rounds/s, logit bytes the method read (counted from the outputs) and
    the HBM fraction for the other workloads, measured in this run.  When
    `checks` is a list, each workload appends one input set and its GPU
    outputs to it, for the oracle comparison of the CPU-baseline leg."""
    from speculative_decoding_verification_temperature_gb300 import api
    out = {}
    steps = args.aux_steps
    args.checks = checks

    def entry(name, ms, rows, V, elt, full_rows, extra=None):
        gbs = rows * V * elt / (ms / 1e3) / 1e9
        e = {"rounds_s": 1e3 / ms, "ms_per_round": ms,
             "bytes_read": rows * V * elt,
             "full_tensor_bytes": full_rows * V * elt,
             "achieved_gbs": gbs, "frac_of_measured_hbm": gbs / peak}
        if extra:
            e.update(extra)
        out[name] = e

    want = lambda name: not args.only or args.only == name
    if want("tiny"):
        _tiny(args, dev, entry, steps)
    if want("linear"):
        _linear(args, dev, entry, steps)
    if want("kcand"):
        _kcand(args, dev, entry, steps)
    if want("tree"):
        _tree(args, dev, entry, steps)
    if want("filtered"):
        _filtered(args, dev, entry, steps)
    if want("cache_hit"):
        out["cache_hit"] = _cache_hit(args, dev)
    if want("presto"):
        _presto(args, dev, entry, steps)
    if want("fork"):
        _fork(args, dev, entry, steps)
    return out


def _presto(args, dev, entry, steps):
    """PRESTO tree construction on the tree workload's shape: B=16, V=151936
    bf16, 8 depths, W=8 paths, b=4 tokens per path, a 64-node budget,
    T=0.8, lambda=1; synthetic drafter marginals N(0, 2^2) and log rho of
    U(0.01, 1).  One round = sd_presto_init + 8 sd_presto_expand calls."""
    from speculative_decoding_verification_temperature_gb300 import api
    B, D, W, V, b_top, budget = 16, 8, 8, 151936, 4, 64
    sets = []
    for r in range(2):
        g = torch.Generator(device=dev).manual_seed(700 + r)
        q = (torch.randn((B, D, V), generator=g, device=dev) * 2.0).to(
            torch.bfloat16)
        rho = torch.log(torch.rand((D, B, W, V), generator=g, device=dev) *
                        0.99 + 0.01).to(torch.bfloat16)  # depth-major
        sets.append((q, rho))
    state = {}

    def fn(c):
        q, rho = c
        t = api.PrestoTree(B, W, budget, dev)
        for d in range(D):
            api.presto_expand(t, q[:, d], rho[d], 0.8, 1.0, b_top)
        state["t"] = t
    # one round is 17 small launches: timed as a CUDA graph, as a serving
    # loop with a fixed depth would run it (the host's per-call cost is
    # larger than a depth's device time)
    ms, how = _time_graph(fn, sets, 20, 3, dev)
    # bytes: a depth that runs (node budget not yet spent) reads the
    # sequence's q row once and the log rho rows of its frontier paths (the
    # nodes of that depth, at most W), counted from the built trees
    rows = 0
    for c in sets:
        fn(c)
        par = state["t"].parent.cpu().numpy()
        n = state["t"].n_nodes.cpu().numpy()
        for bi in range(B):
            depth = np.zeros(n[bi], np.int64)
            for v in range(1, n[bi]):
                depth[v] = depth[par[bi, v]] + 1
            for d in range(D):
                if (depth <= d).sum() >= budget:
                    break
                rows += 1 + min(W, int((depth == d).sum()))
    entry("presto_build", ms, rows / len(sets), V, 2, B * D + B * D * W,
          {"nodes": int(n.sum()), "timing": how})


def _fork(args, dev, entry, steps):
    """SpecBranch fork on B=64 rows of V=152064 bf16 (N(0, 2.5^2) logits),
    k_max=8, T=1, x_b the drafted (argmax) token for half the rows and a
    random one for the rest; timed as a CUDA graph."""
    from speculative_decoding_verification_temperature_gb300 import api
    B, V = 64, 152064
    sets = []
    for r in range(8):
        g = torch.Generator(device=dev).manual_seed(800 + r)
        z = (torch.randn((B, V), generator=g, device=dev) * 2.5).to(
            torch.bfloat16)
        x = torch.randint(0, V, (B,), generator=g, device=dev,
                          dtype=torch.int32)
        x[: B // 2] = torch.argmax(z[: B // 2].float(), 1).int()
        sets.append((z, x))
    out = {}

    def fn(c):
        out["o"] = api.branch_fork(c[0], c[1], 1.0, 8)
    ms, how = _time_graph(fn, sets, 200, 5, dev)
    fn(sets[0])
    entry("branch_fork", ms, B, V, 2, B,
          {"timing": how,
           "mean_k": float(out["o"]["k"].float().mean())})


def _filtered(args, dev, entry, steps):
    """Filtered sampling on the large workload's shape: B=256, gamma=8,
    V=128256 fp32, T=1: top_k = 50 with top_p = 0.9 (exact top-k lists),
    top_p = 0.9 alone and top_k = 1000 alone (the threshold select)."""
    from speculative_decoding_verification_temperature_gb300 import api
    sets = []
    for r in range(min(2, args.sets)):
        c = synth.large(r, device=dev, B=B)
        c.draft = c.draft[:, :GAMMA].contiguous()
        sets.append(c)
    for name, top_k, top_p in (("filtered_k50_p0.9", 50, 0.9),
                               ("filtered_p0.9", V, 0.9),
                               ("filtered_k1000", 1000, 1.0)):
        fn = (lambda c, k=top_k, pp=top_p: api.verify_linear_filtered(
            c.target, c.draft, c.tokens, c.uniforms, 1.0, k, pp))
        ms = _time(fn, sets, steps, 3, dev)
        rows = np.mean([_rows_linear(fn(c)["n"].cpu().numpy(), GAMMA, False)
                        for c in sets])
        entry(name, ms, rows, V, ELT, B * (2 * GAMMA + 1),
              {"top_k": top_k, "top_p": top_p, "T": 1.0})
        _register(args, name, "filtered", sets[0],
                  api.verify_linear_filtered(sets[0].target, sets[0].draft,
                                             sets[0].tokens,
                                             sets[0].uniforms, 1.0, top_k,
                                             top_p, want_keep=True),
                  1.0, top_k=top_k, top_p=top_p)
    del sets


def uniform_schedule(K, budget):
    """budget / (K+1) per position, the remainder to the lowest positions."""
    F = [budget // (K + 1)] * (K + 1)
    for k in range(budget - sum(F)):
        F[k] += 1
    return F


def _cache_hit(args, dev):
    """Saguaro cache-hit rate of the verification outcomes on the large
    workload's shape: verify, fan-out with the geometric schedule and with
    a uniform one of the same budget, then sd_fanout_hits."""
    from speculative_decoding_verification_temperature_gb300 import api
    Fg = api.fanout_schedule(FAN["K"], FAN["budget"], FAN["a"], FAN["r"])
    Fu = uniform_schedule(FAN["K"], FAN["budget"])
    res = {"F_geometric": Fg, "F_uniform": Fu, "B": B}
    for T in (0.0, 0.5, 1.0):
        c = synth.linear_case(B, GAMMA, V, torch.float32, T,
                              seed=1004 + int(T * 10), sigma_t=3.0,
                              sigma_d=1.0, draft_rows=GAMMA + 1, device=dev)
        v = api.verify_linear(c.target, None if T == 0 else
                              c.draft[:, :GAMMA].contiguous(), c.tokens,
                              c.uniforms, T)
        row = {"mean_accepted": float(v["n"].float().mean())}
        for name, F in (("geometric", Fg), ("uniform", Fu)):
            f = api.fanout_topk(c.draft, F)
            h = api.fanout_hits(v["n"], v["tokens"], f["tokens"], F)
            row[name] = float((h == 1).float().mean())
        res["T%g" % T] = row
        del c
    return res


def _tiny(args, dev, entry, steps):
    from speculative_decoding_verification_temperature_gb300 import api
    # tiny: B=1, gamma=4, V=1000 fp32 (launch-latency bound)
    sets = [synth.tiny(r, device=dev) for r in range(64)]
    fn = lambda c: api.verify_linear(c.target, c.draft, c.tokens,
                                     c.uniforms, 1.0)
    ms, how = _time_graph(fn, sets, max(steps, 200), 10, dev)
    rows = np.mean([_rows_linear(fn(c)["n"].cpu().numpy(), 4, False)
                    for c in sets[:16]])
    entry("tiny", ms, rows, 1000, 4, 9, {"note": "launch-latency bound",
                                          "timing": how})
    # the oracle check: 1000 tiny rounds in one batch (same inputs recipe)
    big = synth.linear_case(1000, 4, 1000, torch.float32, 1.0, seed=1000,
                            sigma_t=2.0, sigma_d=1.0, device=dev)
    _register(args, "tiny", "linear", big, fn(big), 1.0)


def _linear(args, dev, entry, steps):
    from speculative_decoding_verification_temperature_gb300 import api
    # linear: B=32, gamma=8, V=32000 bf16 at T in {0, 0.7, 1.0}; 16 sets
    # rotated (16 x 34.8 MB > 4 x L2)
    for T in (0.0, 0.7, 1.0):
        sets = [synth.linear(T, r, device=dev) for r in range(16)]
        for c in sets:
            c.draft = c.draft.contiguous()
        fn = (lambda c, T=T: api.verify_linear(
            c.target, None if T == 0 else c.draft, c.tokens, c.uniforms, T))
        ms, how = _time_graph(fn, sets, max(steps, 100), 10, dev)
        rows = np.mean([_rows_linear(fn(c)["n"].cpu().numpy(), 8, T == 0)
                        for c in sets])
        full = 32 * (9 if T == 0 else 17)
        entry("linear_T%g" % T, ms, rows, 32000, 2, full, {"timing": how})
        _register(args, "linear_T%g" % T, "linear", sets[0], fn(sets[0]), T)
        del sets


def _kcand(args, dev, entry, steps):
    from speculative_decoding_verification_temperature_gb300 import api
    # kcand: B=64, K=8, gamma=16, V=152064 bf16, T=1; 2 sets (2.9 GB each)
    sets = [synth.kcand(r, device=dev) for r in range(min(2, args.sets))]
    fn = lambda c: api.verify_kcand(c.target, c.draft, c.tokens, c.uniforms,
                                    1.0)
    ms = _time(fn, sets, steps, 3, dev)
    rows = []
    for c in sets:
        o = fn(c)
        rows.append(_rows_kcand(o["n_per_cand"].cpu().numpy(),
                                o["n"].cpu().numpy(), 16))
    acc = [float(fn(c)["n"].float().mean()) for c in sets]
    entry("kcand", ms, np.mean(rows), 152064, 2, 64 * (8 * 17 + 16),
          {"mean_accepted": float(np.mean(acc))})
    _register(args, "kcand", "kcand", sets[0], fn(sets[0]), 1.0)
    # the same candidates verified as one token tree (distribution-
    # preserving): target and draft rows of the visited nodes
    ft = lambda c: api.verify_kcand_trie(c.target, c.draft, c.tokens,
                                         c.uniforms, 1.0)
    ms = _time(ft, sets, steps, 3, dev)
    rows, acc = [], []
    for c in sets:
        n = ft(c)["n"].cpu().numpy().astype(np.int64)
        rows.append(int(((n + 1) + np.minimum(n + 1, 16)).sum()))
        acc.append(float(n.mean()))
    entry("kcand_trie", ms, np.mean(rows), 152064, 2, 64 * (8 * 17 + 16),
          {"mean_accepted": float(np.mean(acc))})
    _register(args, "kcand_trie", "kcand_trie", sets[0], ft(sets[0]), 1.0)
    del sets


def _tree(args, dev, entry, steps):
    from speculative_decoding_verification_temperature_gb300 import api
    # tree: B=16, N=64, V=151936 bf16, T=0.8; 4 sets (622 MB each)
    sets = [synth.tree(r, device=dev) for r in range(min(4, max(2, args.sets)))]
    fn = lambda c: api.verify_tree(c.target, c.draft, c.parent,
                                   c.node_tokens, c.uniforms, 0.8)
    ms = _time(fn, sets, steps, 3, dev)
    rows, acc = [], []
    for c in sets:
        o = fn(c)
        rows.append(_rows_tree(c.parent.cpu().numpy(),
                               o["nodes"].cpu().numpy(),
                               o["n"].cpu().numpy(), False))
        acc.append(float(o["n"].float().mean()))
    entry("tree", ms, np.mean(rows), 151936, 2, 16 * 128,
          {"mean_accepted": float(np.mean(acc))})
    _register(args, "tree", "tree", sets[0], fn(sets[0]), 0.8)
    # the same top-k trees under the deterministic-draft rule (greedy
    # acceptance): target rows of the visited nodes only
    fd = lambda c: api.verify_tree_det(c.target, c.parent, c.node_tokens,
                                       c.uniforms, 0.8)
    ms = _time(fd, sets, steps, 3, dev)
    rows, acc = [], []
    for c in sets:
        o = fd(c)
        rows.append(_rows_tree(c.parent.cpu().numpy(),
                               o["nodes"].cpu().numpy(),
                               o["n"].cpu().numpy(), True))
        acc.append(float(o["n"].float().mean()))
    entry("tree_deterministic", ms, np.mean(rows), 151936, 2, 16 * 64,
          {"mean_accepted": float(np.mean(acc))})
    _register(args, "tree_deterministic", "tree_det", sets[0], fd(sets[0]),
              0.8)
    del sets


def _register(args, name, kind, case, out, T, **extra):
    """Keep one input set and its GPU outputs for the oracle comparison of
    the CPU-baseline leg (when that leg runs)."""
    if getattr(args, "checks", None) is None:
        return
    args.checks.append((name, kind, case, {k: v.cpu().numpy()
                                           for k, v in out.items()}, T,
                        extra))


# --------------------------------------------------------- CPU oracle
def _over_threads(fn, n):
    """fn(lo, hi) -> dict of arrays over contiguous chunks of range(n) on
    every host core (the C oracle releases the interpreter lock); the dicts
    are concatenated in order."""
    from concurrent.futures import ThreadPoolExecutor
    nt = max(1, min(n, len(os.sched_getaffinity(0))))
    bounds = [(n * i // nt, n * (i + 1) // nt) for i in range(nt)]
    with ThreadPoolExecutor(max_workers=nt) as pool:
        parts = list(pool.map(lambda b: fn(*b), bounds))
    return {k: np.concatenate([p[k] for p in parts]) for k in parts[0]
            if isinstance(parts[0][k], np.ndarray)}


def flag_summary(o, g, T):
    """Flagged draws of one oracle run and the parity of the GPU outputs g
    (n, tokens) with it: accept tests made and those within 1e-5 of their
    threshold; final inverse-CDF draws within 1e-5 of a CDF boundary and
    those whose token differs from the oracle's (inside its admissible
    range, as the tests require); sequences that differ anywhere else."""
    import oracle
    fm = oracle.FLAG_MARGIN
    on, ot = o["n"], o["tokens"]
    gn, gt = g["n"], g["tokens"][:, :ot.shape[1]]
    valid = on >= 0
    acc_seq = o["margin_acc"] < fm
    cdf = (o["margin_cdf"] < fm) & valid & ~acc_seq
    rows = np.arange(len(on))
    fin = np.maximum(on, 0)
    same_n = (gn == on)
    cols = np.arange(ot.shape[1])[None, :]
    exact = ~((cols == on[:, None]) & cdf[:, None])
    tok_ok = ((gt == ot) | ~exact).all(axis=1)
    g_fin = gt[rows, fin]
    in_range = (g_fin >= o["cdf_lo"]) & (g_fin <= o["cdf_hi"])
    bad = ~acc_seq & ~(same_n & tok_ok & (~cdf | in_range))
    tests = int(o["acc_tests"].sum())
    fl = int(o["acc_flagged"].sum())
    draws = int(valid.sum()) if T > 0 else 0
    return {"sequences": int(len(on)), "mismatches": int(bad.sum()),
            "accept_tests": tests, "accept_flagged": fl,
            "accept_frac": fl / tests if tests else 0.0,
            "cdf_draws": draws, "cdf_flagged": int(cdf.sum()),
            "cdf_frac": int(cdf.sum()) / draws if draws else 0.0,
            "cdf_diff": int((cdf & same_n & (g_fin != ot[rows, fin])).sum()),
            "sequences_set_aside": int(acc_seq.sum())}


def oracle_check(kind, c, g, T, extra):
    """The oracle over every sequence of one input set (host threads) and
    its flag summary against the GPU outputs g."""
    import oracle
    t = synth.host_logits(c.target)
    d = None if (T == 0 and kind in ("linear", "filtered", "kcand_trie")) \
        else synth.host_logits(c.draft)
    u = c.uniforms.cpu().numpy()
    tk = c.tokens.cpu().numpy() if hasattr(c, "tokens") else None
    nseq = t.shape[0]
    if kind == "linear":
        gm = t.shape[1] - 1
        o = _over_threads(lambda a, b: oracle.verify_linear(
            t[a:b], None if d is None else np.ascontiguousarray(
                d[a:b, :gm]), tk[a:b], u[a:b], T), nseq)
    elif kind == "filtered":
        # nucleus cuts: the GPU's kept count of every row must lie in the
        # oracle's admissible range; the rest is compared with those counts
        # forced on the oracle
        gm = t.shape[1] - 1

        def run(forced):
            return _over_threads(lambda a, b: oracle.verify_linear_filtered(
                t[a:b], np.ascontiguousarray(d[a:b, :gm]), tk[a:b], u[a:b],
                T, extra["top_k"], extra["top_p"], want_keep=True,
                keep_forced=None if forced is None else forced[a:b]), nseq)
        o0 = run(None)
        gk = g["keep"]
        both = (gk >= 0) & (o0["keep"] >= 0)
        outside = both & ((gk < o0["keep_lo"]) | (gk > o0["keep_hi"]))
        o = run(np.where(gk >= 1, gk, -1).astype(np.int32))
        res = flag_summary(o, g, T)
        res.update({"rows_cut": int(both.sum()),
                    "cuts_outside_range": int(outside.sum()),
                    "cuts_differing_from_oracle": int(
                        (both & (gk != o0["keep"])).sum())})
        return res
    elif kind == "kcand":
        o = _over_threads(lambda a, b: oracle.verify_kcand(
            t[a:b], d[a:b], tk[a:b], u[a:b], T), nseq)
    elif kind == "kcand_trie":
        o = _over_threads(lambda a, b: oracle.verify_kcand_trie(
            t[a:b], None if d is None else d[a:b], tk[a:b], u[a:b], T),
            nseq)
    elif kind == "tree":
        par, nt = c.parent.cpu().numpy(), c.node_tokens.cpu().numpy()
        o = _over_threads(lambda a, b: oracle.verify_tree(
            t[a:b], d[a:b], par[a:b], nt[a:b], u[a:b], T), nseq)
    else:  # tree_det
        par, nt = c.parent.cpu().numpy(), c.node_tokens.cpu().numpy()
        o = _over_threads(lambda a, b: oracle.verify_tree_det(
            t[a:b], par[a:b], nt[a:b], u[a:b], T), nseq)
    return flag_summary(o, g, T)


def oracle_sample(c, seqs, F):
    import oracle
    t = synth.host_logits(c.target[seqs])
    dall = synth.host_logits(c.draft[seqs])
    d = np.ascontiguousarray(dall[:, :GAMMA])
    tk = c.tokens[seqs].cpu().numpy()
    u = c.uniforms[seqs].cpu().numpy()
    t0 = time.perf_counter()
    oracle.verify_linear(t, d, tk, u, T)
    oracle.fanout_topk(dall, np.array(F, np.int32))
    return time.perf_counter() - t0


def oracle_threads(c, seqs, F, nthreads):
    """The oracle over `seqs` split across host threads (the C oracle runs
    with the interpreter lock released); returns the wall time."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    chunks = [seqs[i::nthreads] for i in range(nthreads) if seqs[i::nthreads]]
    inputs = []
    for ch in chunks:
        dall = synth.host_logits(c.draft[ch])
        inputs.append((synth.host_logits(c.target[ch]),
                       np.ascontiguousarray(dall[:, :GAMMA]), dall,
                       c.tokens[ch].cpu().numpy(), c.uniforms[ch].cpu().numpy()))
    oracle.build()

    def work(x):
        t, d, dall, tk, u = x
        return (oracle.verify_linear(t, d, tk, u, T),
                oracle.fanout_topk(dall, np.array(F, np.int32)))
    with ThreadPoolExecutor(max_workers=len(chunks)) as pool:
        t0 = time.perf_counter()
        res = list(pool.map(work, inputs))
        dt = time.perf_counter() - t0
    # put the chunks' sequences back in order
    order = np.argsort(np.concatenate([np.array(ch) for ch in chunks]))
    cat = lambda i, k: np.concatenate([r[i][k] for r in res])[order]
    ov = {k: cat(0, k) for k in res[0][0] if isinstance(res[0][0][k],
                                                       np.ndarray)}
    of = {k: cat(1, k) for k in ("tokens", "logit")}
    return dt, ov, of


def cpu_baseline(sets, nseq, F, gpu_out=None):
    """The oracle on the host cores: all of them, one thread per core over
    the round's sequences, and (sub-field) one thread on a part of them.
    With the GPU's outputs of the same round (gpu_out: verify n, tokens and
    the fan-out tokens), also their parity with the oracle's and the
    flagged fractions (returned as a second value)."""
    cores = len(os.sched_getaffinity(0))
    n1 = max(1, min(nseq, 32))
    dt1 = oracle_sample(sets[0], list(range(n1)), F)
    seqs = list(range(nseq))
    dtn, ov, of = oracle_threads(sets[0], seqs, F, cores)
    flags = None
    if gpu_out is not None:
        g = {k: v[:nseq] for k, v in gpu_out.items()}
        flags = flag_summary(ov, g, T)
        flags["fanout_rows"] = int(nseq * (FAN["K"] + 1))
        diff, off = 0, 0
        for f in F:  # row k of each sequence: columns off .. off + F_k
            diff += int((g["fan_tokens"][:, off:off + f] !=
                         of["tokens"][:, off:off + f]).any(axis=1).sum())
            off += f
        flags["fanout_rows_differing"] = diff
    base = {"value": nseq / dtn / B, "unit": "rounds/s", "cores": cores,
            "kind": "oracle",
            "sample": "fp64 C oracle (verify + fan-out), %d host threads "
                      "over %d of the %d sequences of one round (%.2f s "
                      "wall), scaled to a full round" % (cores, nseq, B, dtn),
            "single_thread": {"value": n1 / dt1 / B, "cores": 1,
                              "sample": "%d sequences, %.2f s" % (n1, dt1)}}
    return base, flags


def reference_arm(args):
    """The oracle as the reference arm, on the host's cores: each step
    verifies one sequence per core of the workload (cycling through the
    batch), one thread per core; rounds/s is scaled from the sequences per
    second."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    oracle.build()
    c = synth.large(0, device="cuda" if torch.cuda.is_available() else "cpu")
    t_all = synth.host_logits(c.target)
    dfull = synth.host_logits(c.draft)
    d_all = np.ascontiguousarray(dfull[:, :GAMMA])
    tk = c.tokens.cpu().numpy()
    u = c.uniforms.cpu().numpy()
    F = np.array(oracle.fanout_schedule(FAN["K"], FAN["budget"], FAN["a"],
                                        FAN["r"]), np.int32)
    del c

    cores = len(os.sched_getaffinity(0))

    def one(b):
        oracle.verify_linear(t_all[b:b + 1], d_all[b:b + 1], tk[b:b + 1],
                             u[b:b + 1], T)
        oracle.fanout_topk(dfull[b:b + 1], F)

    pool = ThreadPoolExecutor(max_workers=cores)

    def step(i):
        list(pool.map(one, [(i * cores + t) % B for t in range(cores)]))

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    pool.shutdown()
    per_seq = dt / (args.steps * cores)
    value = 1.0 / (per_seq * B)
    sample = ("fp64 C oracle, %d host threads; each step verifies %d of the "
              "%d sequences of a round (one per thread) with their fan-out; "
              "rounds/s = sequences per second / B" % (cores, cores, B))
    return {"metric": METRIC, "value": value, "unit": "rounds/s",
            "impl": "reference", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(), "B": B, "gamma": GAMMA,
                       "V": V, "T": T},
            "cpu_baseline": {"value": value, "unit": "rounds/s",
                             "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "rounds/s",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native",
                    choices=["native", "reference"])
    ap.add_argument("--only", default=None,
                    choices=["tiny", "linear", "kcand", "tree", "filtered",
                             "cache_hit", "presto", "fork"],
                    help="time only this other workload (profiling runs); "
                         "no main line")
    ap.add_argument("--batch", type=int, default=256,
                    help="sequences per step (smaller only to profile a "
                         "small case of the same kernels)")
    ap.add_argument("--sets", type=int, default=3,
                    help="input sets rotated between steps")
    ap.add_argument("--e2e-steps", type=int, default=20,
                    help="steps of the host-buffer leg (0: skip it)")
    ap.add_argument("--aux-steps", type=int, default=30,
                    help="timed rounds of each of the other workloads "
                         "(0: skip them)")
    ap.add_argument("--step", choices=("fused", "streams"), default="fused",
                    help="the large step: one sd_verify_linear_fanout launch "
                         "(default), or the two calls on two streams")
    ap.add_argument("--tune", action="append", default=[],
                    metavar="NAME=VALUE",
                    help="set a library tuning switch (sd_tune_set) before "
                         "timing, e.g. --tune cluster=4 (A/B measurements)")
    ap.add_argument("--oracle-seqs", type=int, default=256,
                    help="sequences of one round the CPU oracle times "
                         "(0: skip the CPU baseline)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    global B
    B = args.batch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args)))
        return
    if args.tune:
        from speculative_decoding_verification_temperature_gb300 import api
        for kv in args.tune:
            k, v = kv.split("=")
            api.tune_set(k, int(v))
    if args.only:  # one other workload alone (for profiler runs)
        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
        torch.cuda.set_device(dev)
        peak, _ = hbm_peak()
        if rank == 0:
            print(json.dumps({"only": args.only,
                              "workloads": other_workloads(args, dev, peak)}))
        return
    if world > 1:
        torch.distributed.init_process_group("nccl")
    res = gpu_arm(args, rank, world)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
