#!/usr/bin/env python
"""Throughput of the fused per-token layer path on one packed batch.

One step = RMSNorm fwd, SwiGLU fwd, QK-RoPE fwd, QK-RoPE bwd, SwiGLU bwd,
RMSNorm bwd (+ its dw reduction) over one batch, inputs resident in HBM.
Reported: achieved HBM GB/s over the algorithmic bytes of the step (every
input read once, every output written once), tokens/s, and the same per
kernel; the roofline of the dominant kernel against the measured HBM copy
bandwidth; an end-to-end figure through the same API with pinned host
buffers copied in and out every step; and the CPU oracle timed on a bounded
sample of the workload (which also re-checks parity in the same run).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle arm

Under torchrun each rank runs its own batch (weak scaling, no collective on
the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s (% of GB300 peak) and tokens/s per fused fwd+bwd kernel"
OPS = ("rmsnorm_fwd", "swiglu_fwd", "qk_rope_fwd", "qk_rope_bwd", "swiglu_bwd", "rmsnorm_bwd")
LAUNCHES_PER_STEP = 7  # rmsnorm_bwd is two kernels (rows + fixed-order dw reduction)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="qwen2.5-0.5b")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-ext", action="store_true", help="skip timing the widened ops")
    p.add_argument("--no-cce", action="store_true", help="skip the LM-head cross-entropy leg")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="CPU work of the oracle baseline sample")
    p.add_argument("--reference-seconds", type=float, default=90.0,
                   help="total CPU time budget of the --impl reference run")
    return p.parse_args(argv)


# ----------------------------------------------------------------- helpers

def rank_info():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def reduce_timing(elapsed_s: float, units: float, group=None):
    """(max elapsed over ranks, sum of units over ranks): whole-job numbers."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_s, units
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 TFLOP/s for a kernel timed on its own (the burst figure)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


_ROPE = ("qk_rope.cu", "rope_common.cuh")
KERNEL_SOURCES = {"rmsnorm_fwd": ("rmsnorm_fwd.cu",),
                  "rmsnorm_bwd": ("rmsnorm_bwd.cu", "rmsnorm_bwd.cuh", "dw_reduce.cuh"),
                  "swiglu_fwd": ("swiglu.cu",), "swiglu_bwd": ("swiglu.cu",),
                  "qk_rope_fwd": _ROPE, "qk_rope_bwd": _ROPE,
                  "rmsnorm_add_fwd": ("rmsnorm_fwd.cu",),
                  "rmsnorm_add_bwd": ("rmsnorm_add_bwd.cu", "rmsnorm_bwd.cuh", "dw_reduce.cuh"),
                  "swiglu_bwd_h": ("swiglu.cu",), "qk_rope_freq_fwd": _ROPE,
                  "qk_norm_rope_fwd": ("qk_norm_rope.cu", "rope_common.cuh", "dw_reduce.cuh"),
                  "qk_norm_rope_bwd": ("qk_norm_rope.cu", "rope_common.cuh", "dw_reduce.cuh")}
# widened ops timed beside the step (not part of it), with their launches
EXT_OPS = {"rmsnorm_add_fwd": 1, "rmsnorm_add_bwd": 2, "swiglu_bwd_h": 1, "qk_rope_freq_fwd": 1,
           "qk_norm_rope_fwd": 1, "qk_norm_rope_bwd": 2}


def kernel_source_hash(op: str) -> str:
    """Hash of the sources an op's kernels are built from (its .cu file and
    the shared device/launch headers)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fine_tuning_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[op] + ("common.cuh", "launch.h")):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash(kernel)
    for line in open(path):
        parts = line.split()
        if len(parts) == 4 and not line.startswith("#") and parts[0] == kernel \
                and parts[1] == workload and parts[3] == src:
            return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str):
        self.uuid = uuid
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def _mine(self):
        uuids = {s[0] for _, s in self.samples}
        if self.uuid in uuids:
            return [(t, s) for t, s in self.samples if s[0] == self.uuid]
        return self.samples if len(uuids) == 1 else []

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        mine = self._mine()
        inside = [s for t, s in mine if t0 <= t <= t1]
        window = inside or [s for t, s in mine if t0 - 0.5 <= t <= t1 + 0.5]
        if not window:
            return None
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for s in window for n, v in zip(names, s[4:8]) if v == "Active"})

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(s[1]) for s in window if num(s[1]) is not None]
        mx = [num(s[2]) for s in window if num(s[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(window), "samples_inside_timed_region": len(inside)}


# --------------------------------------------------------- the device step

class Batch:
    """Every tensor of one step, resident on the device."""

    def __init__(self, wl, device, seed_offset=0):
        import dataclasses

        import torch

        from fine_tuning_gb300 import ftk
        from fine_tuning_gb300 import workloads as W
        if seed_offset:
            wl = dataclasses.replace(wl, seed=wl.seed + 1000 * seed_offset)
        self.wl = wl
        r = W.rmsnorm_inputs(wl, device)
        s = W.swiglu_inputs(wl, device)
        q = W.rope_inputs(wl, device)
        self.cu_host = W.cu_seqlens_from_lengths(W.draw_lengths(wl))
        self.inputs = {**r, **s, **q,
                       "cu": torch.as_tensor(self.cu_host, device=device)}
        dt = wl.torch_dtype
        T, H, I, Ts = wl.T, wl.H, wl.I, wl.T_swiglu
        ws_bytes = ftk.rmsnorm_bwd_workspace_bytes(T, H, dt)
        self.outputs = {
            "y": torch.empty((T, H), dtype=dt, device=device),
            "rstd": torch.empty((T,), dtype=torch.float32, device=device),
            "dx": torch.empty((T, H), dtype=dt, device=device),
            "dw": torch.empty((H,), dtype=torch.float32, device=device),
            "h": torch.empty((Ts, I), dtype=dt, device=device),
            "dg": torch.empty((Ts, I), dtype=dt, device=device),
            "du": torch.empty((Ts, I), dtype=dt, device=device),
        }
        self.ws = torch.empty(((ws_bytes + 15) // 16) * 4, dtype=torch.float32, device=device)

    def ops(self):
        """The step as six callables, in order."""
        from fine_tuning_gb300 import ftk
        i, o, wl = self.inputs, self.outputs, self.wl
        return (
            lambda: ftk.rmsnorm_fwd(i["x"], i["w"], wl.eps, y=o["y"], rstd=o["rstd"]),
            lambda: ftk.swiglu_fwd(i["g"], i["u"], h=o["h"]),
            lambda: ftk.qk_rope_fwd(i["q"], i["k"], i["cu"], wl.theta),
            lambda: ftk.qk_rope_bwd(i["dq"], i["dk"], i["cu"], wl.theta),
            lambda: ftk.swiglu_bwd(i["dh"], i["g"], i["u"], dg=o["dg"], du=o["du"]),
            lambda: ftk.rmsnorm_bwd(i["dy"], i["x"], i["w"], o["rstd"], wl.eps, dx=o["dx"],
                                    dw=o["dw"], workspace=self.ws),
        )

    # tensors a user copies in / out around one step (RoPE is in place, so
    # q, k, dq, dk go both ways)
    IN = ("x", "w", "dy", "g", "u", "dh", "q", "k", "dq", "dk", "cu")
    OUT_FROM_INPUTS = ("q", "k", "dq", "dk")
    OUT = ("y", "rstd", "dx", "dw", "h", "dg", "du")


def sample_tokens(batch, n):
    """CPU copies of the first n tokens of every input (the oracle sample)."""
    i = batch.inputs
    cut = {k: i[k][:n].cpu() for k in ("x", "dy", "g", "u", "dh", "q", "k", "dq", "dk")}
    cut["w"] = i["w"].cpu()
    return cut


def sample_outputs(batch, n):
    o, i = batch.outputs, batch.inputs
    out = {k: o[k][:n].cpu() for k in ("y", "rstd", "dx", "h", "dg", "du")}
    out.update({k: i[k][:n].cpu() for k in ("q", "k", "dq", "dk")})
    return out


def op_ms(op_events, flush_events):
    """An op's device time: the median over repetitions of its graph [L2
    flush, op] minus the same repetition's graph [L2 flush] (CUDA event
    pairs, in ms)."""
    return statistics.median(a.elapsed_time(b) - fa.elapsed_time(fb)
                             for (a, b), (fa, fb) in zip(op_events, flush_events))


def oracle_step(wl, cut, cu_host, n, scales=False, times=None):
    """The whole path in the CPU oracle over the first n tokens; `times`, if
    given, accumulates each op's wall seconds."""
    import numpy as np

    import oracle
    cu = np.asarray(cu_host)
    cu = np.append(cu[cu < n], n)
    res = {}
    clock = [time.perf_counter()]

    def lap(op):
        t = time.perf_counter()
        if times is not None:
            times[op] = times.get(op, 0.0) + t - clock[0]
        clock[0] = t
    res["y"], res["rstd"] = oracle.rmsnorm_fwd(cut["x"][:n], cut["w"], wl.eps)
    lap("rmsnorm_fwd")
    r = oracle.rmsnorm_bwd(cut["dy"][:n], cut["x"][:n], cut["w"], wl.eps, scales=scales)
    res["dx"], res["dw"] = r[0], r[1]
    if scales:
        res["dx_s"] = r[2]
    lap("rmsnorm_bwd")
    res["h"] = oracle.swiglu_fwd(cut["g"][:n], cut["u"][:n])
    lap("swiglu_fwd")
    r = oracle.swiglu_bwd(cut["dh"][:n], cut["g"][:n], cut["u"][:n], scales=scales)
    res["dg"], res["du"] = r[0], r[1]
    if scales:
        res["dg_s"] = r[2]
    lap("swiglu_bwd")
    r = oracle.qk_rope(cut["q"][:n], cut["k"][:n], cu, wl.theta, +1, scales=scales)
    res["q"], res["k"] = r[0], r[1]
    if scales:
        res["q_s"], res["k_s"] = r[2], r[3]
    lap("qk_rope_fwd")
    r = oracle.qk_rope(cut["dq"][:n], cut["dk"][:n], cu, wl.theta, -1, scales=scales)
    res["dq"], res["dk"] = r[0], r[1]
    if scales:
        res["dq_s"], res["dk_s"] = r[2], r[3]
    lap("qk_rope_bwd")
    return res


def cpu_model() -> str:
    """The host CPU's model name as lscpu reports it."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


def f64_inputs(cut):
    import torch
    return {k: v.to(torch.float64).numpy() for k, v in cut.items()}


def calibrate_tokens(wl, cut64, cu_host, seconds, cap):
    """Tokens of oracle work that take about `seconds` on this host."""
    n0 = min(cap, 64)
    t = time.perf_counter()
    oracle_step(wl, cut64, cu_host, n0)
    per_tok = max((time.perf_counter() - t) / n0, 1e-7)
    return max(1, min(cap, int(seconds / per_tok)))


def cpu_leg(wl, batch, gpu_out, cut, seconds):
    """Oracle on the host cores over a bounded sample; also the parity gate."""
    import oracle
    from fine_tuning_gb300 import workloads as W
    from oracle.tolerance import assert_close
    cap = cut["x"].shape[0]
    cut64 = f64_inputs(cut)
    n = calibrate_tokens(wl, cut64, batch.cu_host, seconds, cap)
    # repeat the sample until about `seconds` of oracle work has run (the
    # sample is capped at the tokens copied to the host)
    passes = 0
    per_op = {}
    t = time.perf_counter()
    while True:
        res = oracle_step(wl, cut64, batch.cu_host, n, times=per_op)
        passes += 1
        el = time.perf_counter() - t
        if el >= seconds or passes >= 100000:
            break
    ib = W.ideal_bytes(wl)

    def tok_bytes(k, ntok):
        return ib[k] * ntok / (wl.T_swiglu if "swiglu" in k else wl.T)
    sample_bytes = passes * sum(tok_bytes(k, n) for k in ib)
    # one pass on a single thread, over about a thread's share of the sample
    cores = oracle.threads()
    n1 = max(1, n // max(cores, 1))
    prev = oracle.set_threads(1)
    t1 = time.perf_counter()
    oracle_step(wl, cut64, batch.cu_host, n1)
    el1 = time.perf_counter() - t1
    oracle.set_threads(prev)
    # parity of the GPU step on the same tokens (the CPU sample is a prefix)
    code = "f32" if wl.dtype == "f32" else "bf16"
    m = min(n, 256)
    ref = oracle_step(wl, cut64, batch.cu_host, m, scales=True)
    worst = 0.0
    worst = max(worst, assert_close("y", gpu_out["y"][:m], ref["y"], dtype=code))
    worst = max(worst, assert_close("rstd", gpu_out["rstd"][:m], ref["rstd"], dtype="f32"))
    worst = max(worst, assert_close("dx", gpu_out["dx"][:m], ref["dx"], ref["dx_s"], dtype=code))
    worst = max(worst, assert_close("h", gpu_out["h"][:m], ref["h"], dtype=code))
    worst = max(worst, assert_close("dg", gpu_out["dg"][:m], ref["dg"], ref["dg_s"], dtype=code))
    worst = max(worst, assert_close("du", gpu_out["du"][:m], ref["du"], dtype=code))
    for k in ("q", "k", "dq", "dk"):
        worst = max(worst, assert_close(k, gpu_out[k][:m], ref[k], ref[k + "_s"], dtype=code))
    del res
    return {
        "value": sample_bytes / el / 1e9, "unit": "GB/s", "cores": cores,
        "kind": "oracle", "tokens_per_s": passes * n / el, "seconds": round(el, 3),
        "sample": f"{passes} passes over the first {n} of {wl.T} tokens ({el:.1f} s), all six "
                  f"ops (oracle in double, OpenMP over rows), GB/s over the passes' "
                  f"algorithmic bytes",
        "per_op_s": {k: round(v / passes, 6) for k, v in per_op.items()},
        "one_thread": {"tokens": n1, "seconds": round(el1, 4),
                       "GB_s": round(sum(tok_bytes(k, n1) for k in ib) / el1 / 1e9, 3)},
        "nproc": os.cpu_count(), "cpu_model": cpu_model(),
    }, {"tokens_checked": m, "ops": 10, "max_err_over_bound": round(worst, 4)}


# -------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    import torch.distributed as dist

    from fine_tuning_gb300 import build, ftk
    from fine_tuning_gb300 import workloads as W

    rank, local_rank, world = rank_info()
    torch.cuda.set_device(local_rank)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank)
    build.build()
    ftk.library()
    wl = W.WORKLOADS[args.workload]
    batch = Batch(wl, dev, seed_offset=rank)
    ops = batch.ops()
    ib = W.ideal_bytes(wl)
    step_bytes = sum(ib[k] for k in OPS)

    do_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    cut = sample_tokens(batch, min(wl.T, 8192)) if do_cpu else None
    for op in ops:  # the parity step, on the untouched inputs
        op()
    torch.cuda.synchronize(dev)
    gpu_out = sample_outputs(batch, min(wl.T, 256)) if do_cpu else None

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(max(args.warmup, 0)):
        flush.fill_(1)
        for op in ops:
            op()
    torch.cuda.synchronize(dev)

    # The step as one CUDA graph (its 7 launches replayed without host
    # overhead, as a training loop would run it).
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for op in ops:
            op()
    # per kernel: a graph [L2 flush, op] and a graph [L2 flush]; the op's
    # time is the difference of their replay times, so the graph launch
    # latency cancels while the flush-to-op gap of a real stream stays in
    op_graphs = []
    for op in ops:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            flush.fill_(3)
            op()
        op_graphs.append(g)
    flush_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(flush_graph):
        flush.fill_(3)
    graph.replay()
    for g in op_graphs + [flush_graph]:
        g.replay()
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    Kk = max(1, min(K, 300))
    evk = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(len(ops) + 1)] for _ in range(Kk)]
    whole0, whole1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = ""
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    sampler = ClockSampler(uuid).start()
    time.sleep(0.6)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    whole0.record()
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record()
        graph.replay()
        ev[i][1].record()
    whole1.record()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    t1 = time.time()
    for i in range(Kk):
        for (a, b), g in zip(evk[i], op_graphs + [flush_graph]):
            a.record()
            g.replay()
            b.record()
    torch.cuda.synchronize(dev)
    time.sleep(0.3)
    sampler.stop()

    step_ms = sum(a.elapsed_time(b) for a, b in ev) / K
    per_op = [op_ms([e[j] for e in evk], [e[-1] for e in evk]) for j in range(len(ops))]
    wall_ms = whole0.elapsed_time(whole1)

    el_max, bytes_all = reduce_timing(step_ms * K / 1e3, step_bytes * K)
    _, tok_all = reduce_timing(0.0, float(wl.T) * K)
    value = bytes_all / el_max / 1e9
    hbm, src = peaks()
    kernels = {}
    for j, name in enumerate(OPS):
        gbs = ib[name] / (per_op[j] * 1e-3) / 1e9
        toks = W.tokens_per_call(wl)[name]
        kernels[name] = {"us": round(per_op[j] * 1e3, 2), "GB_s": round(gbs, 1),
                         "frac_of_measured_hbm" if src == "measured" else "frac_of_fallback_hbm":
                             round(gbs / hbm, 4),
                         "tokens_per_s": round(toks / (per_op[j] * 1e-3), 1),
                         "ideal_bytes": ib[name]}
    dom = max(range(len(ops)), key=lambda j: per_op[j])
    dname = OPS[dom]
    achieved = ib[dname] / (per_op[dom] * 1e-3) / 1e9
    traffic = ncu_traffic(dname, wl.name)

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(el_max * 1e3 / K, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded packed batch; no dataset, no weights)",
        "config": {"workload": wl.name, "T": wl.T, "B": int(len(batch.cu_host) - 1),
                   "H": wl.H, "I": wl.I, "T_swiglu": wl.T_swiglu, "Hq": wl.Hq, "Hkv": wl.Hkv,
                   "D": wl.D, "theta": wl.theta, "eps": wl.eps,
                   "parallelism": f"replicas x{world} (one batch per GPU, no collective)",
                   "l2": "flushed before every step (256 MiB write, outside the step events)",
                   "step": list(OPS)},
        "tokens_per_s": round(tok_all / el_max, 1),
        "frac_of_hbm": round(value / hbm, 4), "hbm_peak_GB_s": hbm, "hbm_peak_source": src,
        "kernels": kernels,
        "roofline": {"kernel": dname, "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "traffic": traffic, "algorithmic_bytes": ib[dname],
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured"
                     else "fallback 6.8 TB/s"},
        # this library's launches inside the timed region (the K steps), and
        # over every leg of the run
        "gpu_launches": LAUNCHES_PER_STEP * K,
        "gpu_launches_all_legs": LAUNCHES_PER_STEP * (K + Kk),
        "timing": (f"step: {K} replays of a CUDA graph of the step's {LAUNCHES_PER_STEP} "
                   f"launches, CUDA events around each replay; per kernel: the median over {Kk} "
                   "replays of a graph [L2 flush, op] minus the same repetition's graph [L2 flush], "
                   "CUDA events around each"),
        "wall_ms_timed_region": round(wall_ms, 3),
    }
    if not args.no_ext:
        out["extensions"] = ext_leg(batch, flush, flush_graph, dev, Kk, hbm, src)
        if rank == 0 and not args.no_cce:
            out["cce"] = cce_leg(dev, flush, flush_graph, max(3, min(Kk, 20)))
            out["gpu_launches_all_legs"] += out["cce"].pop("launches")
        out["gpu_launches_all_legs"] += sum(EXT_OPS.values()) * Kk
    out["clocks"] = sampler.summary(t0, t1)
    out["device_status"] = ftk.device_status(clear=True)  # 0: no pipeline wait ran out

    if not args.no_e2e:
        out["e2e"] = e2e_leg(batch, ops, dev, args.e2e_steps, step_bytes)
    if do_cpu:
        out["cpu_baseline"], out["parity"] = cpu_leg(wl, batch, gpu_out, cut, args.cpu_seconds)
        out["packing"] = packing_leg(wl)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def ext_leg(batch, flush, flush_graph, dev, reps, hbm, src):
    """The widened ops (not part of the step), each timed like a step kernel:
    replays of a graph [L2 flush, op] minus the graph [L2 flush].  They run
    after the timed step region, on the same batch (the residual stream and
    its gradient drawn beside it)."""
    import torch

    from fine_tuning_gb300 import ftk
    from fine_tuning_gb300 import workloads as W
    wl, i, o = batch.wl, batch.inputs, batch.outputs
    extra = W.rmsnorm_add_inputs(wl, dev)
    res, dres = extra["res"], extra["dh"]
    T, H, dt = wl.T, wl.H, wl.torch_dtype
    h = torch.empty((T, H), dtype=dt, device=dev)
    y = torch.empty((T, H), dtype=dt, device=dev)
    rstd = torch.empty((T,), dtype=torch.float32, device=dev)
    dx = torch.empty((T, H), dtype=dt, device=dev)
    dw = torch.empty((H,), dtype=torch.float32, device=dev)
    llama3 = ftk.rope_llama3_inv_freq(wl.D, wl.theta, 32.0, 1.0, 4.0, 8192.0)
    nr = W.qk_norm_rope_inputs(wl, dev, T=1)  # only the weights wq, wk are used
    wq, wk = nr["wq"], nr["wk"]
    qo, ko = torch.empty_like(i["q"]), torch.empty_like(i["k"])
    rq = torch.empty((T, wl.Hq), dtype=torch.float32, device=dev)
    rk = torch.empty((T, wl.Hkv), dtype=torch.float32, device=dev)
    nr_bytes = max(16, ftk.qk_norm_rope_bwd_workspace_bytes(T, wl.D, dt))
    nr_ws = torch.empty((nr_bytes + 3) // 4, dtype=torch.float32, device=dev)
    ops = {
        "rmsnorm_add_fwd": lambda: ftk.rmsnorm_add_fwd(i["x"], res, i["w"], wl.eps, h=h, y=y,
                                                       rstd=rstd),
        "rmsnorm_add_bwd": lambda: ftk.rmsnorm_add_bwd(i["dy"], dres, h, i["w"], rstd, wl.eps,
                                                       dx=dx, dw=dw, workspace=batch.ws),
        "swiglu_bwd_h": lambda: ftk.swiglu_bwd_h(i["dh"], i["g"], i["u"], dg=o["dg"],
                                                 du=o["du"], h=o["h"]),
        # the Llama-3.2 rope_scaling table (factor 32, low 1, high 4, 8192)
        "qk_rope_freq_fwd": lambda: ftk.qk_rope_freq_fwd(i["q"], i["k"], i["cu"], llama3),
        "qk_norm_rope_fwd": lambda: ftk.qk_norm_rope_fwd(i["q"], i["k"], wq, wk, i["cu"], wl.eps,
                                                         theta=wl.theta, q_out=qo, k_out=ko,
                                                         rstd_q=rq, rstd_k=rk),
        "qk_norm_rope_bwd": lambda: ftk.qk_norm_rope_bwd(
            i["dq"], i["dk"], i["q"], i["k"], wq, wk, rq, rk, i["cu"], wl.eps, theta=wl.theta,
            dq=qo, dk=ko, workspace=nr_ws),
    }
    assert set(ops) == set(EXT_OPS)
    for op in ops.values():  # warm-up (and the first, allocating, launch)
        op()
    graphs = {}
    for name, op in ops.items():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            flush.fill_(5)
            op()
        graphs[name] = g
    for g in list(graphs.values()) * 3:
        g.replay()
    torch.cuda.synchronize(dev)
    ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)] for n in list(graphs) + ["flush"]}
    for k in range(reps):
        for n, g in list(graphs.items()) + [("flush", flush_graph)]:
            a, b = ev[n][k]
            a.record()
            g.replay()
            b.record()
    torch.cuda.synchronize(dev)
    ib, toks = W.ideal_bytes(wl), W.tokens_per_call(wl)
    out = {}
    for n in graphs:
        ms = op_ms(ev[n], ev["flush"])
        gbs = ib[n] / (ms * 1e-3) / 1e9
        out[n] = {"us": round(ms * 1e3, 2), "GB_s": round(gbs, 1),
                  "frac_of_measured_hbm" if src == "measured" else "frac_of_fallback_hbm":
                      round(gbs / hbm, 4),
                  "tokens_per_s": round(toks[n] / (ms * 1e-3), 1), "ideal_bytes": ib[n],
                  "launches": EXT_OPS[n]}
    out["timing"] = (f"the median over {reps} replays of a graph [L2 flush, op] minus the same "
                     "repetition's graph [L2 flush], CUDA events around each; outside the step's "
                     "timed region")
    del h, y, rstd, dx, dw, res, dres, extra, qo, ko, rq, rk, nr_ws
    return out


def cce_leg(dev, flush, flush_graph, reps):
    """The LM-head cross-entropy (a second workload, tensor-core bound):
    Qwen2.5-0.5B's head on 8,192 tokens, forward and backward each captured
    as a graph [L2 flush, op] and timed against the graph [L2 flush]."""
    import torch

    from fine_tuning_gb300 import ftk
    from fine_tuning_gb300 import workloads as W
    hw = W.HEAD_WORKLOADS["qwen2.5-0.5b-head"]
    d = W.head_inputs(hw, dev)
    h, Wt, y = d["h"], d["W"], d["y"]
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(hw.T, dtype=torch.float32, device=dev)
    g = torch.ones(1, dtype=torch.float32, device=dev)
    dh = torch.empty_like(h)
    dW = torch.empty((hw.V, hw.H), dtype=torch.float32, device=dev)
    wsf = torch.empty(int(ftk.library().ftk_cce_fwd_workspace_bytes(hw.T, hw.V)),
                      dtype=torch.uint8, device=dev)
    wsb = torch.empty(int(ftk.library().ftk_cce_bwd_workspace_bytes(hw.T, hw.H, hw.V)),
                      dtype=torch.uint8, device=dev)
    ops = {"cce_fwd": lambda: ftk.cce_fwd(h, Wt, y, loss=loss, lse=lse, workspace=wsf),
           "cce_bwd": lambda: ftk.cce_bwd(h, Wt, y, lse, g, dh=dh, dW=dW, workspace=wsb)}
    for op in ops.values():
        op()
    graphs = {}
    for name, op in ops.items():
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            flush.fill_(9)
            op()
        graphs[name] = gr
    for gr in graphs.values():
        gr.replay()
    torch.cuda.synchronize(dev)
    ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)] for n in list(graphs) + ["flush"]}
    for k in range(reps):
        for n, gr in list(graphs.items()) + [("flush", flush_graph)]:
            a, b = ev[n][k]
            a.record()
            gr.replay()
            b.record()
    torch.cuda.synchronize(dev)
    peak, psrc = tensor_peak()
    flops = {"cce_fwd": 2 * hw.T * hw.H * hw.V, "cce_bwd": 6 * hw.T * hw.H * hw.V}
    chunk = ftk.cce_bwd_chunk(hw.T, hw.H, hw.V)
    nchunk = -(-hw.V // chunk)
    launches = {"cce_fwd": 3, "cce_bwd": 1 + 2 * nchunk}
    out = {"workload": {"name": hw.name, "T": hw.T, "H": hw.H, "V": hw.V,
                        "ignored_share": hw.ignored, "bwd_chunk": chunk},
           "loss": round(float(loss.item()), 6)}
    for n in graphs:
        ms = op_ms(ev[n], ev["flush"])
        tf = flops[n] / (ms * 1e-3) / 1e12
        out[n] = {"ms": round(ms, 4), "TFLOP_s": round(tf, 1), "algorithmic_flops": flops[n],
                  "tokens_per_s": round(hw.T / (ms * 1e-3), 1),
                  "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak,
                               "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                               "peak_source": f"{psrc} bf16 dense (burst)"}}
    out["launches"] = (launches["cce_fwd"] + launches["cce_bwd"]) * reps
    out["timing"] = (f"the median over {reps} replays of a graph [L2 flush, op] minus the same "
                     "repetition's graph [L2 flush], CUDA events around each; outside the step's "
                     "timed region")
    return out


def e2e_leg(batch, ops, dev, steps, step_bytes):
    """The step through the public API with host buffers: every step copies
    all of its inputs in from pinned host memory and all of its outputs
    back.  As a user would run consecutive steps, three streams overlap
    step k+1's copy-in, step k's kernels and step k-1's copy-out, with two
    device-side buffer sets; events order every reuse of a buffer."""
    import torch
    wl = batch.wl
    sets = [batch, Batch(wl, dev)]
    set_ops = [ops, sets[1].ops()]
    host_in = {k: batch.inputs[k].cpu().pin_memory() for k in Batch.IN}

    def outs(b):
        return {**b.outputs, **{k: b.inputs[k] for k in Batch.OUT_FROM_INPUTS}}
    host_out = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in outs(batch).items()}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    s_in, s_run, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event(enable_timing=False)

    def run(n, t0=None):
        done_run = [None, None]   # last compute on each set
        done_out = [None, None]   # last copy-out of each set
        last = None
        for i in range(n):
            j = i & 1
            b = sets[j]
            with torch.cuda.stream(s_in):
                if done_run[j] is not None:
                    s_in.wait_event(done_run[j])   # inputs of set j no longer read
                if i == 0 and t0 is not None:
                    t0.record(s_in)
                for k, v in host_in.items():
                    b.inputs[k].copy_(v, non_blocking=True)
                e_in = ev()
                e_in.record(s_in)
            with torch.cuda.stream(s_run):
                s_run.wait_event(e_in)
                if done_out[j] is not None:
                    s_run.wait_event(done_out[j])  # outputs of set j already copied out
                for op in set_ops[j]:
                    op()
                done_run[j] = ev()
                done_run[j].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_run[j])
                for k, v in outs(b).items():
                    host_out[k].copy_(v, non_blocking=True)
                done_out[j] = ev()
                done_out[j].record(s_out)
                last = s_out
        return last

    run(2)
    torch.cuda.synchronize(dev)
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    last = run(steps, t0=a)
    z.record(last)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(z) / steps
    del sets[1]
    el_max, bytes_all = reduce_timing(ms * steps / 1e3, step_bytes * steps)
    return {"value": round(bytes_all / el_max / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(el_max * 1e3 / steps, 3), "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "3 streams: copy-in of step k+1, kernels of step k, copy-out of step k-1"}


# ------------------------------------------------------ packing (host)

def packing_leg(wl, n_seq=200_000, batch=8):
    """Best-Fit-Decreasing packing of a corpus with the workload's length mix
    into bins of T tokens: host throughput of the library routine and of the
    oracle (bounded sample), and how much of the padding waste of plain
    padded batching (batches of `batch` sequences padded to their longest)
    the packing recovers."""
    import numpy as np

    from fine_tuning_gb300 import ftk
    from fine_tuning_gb300 import workloads as W
    from oracle.packing import bfd_pack as oracle_bfd
    reps = []
    total = 0
    i = 0
    while total < n_seq:
        lens = W.draw_lengths(__import__("dataclasses").replace(wl, seed=wl.seed + 7919 * i))
        reps.append(lens)
        total += lens.size
        i += 1
    lens = np.concatenate(reps)[:n_seq].astype(np.int32)
    t = time.perf_counter()
    bin_of, order, bin_start = ftk.bfd_pack(lens, wl.T)
    el = time.perf_counter() - t
    bins = len(bin_start) - 1
    real = int(lens.sum())
    m = 20_000
    t = time.perf_counter()
    oracle_bfd(lens[:m].tolist(), wl.T)
    el_o = time.perf_counter() - t
    nb = (lens.size + batch - 1) // batch
    padded = sum(int(lens[b * batch:(b + 1) * batch].max()) * min(batch, lens.size - b * batch)
                 for b in range(nb))
    waste_pad = padded - real
    waste_pack = bins * wl.T - real
    return {"sequences": int(lens.size), "capacity_tokens": wl.T, "bins": bins,
            "sequences_per_s": round(lens.size / el, 1),
            "oracle_sequences_per_s": round(m / el_o, 1), "oracle_sample": m,
            "fill": round(real / (bins * wl.T), 4),
            "padding_waste_recovered": round(1 - waste_pack / waste_pad, 4),
            "vs": f"batches of {batch} padded to their longest sequence"}


# -------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle as the reference arm, on rank 0 only."""
    rank, _, world = rank_info()
    if rank != 0:
        return
    import oracle
    from fine_tuning_gb300 import workloads as W
    from oracle.build import build_oracle
    build_oracle()
    wl = W.WORKLOADS[args.workload]
    lens = W.draw_lengths(wl)
    cu = W.cu_seqlens_from_lengths(lens)
    cap = min(wl.T, 4096)
    cut = {}
    for k, v in (("x", W.rmsnorm_inputs(wl, "cpu", T=cap)), ("g", W.swiglu_inputs(wl, "cpu", T=cap)),
                 ("q", W.rope_inputs(wl, "cpu", T=cap))):
        cut.update(v)
    cut64 = f64_inputs(cut)
    per_step_s = args.reference_seconds / max(1, args.steps + args.warmup)
    n = calibrate_tokens(wl, cut64, cu, per_step_s, cap)
    for _ in range(args.warmup):
        oracle_step(wl, cut64, cu, n)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(wl, cut64, cu, n)
    el = time.perf_counter() - t
    ib = W.ideal_bytes(wl)
    sample_bytes = sum(v * (n / (wl.T_swiglu if "swiglu" in k else wl.T)) for k, v in ib.items())
    value = sample_bytes * args.steps / el / 1e9
    sample = (f"first {n} of {wl.T} tokens per step, all six ops, oracle in double "
              f"(OpenMP over rows) on the host cores")
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded packed batch; no dataset, no weights)",
        "config": {"workload": wl.name, "T": wl.T, "tokens_per_step": n},
        "tokens_per_s": round(n * args.steps / el, 1),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(out), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
