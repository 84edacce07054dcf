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

The default workload is the largest single-GPU one: Qwen3-32B layer shapes
on one 524,288-token sequence.  The smaller workloads are timed in the same
run, with the same per-kernel method, in a compact `per_workload` block.
`--tokens N` cuts a workload to its first N tokens (a slice with the same
row shapes, for profiler captures that must stay small).

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
NOMINAL_HBM_GBS = 8000.0  # GB300's HBM3e spec figure (a second column beside the measured copy)
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="qwen3-32b-524k")
    p.add_argument("--tokens", type=int, default=0,
                   help="cut the workload to its first N tokens (0: the whole batch)")
    p.add_argument("--per-workload", default="qwen2.5-0.5b,llama-3.2-1b,qwen3-8b",
                   help="comma-separated workloads also timed per kernel ('none': skip)")
    p.add_argument("--kernel-reps", type=int, default=0,
                   help="repetitions of each one-op graph (0: min(steps, 300))")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-ext", action="store_true", help="skip timing the widened ops")
    p.add_argument("--no-cce", action="store_true", help="skip the LM-head cross-entropy leg")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="CPU work of the oracle baseline sample")
    p.add_argument("--reference-seconds", type=float, default=90.0,
                   help="total CPU time budget of the --impl reference run")
    p.add_argument("--records", default="",
                   help="also write one JSON record per (workload, op) to this .jsonl file")
    return p.parse_args(argv)


def records_from(out):
    """One flat record per (workload, op) of a bench line: the shapes, the
    op's algorithmic bytes and the ncu DRAM traffic on file, its time, GB/s,
    fractions of the measured copy rate and of 8 TB/s, tokens/s, and the
    run's parity figures and clocks."""
    cfg = out.get("config", {})
    shapes = {k: cfg[k] for k in ("T", "H", "I", "T_swiglu", "Hq", "Hkv", "D") if k in cfg}
    legs = [(cfg.get("workload"), shapes, out.get("kernels", {}), out.get("extensions", {}),
             out.get("parity"))]
    for name, w in out.get("per_workload", {}).items():
        legs.append((name, {k: w[k] for k in ("T", "H", "I", "Hq", "Hkv", "D") if k in w},
                     w.get("kernels", {}), w.get("extensions", {}), w.get("parity")))
    recs = []
    for name, shp, kern, ext, par in legs:
        for op, k in list(kern.items()) + [(o, v) for o, v in ext.items() if isinstance(v, dict)
                                           and "us" in v]:
            op_base = op.replace("_fwd", "").replace("_bwd", "")
            rec = {"workload": name, "op": op_base,
                   "dir": "bwd" if "bwd" in op else "fwd", "kernel": op, "shapes": shp,
                   "ideal_bytes": k.get("ideal_bytes"),
                   "ncu_dram_bytes": ncu_traffic(op, name) if name else None,
                   "us": k["us"], "GB_s": k.get("GB_s"),
                   "frac_of_hbm": k.get("frac_of_measured_hbm", k.get("frac_of_fallback_hbm")),
                   "frac_of_nominal_8tbs": k.get("frac_of_nominal_8tbs"),
                   "tokens_per_s": k.get("tokens_per_s")}
            if par:
                rec["parity_max_err_over_bound"] = par.get("max_err_over_bound")
                lit = par.get("literal", {})
                outs = {o: lit[o] for o in OUTPUTS_OF.get(op, ()) if o in lit}
                if outs:
                    rec["parity_literal"] = outs  # max rel / ulp error and ulp histogram
            cpu = out.get("cpu_baseline")
            if cpu and name == cfg.get("workload") and op in cpu.get("per_op_s", {}):
                rec["oracle_s_per_pass"] = cpu["per_op_s"][op]
                rec["oracle_sample"] = cpu.get("sample")
                rec["oracle_cores"] = cpu.get("cores")
            recs.append(rec)
    return recs


# the outputs of each step op in the parity block
OUTPUTS_OF = {"rmsnorm_fwd": ("y", "rstd"), "rmsnorm_bwd": ("dx",), "swiglu_fwd": ("h",),
              "swiglu_bwd": ("dg", "du"), "qk_rope_fwd": ("q", "k"), "qk_rope_bwd": ("dq", "dk")}


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


_ROPE = ("qk_rope.cu", "rope_common.cuh", "pair_math.cuh")
KERNEL_SOURCES = {"rmsnorm_fwd": ("rmsnorm_fwd.cu", "pair_math.cuh"),
                  "rmsnorm_bwd": ("rmsnorm_bwd.cu", "rmsnorm_bwd.cuh", "dw_reduce.cuh",
                                  "pair_math.cuh"),
                  "swiglu_fwd": ("swiglu.cu",), "swiglu_bwd": ("swiglu.cu",),
                  "qk_rope_fwd": _ROPE, "qk_rope_bwd": _ROPE,
                  "rmsnorm_add_fwd": ("rmsnorm_fwd.cu", "pair_math.cuh"),
                  "rmsnorm_add_bwd": ("rmsnorm_add_bwd.cu", "rmsnorm_bwd.cuh", "dw_reduce.cuh",
                                      "pair_math.cuh"),
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
    """nvidia-smi samples (100 ms) of SM clock and throttle reasons."""

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
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
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


def select_workload(name: str, tokens: int = 0):
    """The named workload, or (tokens > 0) a slice of it: its first `tokens`
    tokens with the same row shapes (sequences cut at the slice's end)."""
    import dataclasses

    from fine_tuning_gb300 import workloads as W
    wl = W.WORKLOADS[name]
    if not tokens or tokens >= wl.T:
        return wl
    cut, total = [], 0
    for n in W.draw_lengths(wl).tolist():
        take = min(int(n), tokens - total)
        if take <= 0:
            break
        cut.append(take)
        total += take
    return dataclasses.replace(wl, name=f"{wl.name}[:{tokens}]", T=tokens,
                               T_swiglu=min(wl.T_swiglu, tokens), lengths=tuple(cut))


def parity_rows(wl, cu_host, n_edge=64, n_mid=64, n_bounds=16, seed=99):
    """Token rows whose outputs the oracle recomputes in the bench run: the
    first and last n_edge tokens, n_mid drawn in between, and the tokens on
    both sides of the first n_bounds sequence boundaries; the same rule over
    the SwiGLU tokens.  Spans the whole batch at any size."""
    import numpy as np

    def pick(T, extra=()):
        if T <= 2 * n_edge + n_mid:
            return np.arange(T)
        rng = np.random.default_rng(seed)
        mid = rng.choice(np.arange(n_edge, T - n_edge), n_mid, replace=False)
        rows = np.concatenate([np.arange(n_edge), mid, np.arange(T - n_edge, T),
                               np.asarray(list(extra), dtype=np.int64)])
        return np.unique(rows[(rows >= 0) & (rows < T)])
    starts = [int(c) for c in cu_host[1:-1][:n_bounds]]
    return pick(wl.T, starts + [c - 1 for c in starts]), pick(wl.T_swiglu)


def gather_inputs(batch, rows, srows):
    """CPU copies of the inputs at the parity rows (taken before the in-place
    RoPE runs)."""
    import torch
    i = batch.inputs
    dev = i["x"].device
    ri, si = torch.as_tensor(rows, device=dev), torch.as_tensor(srows, device=dev)
    out = {k: i[k][ri].cpu() for k in ("x", "dy", "q", "k", "dq", "dk")}
    out.update({k: i[k][si].cpu() for k in ("g", "u", "dh")})
    out["w"] = i["w"].cpu()
    return out


def gather_outputs(batch, rows, srows):
    import torch
    o, i = batch.outputs, batch.inputs
    dev = i["x"].device
    ri, si = torch.as_tensor(rows, device=dev), torch.as_tensor(srows, device=dev)
    out = {k: o[k][ri].cpu() for k in ("y", "rstd", "dx")}
    out.update({k: o[k][si].cpu() for k in ("h", "dg", "du")})
    out.update({k: i[k][ri].cpu() for k in ("q", "k", "dq", "dk")})
    return out


def check_parity(wl, cu_host, rows, srows, inp, got):
    """The oracle on the parity rows against the GPU step's outputs there;
    raises on any element out of tolerance, else returns the worst
    error / bound."""
    import oracle
    from oracle.tolerance import assert_close, literal_figures
    code = "f32" if wl.dtype == "f32" else "bf16"
    yr, rr = oracle.rmsnorm_fwd(inp["x"], inp["w"], wl.eps)
    dxr, _, dxs, _ = oracle.rmsnorm_bwd(inp["dy"], inp["x"], inp["w"], wl.eps, scales=True)
    hr = oracle.swiglu_fwd(inp["g"], inp["u"])
    dgr, dur, dgs = oracle.swiglu_bwd(inp["dh"], inp["g"], inp["u"], scales=True)
    qr, kr, qs, ks = oracle.qk_rope(inp["q"], inp["k"], cu_host, wl.theta, +1, tok=rows,
                                    scales=True)
    dqr, dkr, dqs, dks = oracle.qk_rope(inp["dq"], inp["dk"], cu_host, wl.theta, -1, tok=rows,
                                        scales=True)
    worst, literal = 0.0, {}
    for name, ref, sc, kind in (("y", yr, None, code), ("rstd", rr, None, "f32"),
                                ("dx", dxr, dxs, code), ("h", hr, None, code),
                                ("dg", dgr, dgs, code), ("du", dur, None, code),
                                ("q", qr, qs, code), ("k", kr, ks, code),
                                ("dq", dqr, dqs, code), ("dk", dkr, dks, code)):
        worst = max(worst, assert_close(name, got[name], ref, sc, dtype=kind))
        lit = literal_figures(got[name], ref, dtype=kind)
        literal[name] = {k: (round(v, 9) if isinstance(v, float) else v) for k, v in lit.items()}
    return {"tokens_checked": int(len(rows)), "swiglu_tokens_checked": int(len(srows)),
            "outputs": 10, "max_err_over_bound": round(worst, 4),
            "literal": literal,
            "literal_note": "error against the literal bars alone (relative 1e-5 in fp32, 2 bf16 "
                            "ulps); needed_floor counts the elements that passed only through "
                            "the condition-scale term",
            "rows": "first and last 64 tokens, 64 drawn in between, both sides of the first "
                    "16 sequence boundaries (dw, a sum over every row, is checked in full by "
                    "the GPU tests)"}


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


def head_tokens(batch, n):
    """CPU copies of the first n tokens of every input (the oracle's timing
    sample)."""
    i = batch.inputs
    cut = {k: i[k][:n].cpu() for k in ("x", "dy", "g", "u", "dh", "q", "k", "dq", "dk")}
    cut["w"] = i["w"].cpu()
    return cut


def cpu_leg(wl, cu_host, cut, seconds):
    """The oracle as it stands on the host cores over a bounded sample of the
    workload: repeated passes over its first tokens for about `seconds`."""
    import oracle
    from fine_tuning_gb300 import workloads as W
    cap = cut["x"].shape[0]
    cut64 = f64_inputs(cut)
    n = calibrate_tokens(wl, cut64, cu_host, seconds, cap)
    passes = 0
    per_op = {}
    t = time.perf_counter()
    while True:
        oracle_step(wl, cut64, cu_host, n, times=per_op)
        passes += 1
        el = time.perf_counter() - t
        if el >= seconds or passes >= 100000:
            break
    ib = W.ideal_bytes(wl)

    def tok_bytes(k, ntok):
        return ib[k] * ntok / (wl.T_swiglu if "swiglu" in k else wl.T)
    sample_bytes = passes * sum(tok_bytes(k, n) for k in ib if k in OPS)
    # one pass on a single thread, over about a thread's share of the sample
    cores = oracle.threads()
    n1 = max(1, n // max(cores, 1))
    prev = oracle.set_threads(1)
    t1 = time.perf_counter()
    oracle_step(wl, cut64, cu_host, n1)
    el1 = time.perf_counter() - t1
    oracle.set_threads(prev)
    return {
        "value": sample_bytes / el / 1e9, "unit": "GB/s", "cores": cores,
        "kind": "oracle", "tokens_per_s": passes * n / el, "seconds": round(el, 3),
        "sample": f"{passes} passes over the first {n} of {wl.T} tokens ({el:.1f} s), all six "
                  f"ops (oracle in double, OpenMP over rows), GB/s over the passes' "
                  f"algorithmic bytes",
        "per_op_s": {k: round(v / passes, 6) for k, v in per_op.items()},
        # the whole step at the sample's rate: each op's time per pass scaled
        # by the tokens it sees in a full step over those of one pass
        "full_step_s_extrapolated": round(sum(
            v / passes * ((wl.T_swiglu / min(n, wl.T_swiglu)) if "swiglu" in k else wl.T / n)
            for k, v in per_op.items()), 3),
        "one_thread": {"tokens": n1, "seconds": round(el1, 4),
                       "GB_s": round(sum(tok_bytes(k, n1) for k in ib if k in OPS) / el1 / 1e9,
                                     3)},
        "nproc": os.cpu_count(), "cpu_model": cpu_model(),
    }


# -------------------------------------------------------------- our arm

def workload_config(wl, B, world):
    """The `config` object of the JSON line (both arms print the same)."""
    return {"workload": wl.name, "T": wl.T, "B": int(B), "H": wl.H, "I": wl.I,
            "T_swiglu": wl.T_swiglu, "Hq": wl.Hq, "Hkv": wl.Hkv, "D": wl.D,
            "theta": wl.theta, "eps": wl.eps,
            "parallelism": f"replicas x{world} (one batch per GPU, no collective)",
            "l2": "flushed before every step (256 MiB write, outside the step events); "
                  "the inputs are also larger than L2",
            "step": list(OPS)}


def kernel_entry(name, ms, ib, toks, hbm, src):
    gbs = ib / (ms * 1e-3) / 1e9
    return {"us": round(ms * 1e3, 2), "GB_s": round(gbs, 1),
            "frac_of_measured_hbm" if src == "measured" else "frac_of_fallback_hbm":
                round(gbs / hbm, 4),
            "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
            "tokens_per_s": round(toks / (ms * 1e-3), 1), "ideal_bytes": ib}


def copy_ops(batch, ib):
    """For each step op, a trivial streaming kernel over the same algorithmic
    bytes (half read, half written) at the same size: an elementwise fp32
    multiply by one, dst = src * 1, run on the SMs like the op (a device
    memcpy may take other engines and paths).  What bandwidth a kernel with
    no arithmetic reaches at this size, beside the op's own."""
    import torch
    dev = batch.inputs["x"].device
    # fp32 words, sizes rounded to 64 KiB (below 0.2% of any op's bytes)
    words = [max(1, ib[k] // 2 // 65536) * 16384 for k in OPS]
    src = torch.empty(max(words), dtype=torch.float32, device=dev)
    dst = torch.empty(max(words), dtype=torch.float32, device=dev)
    src.fill_(0.5)
    return [(lambda n=n: torch.mul(src[:n], 1.0, out=dst[:n])) for n in words], (src, dst)


def hold_gpu(ms=20.0):
    """Keeps the device busy for about `ms` so that the host enqueues the
    timed graphs ahead of it: no host submission gap lands inside a timed
    pair of events."""
    import torch
    torch.cuda._sleep(int(ms * 2.1e6))  # cycles at ~2.1 GHz


def reps_in_graph(op_bytes, target_us=300.0, cap=16):
    """How many [L2 flush, op] pairs one timed graph holds: enough that the
    smallest op's work in one replay reaches ~target_us.  The start and end
    of a graph replay, as CUDA events see them, move in steps of ~2 us (one
    process measured the same kernel at 10.24 and 12.29 us by turns), so
    small ops are timed over several pairs per replay and the difference is
    divided by their number."""
    est_us = min(op_bytes) / 6.0e6  # bytes over ~6 TB/s, in us
    return max(1, min(cap, int(round(target_us / max(est_us, 1.0)))))


def pair_graphs(ops, flush, m, fill):
    """Per op a graph of m pairs [L2 flush, op], and the graph of the m
    flushes alone."""
    import torch
    graphs = []
    for op in ops:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(m):
                flush.fill_(fill)
                op()
        graphs.append(g)
    fg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(fg):
        for _ in range(m):
            flush.fill_(fill)
    return graphs, fg


def time_pairs(graphs, fg, m, reps, dev):
    """Each op's device time: the median over `reps` repetitions of (its
    graph's time minus the flush graph's) / m, CUDA events around every
    replay, all enqueued behind a sleep kernel.  Returns per-op ms."""
    import torch
    for g in graphs + [fg]:
        g.replay()
    torch.cuda.synchronize(dev)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(len(graphs) + 1)] for _ in range(reps)]
    hold_gpu()
    for i in range(reps):
        for (a, b), g in zip(ev[i], graphs + [fg]):
            a.record()
            g.replay()
            b.record()
    torch.cuda.synchronize(dev)
    return [op_ms([e[j] for e in ev], [e[-1] for e in ev]) / m for j in range(len(graphs))]


def time_batch(batch, flush, K, Kk, dev, world=1, with_reference=True):
    """The step as one CUDA graph replayed K times (CUDA events around each
    replay), then each op as a graph of m pairs [L2 flush, op] beside a graph
    of m flushes (m from reps_in_graph), Kk repetitions.  With
    `with_reference`, the same repetitions also time an empty op (a
    one-element fill: the launch gap every op's time includes) and, per op,
    a streaming kernel over its algorithmic bytes.  Returns (step ms per
    replay, per-op ms, (t0, t1) of the step region, (t1, t2) of the
    per-kernel region, references with the pairs per graph)."""
    import torch
    import torch.distributed as dist

    from fine_tuning_gb300 import workloads as W
    ops = list(batch.ops())
    n_ops = len(ops)
    refs = {}
    keep = None
    if with_reference:
        tiny = torch.empty(1, dtype=torch.float32, device=dev)
        copies, keep = copy_ops(batch, W.ideal_bytes(batch.wl))
        ops += [lambda: tiny.fill_(1.0)] + copies
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for op in ops[:n_ops]:
            op()
    ib = W.ideal_bytes(batch.wl)
    m = reps_in_graph([ib[k] for k in OPS])
    op_graphs, flush_graph = pair_graphs(ops, flush, m, 3)
    graph.replay()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record()
        graph.replay()
        ev[i][1].record()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    t1 = time.time()
    per = time_pairs(op_graphs, flush_graph, m, Kk, dev)
    t2 = time.time()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    if with_reference:
        refs = {"launch_gap_ms": per[n_ops], "copy_ms": per[n_ops + 1:], "pairs_per_graph": m}
    del keep, op_graphs, flush_graph
    return step_ms, per[:n_ops], (t0, t1), (t1, t2), refs


def add_references(kernels, refs, ib):
    """Per kernel: the launch gap its time includes, and the same-size copy."""
    if not refs:
        return
    gap = refs["launch_gap_ms"]
    for j, name in enumerate(OPS):
        c = refs["copy_ms"][j]
        k = kernels[name]
        k["launch_gap_us"] = round(gap * 1e3, 2)
        k["copy_same_bytes_us"] = round(c * 1e3, 2)
        k["frac_of_same_size_copy"] = round(c * 1e3 / k["us"], 4)
        # the same figures with the launch gap taken out of the time: what the
        # kernel reaches when its launch overlaps the previous kernel (as in
        # the step's graph, launched with programmatic dependent launch)
        if k["us"] > 2 * gap * 1e3:
            scale = k["us"] / (k["us"] - gap * 1e3)
            k["GB_s_excl_launch_gap"] = round(k["GB_s"] * scale, 1)
            for key in ("frac_of_measured_hbm", "frac_of_fallback_hbm"):
                if key in k:
                    k[key + "_excl_launch_gap"] = round(k[key] * scale, 4)


def per_workload_leg(names, flush, K, Kk, dev, hbm, src, sampler, with_ext=True):
    """The smaller workloads, each timed like the main one (step graph and
    one-op graphs, and the widened ops) after its own sampled parity check,
    in the same run."""
    import torch

    from fine_tuning_gb300 import workloads as W
    out = {}
    for name in names:
        wl = W.WORKLOADS[name]
        b = Batch(wl, dev)
        rows, srows = parity_rows(wl, b.cu_host)
        inp = gather_inputs(b, rows, srows)
        for op in b.ops():
            op()
        torch.cuda.synchronize(dev)
        par = check_parity(wl, b.cu_host, rows, srows, inp, gather_outputs(b, rows, srows))
        for _ in range(3):
            flush.fill_(1)
            for op in b.ops():
                op()
        step_ms, per_op, _, (k0, k1), refs = time_batch(b, flush, K, Kk, dev)
        ib, toks = W.ideal_bytes(wl), W.tokens_per_call(wl)
        step_bytes = sum(ib[k] for k in OPS)
        ms = sum(step_ms) / len(step_ms)
        kern = {n: kernel_entry(n, per_op[j], ib[n], toks[n], hbm, src)
                for j, n in enumerate(OPS)}
        add_references(kern, refs, ib)
        dom = max(range(len(OPS)), key=lambda j: per_op[j])
        out[name] = {
            "T": wl.T, "B": int(len(b.cu_host) - 1), "H": wl.H, "I": wl.I, "Hq": wl.Hq,
            "Hkv": wl.Hkv, "D": wl.D, "step_ms": round(ms, 4),
            "step_GB_s": round(step_bytes / (ms * 1e-3) / 1e9, 1),
            "step_frac_of_hbm": round(step_bytes / (ms * 1e-3) / 1e9 / hbm, 4),
            "tokens_per_s": round(wl.T / (ms * 1e-3), 1), "kernels": kern,
            "pairs_per_graph": refs.get("pairs_per_graph", 1),
            "dominant": {"kernel": OPS[dom], "traffic": ncu_traffic(OPS[dom], wl.name)},
            "parity": par, "clocks_kernel_leg": sampler.summary(k0, k1)}
        if with_ext:
            ext = ext_leg(b, flush, dev, Kk, hbm, src)
            out[name]["extensions"] = {n: {f: v[f] for f in ("us", "GB_s", "frac_of_measured_hbm"
                                                              if src == "measured" else
                                                              "frac_of_fallback_hbm")}
                                       for n, v in ext.items() if isinstance(v, dict)}
        del b
        torch.cuda.empty_cache()
    return out


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
    wl = select_workload(args.workload, args.tokens)
    batch = Batch(wl, dev, seed_offset=rank)
    ops = batch.ops()
    ib = W.ideal_bytes(wl)
    step_bytes = sum(ib[k] for k in OPS)

    do_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    cut = head_tokens(batch, min(wl.T, 8192)) if do_cpu else None
    # parity of the step on rows spanning the whole batch, before any timing:
    # no number is printed unless it holds
    rows, srows = parity_rows(wl, batch.cu_host)
    inp = gather_inputs(batch, rows, srows)
    for op in ops:  # the parity step, on the untouched inputs
        op()
    torch.cuda.synchronize(dev)
    parity = check_parity(wl, batch.cu_host, rows, srows, inp,
                          gather_outputs(batch, rows, srows))
    del inp

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(max(args.warmup, 0)):
        flush.fill_(1)
        for op in ops:
            op()
    torch.cuda.synchronize(dev)

    K = args.steps
    Kk = args.kernel_reps if args.kernel_reps > 0 else max(1, min(K, 300))
    uuid = ""
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    sampler = ClockSampler(uuid).start()
    time.sleep(0.6)
    step_ms, per_op, (t0, t1), (k0, k1), refs = time_batch(batch, flush, K, Kk,
                                                                        dev, world)
    el_max, bytes_all = reduce_timing(sum(step_ms) / 1e3, step_bytes * K)
    _, tok_all = reduce_timing(0.0, float(wl.T) * K)
    value = bytes_all / el_max / 1e9
    hbm, src = peaks()
    toks = W.tokens_per_call(wl)
    kernels = {n: kernel_entry(n, per_op[j], ib[n], toks[n], hbm, src) for j, n in enumerate(OPS)}
    add_references(kernels, refs, ib)
    dom = max(range(len(OPS)), key=lambda j: per_op[j])
    dname = OPS[dom]
    achieved = ib[dname] / (per_op[dom] * 1e-3) / 1e9
    traffic = ncu_traffic(dname, wl.name)

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(el_max * 1e3 / K, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded packed batch; no dataset, no weights)",
        "config": workload_config(wl, len(batch.cu_host) - 1, world),
        "tokens_per_s": round(tok_all / el_max, 1),
        "frac_of_hbm": round(value / hbm, 4), "hbm_peak_GB_s": hbm, "hbm_peak_source": src,
        "frac_of_nominal_8tbs": round(value / NOMINAL_HBM_GBS, 4),
        "parity": parity,
        "kernels": kernels,
        "roofline": {"kernel": dname, "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "traffic": traffic, "algorithmic_bytes": ib[dname],
                     "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs, copy burst)"
                     if src == "measured" else "fallback 6.8 TB/s"},
        # this library's launches inside the timed region (the K steps), and
        # over every leg of the run
        "gpu_launches": LAUNCHES_PER_STEP * K,
        "gpu_launches_all_legs": LAUNCHES_PER_STEP * (K + Kk),
        "timing": (f"step: {K} replays of a CUDA graph of the step's {LAUNCHES_PER_STEP} "
                   f"launches, CUDA events around each replay; per kernel: the median over {Kk} "
                   f"replays of a graph of {refs.get('pairs_per_graph', 1)} pairs [L2 flush, op] "
                   "minus the same repetition's graph of as many L2 flushes, over their number "
                   "(several pairs per graph when the ops are small: a replay's start and end "
                   "move in ~2 us steps), CUDA events around each replay, enqueued behind a "
                   "sleep kernel so no host submission gap falls inside; launch_gap_us is an "
                   "empty one-element op timed the same way (included in every op's us; the "
                   "*_excl_launch_gap figures take it out); copy_same_bytes_us an elementwise "
                   "kernel (fp32 x 1) reading and writing the op's algorithmic bytes at the "
                   "same size"),
        "wall_ms_timed_region": round((t1 - t0) * 1e3, 3),
    }
    out["clocks"] = sampler.summary(t0, t1)
    out["clocks_kernel_leg"] = sampler.summary(k0, k1)
    if not args.no_ext:
        e0 = time.time()
        out["extensions"] = ext_leg(batch, flush, dev, Kk, hbm, src)
        out["extensions"]["clocks"] = sampler.summary(e0, time.time())
        out["gpu_launches_all_legs"] += sum(EXT_OPS.values()) * Kk
    torch.cuda.empty_cache()
    if rank == 0:
        names = [n for n in args.per_workload.split(",") if n and n != "none" and n != wl.name]
        if names:
            out["per_workload"] = per_workload_leg(names, flush, K, Kk, dev, hbm, src, sampler,
                                                   with_ext=not args.no_ext)
            out["gpu_launches_all_legs"] += len(names) * (LAUNCHES_PER_STEP * (K + Kk) + (
                0 if args.no_ext else sum(EXT_OPS.values()) * Kk))
        if not args.no_ext and not args.no_cce:
            c0 = time.time()
            out["cce"] = cce_leg(dev, flush, max(3, min(Kk, 20)))
            out["cce"]["clocks"] = sampler.summary(c0, time.time())
            out["gpu_launches_all_legs"] += out["cce"].pop("launches")
    sampler.stop()
    out["device_status"] = ftk.device_status(clear=True)  # 0: no pipeline wait ran out
    if out["device_status"] != 0:
        raise RuntimeError(f"a bounded pipeline wait ran out (status {out['device_status']})")

    if not args.no_e2e:
        out["e2e"] = e2e_leg(batch, ops, dev, args.e2e_steps, step_bytes)
    if do_cpu:
        out["cpu_baseline"] = cpu_leg(wl, batch.cu_host, cut, args.cpu_seconds)
        out["packing"] = packing_leg(wl)
    if rank == 0:
        print(json.dumps(out), flush=True)
        if args.records:
            with open(args.records, "w") as f:
                for rec in records_from(out):
                    f.write(json.dumps(rec) + "\n")
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def ext_leg(batch, flush, dev, reps, hbm, src):
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
    ib, toks = W.ideal_bytes(wl), W.tokens_per_call(wl)
    names = list(ops)
    m = reps_in_graph([ib[n] for n in names])
    graphs, fg = pair_graphs([ops[n] for n in names], flush, m, 5)
    per = dict(zip(names, time_pairs(graphs, fg, m, reps, dev)))
    del graphs, fg
    out = {}
    for n in names:
        out[n] = kernel_entry(n, per[n], ib[n], toks[n], hbm, src)
        out[n]["launches"] = EXT_OPS[n]
    out["timing"] = (f"the median over {reps} replays of a graph of {m} pairs [L2 flush, op] "
                     f"minus the same repetition's graph of {m} L2 flushes, over {m}, CUDA events "
                     "around each replay; outside the step's timed region")
    del h, y, rstd, dx, dw, res, dres, extra, qo, ko, rq, rk, nr_ws
    return out


def cce_leg(dev, flush, reps):
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
    names = list(ops)
    graphs, fg = pair_graphs([ops[n] for n in names], flush, 1, 9)  # ms-long ops: one pair
    per = dict(zip(names, time_pairs(graphs, fg, 1, reps, dev)))
    del graphs, fg
    peak, psrc = tensor_peak()
    flops = {"cce_fwd": 2 * hw.T * hw.H * hw.V, "cce_bwd": 6 * hw.T * hw.H * hw.V}
    chunk = ftk.cce_bwd_chunk(hw.T, hw.H, hw.V)
    nchunk = -(-hw.V // chunk)
    launches = {"cce_fwd": 3, "cce_bwd": 1 + 2 * nchunk}
    out = {"workload": {"name": hw.name, "T": hw.T, "H": hw.H, "V": hw.V,
                        "ignored_share": hw.ignored, "bwd_chunk": chunk},
           "loss": round(float(loss.item()), 6)}
    for n in names:
        ms = per[n]
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


class HostBuffers:
    """Page-locked host tensors of exactly the requested sizes, from
    cudaHostAlloc through the CUDA runtime the process already loaded
    (torch's pinned allocator rounds each allocation up to a power of two,
    which at the 524k-token shapes would cost ~92 GB of host memory instead of
    80).  Falls back to registering a plain host allocation
    (cudaHostRegister; slower on this host when both directions copy at
    once), then to torch's pinned allocator."""

    def __init__(self):
        self.allocated = []   # (ptr, cudart) to free with cudaFreeHost
        self.registered = []  # tensors to unregister
        self.rt = self._runtime()

    @staticmethod
    def _runtime():
        import ctypes
        for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
            try:
                rt = ctypes.CDLL(name)
                rt.cudaHostAlloc.restype = ctypes.c_int
                rt.cudaHostAlloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t,
                                             ctypes.c_uint]
                rt.cudaFreeHost.restype = ctypes.c_int
                rt.cudaFreeHost.argtypes = [ctypes.c_void_p]
                return rt
            except (OSError, AttributeError):
                continue
        return None

    def empty(self, shape, dtype):
        import ctypes

        import torch
        nbytes = int(torch.empty(0, dtype=dtype).element_size())
        for d in shape:
            nbytes *= int(d)
        if self.rt is not None and nbytes:
            ptr = ctypes.c_void_p()
            if self.rt.cudaHostAlloc(ctypes.byref(ptr), nbytes, 0) == 0 and ptr.value:
                buf = (ctypes.c_ubyte * nbytes).from_address(ptr.value)
                t = torch.frombuffer(buf, dtype=torch.uint8).view(dtype).view(*shape)
                if t.is_pinned():
                    self.allocated.append(ptr.value)
                    return t
                self.rt.cudaFreeHost(ptr.value)
        t = torch.empty(shape, dtype=dtype)
        rt = getattr(torch.cuda, "cudart", None)
        if rt is not None and t.numel():
            t.zero_()  # fault the pages in (OpenMP threads) before locking them
            if int(rt().cudaHostRegister(t.data_ptr(), t.numel() * t.element_size(), 0)) == 0:
                self.registered.append(t)
                return t
        return t.pin_memory()

    def kind(self):
        return ("cudaHostAlloc" if self.allocated else
                "cudaHostRegister" if self.registered else "torch pinned")

    def release(self):
        import torch
        for t in self.registered:
            torch.cuda.cudart().cudaHostUnregister(t.data_ptr())
        self.registered = []
        for p in self.allocated:
            self.rt.cudaFreeHost(p)
        self.allocated = []


COPY_CHUNK = 1 << 30  # bytes per host<->device copy piece in the e2e leg


def chunked_copy(dst, src, streams, k0=0):
    """dst.copy_(src) in pieces of at most COPY_CHUNK bytes dealt round-robin
    over `streams` (one host<->device copy of several GB runs slower than the
    same bytes in 1 GB pieces on two streams: 297 against 340 GB/s at 16 GB,
    both directions busy, measured on the GPU host).  Returns the next
    stream index."""
    import torch
    d = dst.reshape(-1).view(torch.uint8)
    s = src.reshape(-1).view(torch.uint8)
    k = k0
    for a in range(0, d.numel(), COPY_CHUNK):
        with torch.cuda.stream(streams[k % len(streams)]):
            d[a:a + COPY_CHUNK].copy_(s[a:a + COPY_CHUNK], non_blocking=True)
        k += 1
    return k


def e2e_leg(batch, ops, dev, steps, step_bytes):
    """The step through the public API with host buffers: every step copies
    all of its inputs in from page-locked host memory and all of its outputs
    back.  As a user would run consecutive steps, step k+1's copy-in, step
    k's kernels and step k-1's copy-out overlap (two copy streams per
    direction, one compute stream), with two device-side buffer sets; events
    order every reuse of a buffer."""
    import torch
    wl = batch.wl
    sets = [batch, Batch(wl, dev)]
    set_ops = [ops, sets[1].ops()]
    hb = HostBuffers()

    def outs(b):
        return {**b.outputs, **{k: b.inputs[k] for k in Batch.OUT_FROM_INPUTS}}
    host_in = {}
    for k in Batch.IN:
        v = batch.inputs[k]
        host_in[k] = hb.empty(v.shape, v.dtype)
        host_in[k].copy_(v)
    host_out = {k: hb.empty(v.shape, v.dtype) for k, v in outs(batch).items()}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    s_in = [torch.cuda.Stream(dev) for _ in range(2)]
    s_out = [torch.cuda.Stream(dev) for _ in range(2)]
    s_run = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=False)

    def mark(streams):
        out = []
        for st in streams:
            e = ev()
            e.record(st)
            out.append(e)
        return out

    def run(n, t0=None):
        done_run = [None, None]   # last compute on each set
        done_out = [None, None]   # last copy-out of each set (one event per stream)
        for i in range(n):
            j = i & 1
            b = sets[j]
            for st in s_in:
                if done_run[j] is not None:
                    st.wait_event(done_run[j])   # inputs of set j no longer read
            if i == 0 and t0 is not None:
                s_in[1].wait_stream(s_in[0])
                t0.record(s_in[0])
                s_in[1].wait_event(t0)
            k = 0
            for name, v in host_in.items():
                k = chunked_copy(b.inputs[name], v, s_in, k)
            e_in = mark(s_in)
            for e in e_in:
                s_run.wait_event(e)
            if done_out[j] is not None:
                for e in done_out[j]:
                    s_run.wait_event(e)        # outputs of set j already copied out
            with torch.cuda.stream(s_run):
                for op in set_ops[j]:
                    op()
            done_run[j] = ev()
            done_run[j].record(s_run)
            for st in s_out:
                st.wait_event(done_run[j])
            k = 0
            for name, v in outs(b).items():
                k = chunked_copy(host_out[name], v, s_out, k)
            done_out[j] = mark(s_out)
        for e in done_out[(n - 1) & 1] + (done_out[n & 1] or []):
            s_out[0].wait_event(e)
        return s_out[0]

    run(2)
    torch.cuda.synchronize(dev)
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    last = run(steps, t0=a)
    z.record(last)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(z) / steps
    del sets[1], set_ops[1]
    kind = hb.kind()
    del host_in, host_out
    hb.release()
    el_max, bytes_all = reduce_timing(ms * steps / 1e3, step_bytes * steps)
    return {"value": round(bytes_all / el_max / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(el_max * 1e3 / steps, 3), "steps": steps,
            "tokens_per_s": round(wl.T * steps / el_max, 1),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "copy_GB_s": round((h2d + d2h) / (el_max / steps) / 1e9, 1),
            "overlap": "copy-in of step k+1, kernels of step k and copy-out of step k-1 "
                       "overlap: two copy streams per direction (1 GB pieces), one compute "
                       "stream, two device buffer sets",
            "host_buffers": f"page-locked at exact size ({kind})"}


# ------------------------------------------------------ packing (host)

def packing_leg(wl, n_seq=200_000, batch=8):
    """See packing_corpus_leg; a workload of one fixed sequence (nothing to
    pack) takes the Qwen2.5-0.5B length mix and token budget instead."""
    from fine_tuning_gb300 import workloads as W
    if wl.lengths is not None and len(wl.lengths) <= 1:
        out = packing_corpus_leg(W.WORKLOADS["qwen2.5-0.5b"], n_seq, batch)
        out["length_mix_of"] = "qwen2.5-0.5b (this workload is one fixed sequence)"
        return out
    out = packing_corpus_leg(wl, n_seq, batch)
    out["length_mix_of"] = wl.name
    return out


def packing_corpus_leg(wl, n_seq=200_000, batch=8):
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
            "padding_waste_recovered": round(1 - waste_pack / waste_pad, 4) if waste_pad else None,
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
    wl = select_workload(args.workload, args.tokens)
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
    # the six step ops only (the oracle step runs those)
    sample_bytes = sum(ib[k] * (n / (wl.T_swiglu if "swiglu" in k else wl.T)) for k in OPS)
    value = sample_bytes * args.steps / el / 1e9
    sample = (f"first {n} of {wl.T} tokens per step, all six ops, oracle in double "
              f"(OpenMP over rows) on the host cores")
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded packed batch; no dataset, no weights)",
        "config": workload_config(wl, len(lens), world),
        "tokens_per_s": round(n * args.steps / el, 1),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample, "tokens_per_step": n},
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
