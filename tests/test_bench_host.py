"""Host-side logic of bench.py that needs no GPU: workload slices, the rows
the in-run parity check samples, the config both arms print, and the
oracle arm at the default (largest) workload."""
import json
import os
import subprocess
import sys

import numpy as np

import bench
from fine_tuning_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_default_workload_is_the_largest_single_gpu_one():
    args = bench.parse_args([])
    assert args.workload == "qwen3-32b-524k"
    assert max(W.WORKLOADS.values(), key=lambda w: w.T).name == args.workload
    # the smaller bf16 workloads are timed beside it in the same run
    assert set(args.per_workload.split(",")) == {"qwen2.5-0.5b", "llama-3.2-1b", "qwen3-8b"}


def test_slice_keeps_row_shapes_and_cuts_sequences():
    full = W.WORKLOADS["qwen3-32b-524k"]
    s = bench.select_workload("qwen3-32b-524k", 32768)
    assert (s.T, s.T_swiglu, s.H, s.I, s.Hq, s.Hkv, s.D) == \
        (32768, 32768, full.H, full.I, full.Hq, full.Hkv, full.D)
    assert W.draw_lengths(s).tolist() == [32768] and s.name == "qwen3-32b-524k[:32768]"
    # a batch of many sequences is cut at the slice's end
    s2 = bench.select_workload("qwen2.5-0.5b", 1000)
    lens = W.draw_lengths(s2)
    full_lens = W.draw_lengths(W.WORKLOADS["qwen2.5-0.5b"])
    assert lens.sum() == 1000 and lens[:-1].tolist() == full_lens[:len(lens) - 1].tolist()
    assert bench.select_workload("qwen2.5-0.5b", 0) is W.WORKLOADS["qwen2.5-0.5b"]


def test_parity_rows_span_the_batch():
    wl = W.WORKLOADS["qwen3-32b-524k"]
    cu = W.cu_seqlens_from_lengths(W.draw_lengths(wl))
    rows, srows = bench.parity_rows(wl, cu)
    assert rows[0] == 0 and rows[-1] == wl.T - 1 and srows[-1] == wl.T_swiglu - 1
    assert np.all(np.diff(rows) > 0) and (rows > wl.T // 2).sum() > 64
    wl2 = W.WORKLOADS["qwen2.5-0.5b"]
    cu2 = W.cu_seqlens_from_lengths(W.draw_lengths(wl2))
    rows2, _ = bench.parity_rows(wl2, cu2)
    for c in cu2[1:17]:  # both sides of the first sequence boundaries
        assert c in rows2 and c - 1 in rows2
    tiny = W.WORKLOADS["tiny_f32"]
    r3, s3 = bench.parity_rows(tiny, W.cu_seqlens_from_lengths(W.draw_lengths(tiny)))
    assert r3.tolist() == list(range(tiny.T)) and s3.tolist() == list(range(tiny.T_swiglu))


def test_packing_leg_on_a_single_sequence_workload_uses_a_length_mix():
    out = bench.packing_leg(W.WORKLOADS["qwen3-32b-524k"], n_seq=3000)
    assert out["length_mix_of"].startswith("qwen2.5-0.5b")
    assert out["bins"] >= 1 and 0 < out["fill"] <= 1


def test_reference_arm_prints_our_config_at_the_default_workload():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "0", "--reference-seconds", "1"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    d = json.loads([ln for ln in out.stdout.splitlines() if ln.startswith("{")][-1])
    wl = W.WORKLOADS["qwen3-32b-524k"]
    assert d["config"] == bench.workload_config(wl, 1, 1)
    assert d["cpu_baseline"]["tokens_per_step"] >= 1 and d["value"] > 0


def test_launch_gap_figures():
    """The per-kernel figures with the launch gap taken out: the same bytes
    over the kernel's time minus the gap; none for a time within twice it."""
    ib = {k: 1000 for k in bench.OPS}
    kernels = {}
    for j, k in enumerate(bench.OPS):
        us = 10.0 if j else 3.0
        kernels[k] = bench.kernel_entry(k, us / 1e3, ib[k] * 1_000_000, 1000, 5000.0, "measured")
    refs = {"launch_gap_ms": 2e-3, "copy_ms": [8e-3] * len(bench.OPS)}
    bench.add_references(kernels, refs, ib)
    k = kernels[bench.OPS[1]]
    assert k["launch_gap_us"] == 2.0 and k["frac_of_same_size_copy"] == 0.8
    assert abs(k["GB_s_excl_launch_gap"] - 1e9 / 8e-6 / 1e9) < 0.1       # 1 GB in 8 us
    assert abs(k["frac_of_measured_hbm_excl_launch_gap"] - 125000 / 5000.0) < 1e-3
    assert "GB_s_excl_launch_gap" not in kernels[bench.OPS[0]]          # 3 us < 2 x 2 us


def test_pairs_per_graph():
    """Small ops are timed over several [flush, op] pairs per graph, large
    ones over one."""
    assert bench.reps_in_graph([58_787_584, 478_150_656]) == 16          # ~10 us op: capped
    assert bench.reps_in_graph([268_570_624]) == 7                       # ~45 us
    assert bench.reps_in_graph([10_739_525_632, 19_327_352_832]) == 1    # ms-long ops


def test_cpu_leg_on_a_small_sample():
    """The oracle baseline leg on CPU inputs: a rate, its sample, and the
    extrapolated full step (SwiGLU scaled by its own token count)."""
    wl = bench.select_workload("qwen2.5-0.5b", 512)
    cut = {}
    cut.update(W.rmsnorm_inputs(wl, "cpu"))
    cut.update(W.swiglu_inputs(wl, "cpu"))
    cut.update(W.rope_inputs(wl, "cpu"))
    cu = W.cu_seqlens_from_lengths(W.draw_lengths(wl))
    out = bench.cpu_leg(wl, cu, {k: cut[k] for k in ("x", "w", "dy", "g", "u", "dh", "q", "k",
                                                    "dq", "dk")}, 0.5)
    assert out["value"] > 0 and out["kind"] == "oracle" and out["cores"] >= 1
    assert set(out["per_op_s"]) == set(bench.OPS)
    full = out["full_step_s_extrapolated"]
    n = int(out["sample"].split(" passes over the first ")[1].split(" ")[0])
    expect = sum(v * (wl.T / n) for v in out["per_op_s"].values())  # T_swiglu = T here
    assert abs(full - expect) <= 1e-3 + 1e-6 * expect


def test_records_flatten_every_workload_and_op():
    k = {"us": 10.0, "GB_s": 5000.0, "frac_of_measured_hbm": 0.75, "frac_of_nominal_8tbs": 0.6,
         "tokens_per_s": 1e9, "ideal_bytes": 5e7}
    out = {"config": {"workload": "qwen3-32b-524k", "T": 524288, "H": 5120},
           "kernels": {"rmsnorm_fwd": dict(k), "qk_rope_bwd": dict(k)},
           "extensions": {"swiglu_bwd_h": dict(k), "timing": "text"},
           "parity": {"max_err_over_bound": 0.25},
           "per_workload": {"qwen2.5-0.5b": {"T": 16384, "H": 896,
                                             "kernels": {"swiglu_fwd": dict(k)},
                                             "parity": {"max_err_over_bound": 0.1}}}}
    recs = bench.records_from(out)
    assert [(r["workload"], r["op"], r["dir"]) for r in recs] == [
        ("qwen3-32b-524k", "rmsnorm", "fwd"), ("qwen3-32b-524k", "qk_rope", "bwd"),
        ("qwen3-32b-524k", "swiglu_h", "bwd"), ("qwen2.5-0.5b", "swiglu", "fwd")]
    assert recs[0]["shapes"] == {"T": 524288, "H": 5120} and recs[0]["frac_of_hbm"] == 0.75
    assert recs[-1]["parity_max_err_over_bound"] == 0.1 and recs[-1]["shapes"]["H"] == 896
