"""The N>1 host logic of bench.py on CPU: two gloo ranks.

Each rank runs its own batch, so the only cross-rank step is the timing
reduction: the job's elapsed time is the slowest rank's, the work done is
the sum over ranks.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        assert bench.rank_info() == (rank, rank, world)
        el, units = bench.reduce_timing(1.0 + rank, 100.0 * (rank + 1))
        out[rank] = (el, units)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_reduce_timing_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    assert out[0] == out[1] == (2.0, 300.0)


def test_reduce_timing_single_process_is_identity():
    import bench
    assert bench.reduce_timing(0.5, 7.0) == (0.5, 7.0)


def test_reference_arm_json_line():
    # the oracle arm of bench.py runs on the host alone: one JSON line with
    # the keys the benchmark contract asks of it
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2",
                          "--warmup", "1", "--reference-seconds", "1", "--workload", "tiny_f32"],
                         cwd=root, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["config"]["workload"] == "tiny_f32" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
