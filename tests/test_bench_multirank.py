"""bench.py's multi-rank host logic on CPU: two gloo ranks agree on the
slowest rank's time, replicas draw independent inputs, and the reference arm
under torchrun prints exactly one line, from rank 0."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _max_worker(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        got = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
        with open(os.path.join(out_dir, f"r{rank}"), "w") as f:
            f.write(repr(got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    port = _free_port()
    mp.start_processes(_max_worker, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    assert [float((tmp_path / f"r{r}").read_text()) for r in (0, 1)] == [15.0, 15.0]


def test_max_over_ranks_without_a_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5


def test_replicas_draw_independent_ids():
    from moe_expert_routing_ids_gb300 import workloads as W
    a = W.SMALL.ids(replica=0)
    b = W.SMALL.ids(replica=1)
    assert a.shape == b.shape and not np.array_equal(a, b)
    assert np.array_equal(a, W.SMALL.ids(replica=0))


def test_reference_slice_is_a_multiple_of_R_within_T():
    sys.path.insert(0, ROOT)
    import bench
    from moe_expert_routing_ids_gb300 import workloads as W
    w = W.STRESS
    for rate, steps in ((1.3e7, 400), (1.3e7, 2), (1e3, 10), (1e12, 1)):
        t = bench.reference_slice_tokens(w, rate, steps, 3, 120.0)
        assert t % w.R == 0 and w.R <= t <= w.T


def test_reference_arm_under_torchrun_prints_one_line():
    env = dict(os.environ, OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1",
           "--ref-budget-s", "2"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 2
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"
