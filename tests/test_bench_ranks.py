"""The bench's bookkeeping for N > 1 ranks (independent replicas, one process per
GPU), exercised with two gloo ranks on CPU: every rank sees the slowest rank's
time, and the reference arm runs on rank 0 alone (the others exit 0 silently).
"""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.ranks_init("cpu")
    assert (w, r, local) == (world, rank, rank)
    bench.ranks_barrier(w)
    # rank i took 10 + 5 i ms: the job took as long as its slowest rank
    t = bench.max_over_ranks(10.0 + 5.0 * rank, w, "cpu")
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(repr(t))
    bench.ranks_done(w)


def test_slowest_rank_time_over_two_gloo_ranks(tmp_path):
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    got = [float((tmp_path / f"rank{i}.txt").read_text()) for i in range(2)]
    assert got == [15.0, 15.0]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    bench.ranks_barrier(1)
    bench.ranks_done(1)


@pytest.mark.parametrize("workload", ["decode", "float_tiny", "qkv_tiny", "gmm_tiny"])
def test_reference_arm_runs_on_rank_zero_only(workload):
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload,
                        "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
