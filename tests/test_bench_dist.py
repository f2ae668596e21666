"""Host logic of bench.py's replica mode, run as two gloo ranks on the CPU.

The path has no exchange step, so N GPUs run N independent replicas; what has
to be right is the bookkeeping around them: every rank joins the barrier, the
reported time is the maximum over ranks, only rank 0 prints, and the oracle
arm (--impl reference) runs on rank 0 alone while the other ranks exit 0.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.dist_barrier(w)
    # Rank r reports 1.5 + r ms; every rank must see the slowest one.
    got = bench.dist_max(1.5 + r, w)
    with open(os.path.join(out_dir, f"rank{r}.txt"), "w") as f:
        f.write(repr(got))
    dist.destroy_process_group()


def test_dist_max_and_barrier_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for r in range(world):
        assert float((tmp_path / f"rank{r}.txt").read_text()) == 1.5 + (world - 1)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_max(3.25, 1) == 3.25
    bench.dist_barrier(1)  # no-op without a process group


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_once_from_rank0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0", "--cpu-seconds", "0.5"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["value"] > 0


def test_cpu_baseline_parallel_oracle_processes():
    """The multi-core baseline runs the unchanged oracle in spawned processes
    from a common start; its figure counts every worker's bytes over the
    wall-clock span, and the single-thread figure is kept beside it."""
    sys.path.insert(0, ROOT)
    import bench
    gbs, nbytes, span = bench.oracle_gemv_parallel(0.3, 2, setup_s=3.0)
    per_block = bench.weight_bytes(1024, 4096, 8, 64)
    assert gbs > 0 and nbytes % per_block == 0 and nbytes >= 2 * per_block
    assert 0.3 <= span < 3.0
    d = bench.cpu_baseline(0.2)
    assert d["kind"] == "oracle" and d["unit"] == "GB/s"
    assert d["single_thread"]["cores"] == 1 and d["single_thread"]["value"] > 0
    if bench.host_cores() > 2:
        assert d["cores"] == bench.host_cores() - 1 and "parallel_error" not in d
