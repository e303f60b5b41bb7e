"""The multi-process (replica) path of bench.py on CPU: two gloo ranks on this host.

The product path does not shard a single product across GPUs (every rank runs its own
replica of the layer step; nothing is exchanged on the data path).  What bench.py does with
several ranks -- a barrier on both sides of the timed region and the slowest rank's time --
is host logic, tested here with world_size 2 over gloo, without a GPU.
"""
import json
import os
import socket
import subprocess
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    args = types.SimpleNamespace(impl="reference")
    w, r, local = bench.dist_setup(args)
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    # each rank reports its own step time; all ranks must agree on the slowest
    slowest = bench.max_over_ranks(10.0 + rank, w)
    bench.barrier(w)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(repr(slowest))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2(tmp_path):
    import torch.multiprocessing as mp
    port = free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    for r in range(2):
        assert float((tmp_path / f"rank{r}.txt").read_text()) == 11.0


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)  # no process group: nothing to wait for


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_world2():
    # the driver's launch for N > 1: rank 0 alone times the oracle and prints one line,
    # the other rank exits 0 without work
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, env=env, timeout=280)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 1
    assert d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle"
