"""The multi-rank path of bench.py, on the CPU with gloo at world size 2.

Every rank draws its own batch (weak scaling, no collective on the data
path); a timed figure is the largest over the ranks; the reference arm prints
one JSON line, from rank 0 only, and the other ranks exit 0 without work."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _max_worker(rank, world, port, values, queue):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        queue.put((rank, bench.max_over_ranks(values[rank], world, device="cpu")))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    values = [1.25, 3.5]
    port = free_port()
    procs = [ctx.Process(target=_max_worker, args=(r, 2, port, values, queue)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert got == {0: 3.5, 1: 3.5}


def test_max_over_ranks_single_rank_is_identity():
    assert bench.max_over_ranks(2.75, 1) == 2.75


def test_each_rank_draws_its_own_batch():
    from gated_deltanet_mixer_gb300 import inputs as I

    assert bench.rank_case(7, 0) == 7
    cases = {bench.rank_case(7, r) for r in range(8)}
    assert len(cases) == 8
    a = I.prefill_problem(1, 64, 1, 2, io="bf16", case=bench.rank_case(5, 0))
    b = I.prefill_problem(1, 64, 1, 2, io="bf16", case=bench.rank_case(5, 1))
    assert not np.array_equal(a["qkv_pre"], b["qkv_pre"])


def test_reference_arm_under_torchrun_prints_once():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3", "--ref-budget", "2",
           "--workload", "0.8b_prefill"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2
    assert line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
