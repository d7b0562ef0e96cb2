"""bench.py's multi-rank host logic on CPU, world size 2 (gloo; no GPU).

The core does not shard: `bench.py --gpus N` under torchrun runs N independent
replicas, and the only cross-rank operations are the barrier around the timed
region and the maximum of the per-rank step times.  Covered here:
  - that maximum (the same helper the GPU arm calls) over two gloo ranks;
  - the reference arm launched exactly as for N > 1 (torchrun, two ranks):
    rank 0 alone runs the oracle and prints one JSON line, the other rank
    exits 0 without work."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _max_worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r reports a step time of 10 + 7 r ms; every rank must see the slowest
        v = bench._max_over_ranks(10.0 + 7.0 * rank, world, torch.device("cpu"))
        out[rank] = v
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_max_worker, args=(world, _free_port(), out), nprocs=world,
                           start_method="spawn", join=True)
        got = dict(out)
    assert got == {0: 17.0, 1: 17.0}


def test_reference_arm_under_torchrun_world_2():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1",
           "--ref-tokens", "64"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2 and line["steps"] == 1 and line["warmup"] == 1
    assert line["unit"] == "tokens/s" and line["value"] > 0
    assert line["config"]["sample_tokens_per_step"] == 64
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
