"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the timing
reduction takes the max over ranks, the reference arm runs on rank 0 only, and
the data path needs no collective (each rank's replica is independent)."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.max_over_ranks(dist, float(10 + 5 * rank))
        bench.barrier(dist)
        q.put((rank, m))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 15.0, 1: 15.0}


def test_reference_arm_rank0_only():
    """Under torchrun with 2 ranks, only rank 0 prints the reference line."""
    port = _free_port()
    env = dict(os.environ, OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--gpus", "2",
           "--impl", "reference", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    import json
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["unit"] == "tokens/s"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0


def _replica_worker(rank, world, port, q):
    """One rank of a replica run: draw this rank's inputs, time a fake step, reduce."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import hashlib
    import torch
    import torch.distributed as dist
    import bench
    import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        d = synth.make_inputs(1, 64, 2, seed=rank, init_dtype="bf16")   # as bench.py: seed = rank
        h = hashlib.sha256()
        for name in ("q", "k", "v", "g", "beta"):
            h.update(d[name].tobytes())
        digest = torch.tensor(list(h.digest()[:8]), dtype=torch.int64)
        all_digests = [torch.zeros_like(digest) for _ in range(world)]
        dist.all_gather(all_digests, digest)
        elapsed = bench.max_over_ranks(dist, 100.0 + 50.0 * rank)   # rank 1 is the slower one
        prof = {"fused_kernel": (elapsed, 4)}
        line = bench.workload_line("prefill_t8192_h96", d, elapsed, prof, 4, world, 1)
        q.put((rank, [t.tolist() for t in all_digests], elapsed, line["value"]))
    finally:
        dist.destroy_process_group()


def test_replicas_draw_different_inputs_and_value_counts_every_rank():
    """Two replica ranks (gloo): rank r draws its inputs with seed r, so the replicas run
    different data; the step time is the slowest rank's, and `value` counts the tokens
    of both ranks over that time."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_replica_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict((r, rest) for r, *rest in (q.get(timeout=180) for _ in range(2)))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    digests0, elapsed0, value0 = res[0]
    digests1, elapsed1, value1 = res[1]
    assert digests0 == digests1 and digests0[0] != digests0[1]
    assert elapsed0 == elapsed1 == 150.0
    tokens_per_step = 64                      # B * T of each rank's inputs
    assert value0 == value1 == pytest.approx(2 * tokens_per_step * 4 / 0.150)
