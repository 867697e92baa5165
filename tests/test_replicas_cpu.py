"""Multi-process host logic of bench.py on CPU (gloo, world size 2).

The decode step does not shard: with N GPUs the bench runs N independent
replicas, each on its own batch, with no collective on the data path.  What
the ranks do share is control: a barrier around the timed region, the maximum
of the per-rank step times, and rank 0 alone printing.  These tests run that
logic as two gloo ranks on the host."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    r, w, _ = bench.dist_env()
    bench.dist_init(w, "gloo")
    try:
        bench.barrier(w)
        # step times differ per rank; every rank must see the slowest
        slowest = bench.max_over_ranks(1.5 + r, w)
        seed = bench.replica_seed(r)
        # each replica draws its own batch of the same shape
        from sparse_latent_attention_decode_b300 import synth
        wl = synth.small_workload(2, [40, 33], k=16, K=16, S_cap=40)
        t = synth.make_inputs(wl, seed=seed, threads=1)
        digest = float(t["q_nope"].float().sum()) + float(t["topk_idx"].sum())
        # the reference arm runs on rank 0 only; other ranks return None
        args = type("A", (), {"workload": "p1000_b1", "seed": 0, "warmup": 0, "steps": 1})()
        ref_is_none = bench.run_reference(args) is None if r != 0 else None
        bench.barrier(w)
        q.put((r, slowest, seed, digest, ref_is_none))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_share_only_control():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, seed0, d0, _), (r1, s1, seed1, d1, ref1) = res
    assert (r0, r1) == (0, 1)
    assert s0 == s1 == 2.5            # max over ranks, seen by both
    assert seed0 != seed1             # independent replicas
    assert d0 != d1                   # ... drawing different batches
    assert ref1 is True               # rank 1 does no reference work


def test_single_process_helpers_need_no_process_group():
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)
    assert bench.replica_seed(0) == 0 and bench.replica_seed(1, base=5) != 5


def test_bench_spawns_its_own_ranks_for_gpus_n():
    # `bench.py --gpus 2` started without torchrun launches two ranks itself;
    # rank 0 alone prints one line, and that line counts both.  The reference
    # arm runs on the host, so the spawn path is exercised without a GPU.
    import json
    import subprocess
    import sys
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    out = subprocess.run([sys.executable, os.path.join(os.path.dirname(bench.__file__), "bench.py"),
                          "--gpus", "2", "--impl", "reference", "--workload", "p1000_b1", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    rec = json.loads(lines[0])
    assert rec["n_gpus"] == 2 and rec["impl"] == "reference"
