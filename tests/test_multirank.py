"""The multi-GPU path is data-parallel over tokens with no collective on the data path.  Its host
logic (token shards, max-over-ranks timing) is checked here with world-size-2 gloo process groups on
the CPU; the arithmetic on each shard is the oracle's."""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _token_range(T, rank, world):
    sys.path.insert(0, ROOT)
    import importlib.util
    spec = importlib.util.spec_from_file_location("shard", os.path.join(ROOT, "moe_finalize_residual_gb300", "shard.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m.token_range(T, rank, world)


@pytest.mark.parametrize("T,world", [(0, 2), (1, 2), (7, 2), (128, 2), (5, 8), (16384, 8)])
def test_token_ranges_partition_the_batch(T, world):
    ranges = [_token_range(T, r, world) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == T
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0
    sizes = [b - a for a, b in ranges]
    assert max(sizes) - min(sizes) <= 1


def _worker(rank, world, port, out_q):
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    case = synth.make_case("dp", T=9, H=256, K=4, R=2, E=16, rsf=2.5, shared=True)
    t0, t1 = _token_range(case.T, rank, world)
    mine = oracle.finalize(case, t0, t1)
    pieces = [None] * world
    dist.all_gather_object(pieces, (t0, t1, mine["residual_out"][t0:t1], mine["norm_out"][t0:t1]))
    # the benchmark's timing rule: the slowest rank decides
    t = torch.tensor([1.0 + rank], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    if rank == 0:
        full = oracle.finalize(case)
        ro = np.concatenate([p[2] for p in sorted(pieces, key=lambda p: p[0])])
        no = np.concatenate([p[3] for p in sorted(pieces, key=lambda p: p[0])])
        out_q.put((bool(np.array_equal(ro, full["residual_out"]) and np.array_equal(no, full["norm_out"])),
                   float(t.item())))
    dist.barrier()
    dist.destroy_process_group()


def test_sharded_oracle_equals_whole_batch_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    ok, tmax = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert ok and tmax == 2.0


def test_reference_arm_under_torchrun_gloo():
    """bench.py --impl reference with two ranks: rank 0 prints one JSON line, rank 1 exits cleanly."""
    port = _free_port()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
                        "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
                        "--gpus", "2", "--impl", "reference", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    import json
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
