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


# --------------------------------------------------------------------------------------------------
# The tensor-parallel one-shot exchange (moe_finalize_residual_gb300/tp.py): every rank finalizes its
# own partial, the rounded rows are exchanged by an all-gather over a gloo group, and every rank sums the
# R slots in rank order with the residual add and RMSNorm.  The compute steps here are the oracle's; the
# protocol (slot order, the masked-route composition, the exchange of raw bits) is the product's.

def _tp_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("tp", os.path.join(ROOT, "moe_finalize_residual_gb300", "tp.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _tp_worker(rank, world, port, act, out_q):
    sys.path.insert(0, ROOT)
    import dataclasses
    import oracle
    import synth
    tp = _tp_module()
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)

    @dataclasses.dataclass
    class P:  # the fields of the library's Partial, in its order
        gemm2_out: torch.Tensor
        perm_idx: torch.Tensor
        expert_scale: object = None
        shared_out: object = None

    case = synth.make_case("tp", T=11, H=512, K=6, R=world, E=32, rsf=2.5, shared=True, act_dtype=act,
                           mask_quarter=True, scale_dtype=torch.float32)
    local = P(case.gemm2[rank], case.perm[rank], case.scale[rank], case.shared[rank])

    def as_act(bits):
        return torch.from_numpy(bits.view(np.int16)).view(act)

    def one_case(parts, rsf, residual, gamma):
        import dataclasses as dc
        return dc.replace(case, R=len(parts), rsf=float(rsf), gemm2=[q.gemm2_out for q in parts],
                          perm=[q.perm_idx for q in parts], scale=[q.expert_scale for q in parts],
                          shared=[q.shared_out for q in parts], expert=[torch.zeros(0)] * len(parts),
                          residual=residual, gamma=gamma,
                          K=parts[0].perm_idx.shape[1], scale_dtype=None if parts[0].expert_scale is None else
                          parts[0].expert_scale.dtype)

    def finalize_partial(part, rsf):  # one partial: the routed output is the rounded partial itself
        return as_act(oracle.finalize(one_case([part], rsf, case.residual, case.gamma))["routed"])

    def fused(parts, residual, gamma, eps):
        o = oracle.finalize(one_case(parts, 1.0, residual, gamma))
        return as_act(o["residual_out"]), as_act(o["norm_out"])

    ro, no = tp.tp_finalize_fused(local, case.residual, case.gamma, routed_scaling_factor=case.rsf, eps=case.eps,
                                  finalize_partial=finalize_partial, fused=fused)
    want = oracle.finalize(case)
    ok = (np.array_equal(ro.view(torch.int16).numpy().view(np.uint16), want["residual_out"]) and
          np.array_equal(no.view(torch.int16).numpy().view(np.uint16), want["norm_out"]))
    out_q.put((rank, ok))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,act", [(2, torch.bfloat16), (4, torch.float16)])
def test_tp_one_shot_exchange_equals_single_gpu_gloo(world, act):
    """Each of `world` gloo ranks holds one partial; after the exchange every rank's residual_out and
    norm_out equal, bit for bit, the single-GPU finalize of all the partials in rank order."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_tp_worker, args=(r, world, port, act, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(results[r] for r in range(world)), results


def test_tp_rank_order_matters():
    """The slots are summed in rank order: on partial rows 2^24, 1 and -2^24 (one route, scale 1, factor 1)
    the FP32 sum in order 0, 1, 2 is 0 while the reverse order gives 1, so a reordered exchange is caught."""
    sys.path.insert(0, ROOT)
    import dataclasses
    import oracle
    import synth
    tp = _tp_module()
    T, H = 4, 64
    case = synth.make_case("tpo", T=T, H=H, K=1, R=3, E=4, rsf=1.0)
    case.residual = torch.zeros_like(case.residual)
    for r, v in enumerate((2.0 ** 24, 1.0, -(2.0 ** 24))):
        case.gemm2[r] = torch.full_like(case.gemm2[r], v)
        case.scale[r] = torch.ones_like(case.scale[r])

    @dataclasses.dataclass
    class P:
        gemm2_out: torch.Tensor
        perm_idx: torch.Tensor
        expert_scale: object = None
        shared_out: object = None
    parts = [P(case.gemm2[r], case.perm[r], case.scale[r], case.shared[r]) for r in range(case.R)]

    def composed(order):
        slots = []
        for r in order:
            one = dataclasses.replace(case, R=1, gemm2=[parts[r].gemm2_out], perm=[parts[r].perm_idx],
                                      scale=[parts[r].expert_scale], shared=[parts[r].shared_out])
            slots.append(torch.from_numpy(oracle.finalize(one)["routed"].view(np.int16)).view(case.act_dtype))
        ex = tp.exchanged_partials(slots, P)
        c2 = dataclasses.replace(case, R=len(ex), K=1, scale_dtype=None, gemm2=[e.gemm2_out for e in ex],
                                 perm=[e.perm_idx for e in ex], scale=[None] * len(ex), shared=[e.shared_out for e in ex])
        return oracle.finalize(c2)["residual_out"]
    want = oracle.finalize(case)["residual_out"]
    assert np.array_equal(composed([0, 1, 2]), want)
    assert (torch.from_numpy(want.view(np.int16)).view(torch.bfloat16) == 0).all()
    assert not np.array_equal(composed([2, 1, 0]), want)
