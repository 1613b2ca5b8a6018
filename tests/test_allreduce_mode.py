"""The masked all-reduce expert-parallel mode, on two CPU ranks (gloo).

HF transformers, "Expert-parallel implementations for ep_dispatch_experts",
the "all_reduce" implementation (table of implementations and the AllReduceEP
discussion): every rank of the expert group holds the same batch, masks the
routes to experts that other ranks own, runs its own experts on the rest, and
one all-reduce sums the outputs; the backward all-reduces the gradient of the
shared input.  With routes masked to -1 the per-rank step is exactly the
single-GPU path (the decode workload: 256 experts, 128 of them local).

Each rank runs the oracle's prepare, dispatch, weighted combine and their
backward passes on its half of the experts, and torch.distributed sums the
results.  Tokens, gradients and weights are small integers, so every partial
result and every sum is exact: the all-reduced outputs must equal the
single-rank step over all experts bit for bit.
"""
import os
import socket
import sys

import numpy as np
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
E, K, T, H = 256, 8, 128, 64


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _inputs():
    """Decode-shaped grouped routing before masking, and small-integer
    tokens, upstream gradient and weights."""
    from combine_ep_prepare_gb300 import workloads as wl
    w = wl.Workload("decode_unmasked", 4, T=T, H=H, E=E, K=K, A=1, routing="grouped")
    idx, _ = wl.routing(w)
    x = wl.small_int_bf16(T, H, seed=51)
    g = wl.small_int_bf16(T, H, seed=52)
    wts = np.random.default_rng(53).integers(-2, 3, (T, K)).astype(np.float32)
    return idx.numpy(), x, g, wts


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _f32(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).float()


def _step(oracle, idx, x, g, wts):
    """Forward (dispatch, identity experts, weighted combine) and backward
    (weighted combine backward, dispatch backward) on one routing."""
    rt = oracle.prepare(idx, E, 1)
    recv, recv_w = oracle.dispatch(rt, _bits(x), wts)
    out = oracle.combine_weighted(rt, recv, recv_w)
    gexp, gw = oracle.combine_bwd_weighted(rt, _bits(g), recv_w, recv)
    gtok, gtw = oracle.dispatch_bwd(rt, gexp, gw.astype(np.float32))
    return _f32(out), _f32(gtok), gtw


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        idx, x, g, wts = _inputs()
        per_rank = E // world
        local = (idx >= rank * per_rank) & (idx < (rank + 1) * per_rank)
        part = _step(oracle, np.where(local, idx, -1), x, g, wts)
        summed = []
        for t in (part[0], part[1], torch.from_numpy(part[2])):
            t = t.clone()
            dist.all_reduce(t, op=dist.ReduceOp.SUM)
            summed.append(t)
        full = _step(oracle, idx, x, g, wts)
        ok = (torch.equal(summed[0], full[0]) and torch.equal(summed[1], full[1])
              and np.array_equal(summed[2].numpy(), full[2]))
        # both ranks own some routes, so neither partial is the whole answer
        ok = ok and bool(local.any()) and not torch.equal(part[0], full[0])
        out[rank] = "ok" if ok else "mismatch"
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_two_rank_masked_all_reduce(oracle_mod):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    assert dict(out) == {0: "ok", 1: "ok"}
