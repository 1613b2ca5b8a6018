"""The masked all-reduce expert-parallel mode through libep on one GPU.

HF transformers, "Expert-parallel implementations for ep_dispatch_experts",
the "all_reduce" implementation: each rank of the expert group masks the
routes to other ranks' experts on the shared batch, runs its own experts,
and one all-reduce sums the outputs (the backward all-reduces the input
gradient).  Here the two ranks' halves of the experts run as two independent
handles of one registered layer on one GPU, one after the other on the same
stream; no kernel waits on another, and the all-reduce is a float32 sum taken
by torch after both finish.  The collective itself is covered on CPU ranks
(test_allreduce_mode.py).

Small-integer tokens, gradients and weights keep every partial result and
every sum exact, so the summed halves must equal the full step bit for bit;
each half is also compared with the oracle bit for bit.
"""
import numpy as np
import pytest
import torch

from combine_ep_prepare_gb300 import workloads as wl
from ep_harness import GpuLayer, bits

pytestmark = pytest.mark.gpu

E, K, T, H = 256, 8, 128, 7168


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_ep_prepare_gb300 as ep
    return ep


def _gpu_step(ep, layer, idx, x, g, wts):
    """dispatch -> identity experts -> weighted combine, and back."""
    R = layer.R
    h = layer.handle()
    dev = "cuda"
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    recv = torch.zeros(R, H, dtype=torch.bfloat16, device=dev)
    recv_w = torch.zeros(R, dtype=torch.float32, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    gexp = torch.zeros(R, H, dtype=torch.bfloat16, device=dev)
    gw = torch.zeros(R, dtype=torch.float32, device=dev)
    gtok = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    gtw = torch.empty(T, K, dtype=torch.float32, device=dev)
    idx_d = idx.to(dev)
    ep.ep_prepare(h, idx_d, counts, 1)
    ep.ep_dispatch(h, idx_d, x.to(dev), wts.to(dev), recv, recv_w)
    ep.ep_combine_weighted(h, recv, recv_w, out)
    ep.ep_combine_weighted_bwd(h, g.to(dev), recv, recv_w, gexp, gw)
    ep.ep_dispatch_bwd(h, gexp, gw, gtok, gtw)
    info = ep.ep_read_info(h)
    assert info["status"] == 0
    return out, gtok, gtw, info["used_rows"]


def _oracle_step(oracle_mod, idx, x, g, wts):
    rt = oracle_mod.prepare(idx.numpy(), E, 1)
    recv, recv_w = oracle_mod.dispatch(rt, bits(x), wts.numpy())
    out = oracle_mod.combine_weighted(rt, recv, recv_w)
    gexp, gw = oracle_mod.combine_bwd_weighted(rt, bits(g), recv_w, recv)
    gtok, gtw = oracle_mod.dispatch_bwd(rt, gexp, gw.astype(np.float32))
    return out, gtok, gtw


def test_two_halves_sum_to_full_step(ep, oracle_mod):
    w = wl.Workload("decode_unmasked", 4, T=T, H=H, E=E, K=K, A=1, routing="grouped")
    idx, _ = wl.routing(w)
    x = wl.small_int_bf16(T, H, seed=61)
    g = wl.small_int_bf16(T, H, seed=62)
    wts = torch.from_numpy(np.random.default_rng(63).integers(-2, 3, (T, K)).astype(np.float32))
    layer = GpuLayer(ep, E, K, H, T, 1)
    halves = []
    for rank in range(2):
        local = (idx >= rank * 128) & (idx < (rank + 1) * 128)
        idx_r = idx.masked_fill(~local, -1)
        out, gtok, gtw, used = _gpu_step(ep, layer, idx_r, x, g, wts)
        o_out, o_gtok, o_gtw = _oracle_step(oracle_mod, idx_r, x, g, wts)
        assert used == int(local.sum())
        assert np.array_equal(bits(out), o_out)
        assert np.array_equal(bits(gtok), o_gtok)
        assert np.array_equal(gtw.cpu().numpy().view(np.uint32), o_gtw.view(np.uint32))
        halves.append((out.float(), gtok.float(), gtw))
    full = _gpu_step(ep, layer, idx, x, g, wts)
    torch.cuda.synchronize()
    assert torch.equal(halves[0][0] + halves[1][0], full[0].float())
    assert torch.equal(halves[0][1] + halves[1][1], full[1].float())
    assert torch.equal(halves[0][2] + halves[1][2], full[2])
    assert not torch.equal(halves[0][0], full[0].float())
