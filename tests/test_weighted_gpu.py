"""GPU parity of the weighted combine (fused weight multiply) and its backward.

The forward and the token-gradient half of the backward are compared bit for
bit with the oracle.  The weight gradient g_w[s] = sum_h grad[t][h] *
expert_out[s][h] is a float32 dot product whose order the pages do not fix:
every product of two bf16 values is exact in float32, so any order of the H
additions is within (H - 1) * 2^-24 * sum_h |grad * expert_out| of the exact
sum, which the oracle gives in float64; that bound is the tolerance.

Weighted combine: TransformerEngine PR #3035, review thread on the weight
multiply inside combine (made optional); backward by differentiation of it.
"""
import numpy as np
import pytest
import torch

from combine_ep_prepare_gb300 import workloads as wl
from ep_harness import GpuLayer, bits, SENTINEL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_ep_prepare_gb300 as ep
    return ep


def run_weighted(ep, oracle_mod, idx, E, H, A, seed, check_rows=None):
    T, K = idx.shape
    rt = oracle_mod.prepare(idx.numpy(), E, A)
    rows = max(rt.P, 1)
    y = wl.bf16_normal(rows, H, seed + 1)
    w = wl.f32_normal(rows, seed + 2)
    g = wl.bf16_normal(T, H, seed + 3)
    layer = GpuLayer(ep, E, K, H, T, A)
    R = layer.R
    h = layer.handle()
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    eo = torch.full((R, H), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    eo[:rows] = y.cuda()
    wd = torch.full((R,), float("nan"), dtype=torch.float32, device="cuda")
    wd[:rows] = w.cuda()
    res = torch.full((T, H), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    gexp = torch.full((R, H), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    gw = torch.full((R,), -7.0, dtype=torch.float32, device="cuda")
    ep.ep_prepare(h, idx.cuda(), counts, A)
    ep.ep_combine_weighted(h, eo, wd, res)
    ep.ep_combine_weighted_bwd(h, g.cuda(), eo, wd, gexp, gw)
    torch.cuda.synchronize()
    P = rt.P
    o_res = oracle_mod.combine_weighted(rt, bits(y), w.numpy())
    o_gexp, o_gw = oracle_mod.combine_bwd_weighted(rt, bits(g), w.numpy(), bits(y))
    assert np.array_equal(bits(res), o_res)
    gexp_b = bits(gexp)
    assert np.array_equal(gexp_b[:P], o_gexp)
    assert np.all(gexp_b[P:] == SENTINEL)
    gw_h = gw.cpu().numpy()
    assert np.all(gw_h[P:] == -7.0)
    pad = rt.inv < 0
    assert np.all(gw_h[:P][pad] == 0.0)
    # weight gradient within the float32 summation bound
    valid = np.nonzero(~pad)[0]
    if check_rows is not None and len(valid) > check_rows:
        valid = np.random.default_rng(seed).choice(valid, check_rows, replace=False)
    tok = rt.inv[valid] // K
    gf = g.double()[torch.from_numpy(tok)]
    yf = y.double()[torch.from_numpy(valid)]
    mag = (gf * yf).abs().sum(1).numpy()
    err = np.abs(gw_h[valid].astype(np.float64) - o_gw[valid])
    assert np.all(err <= (H - 1) * 2.0 ** -24 * mag + 1e-30), err.max()
    return rt


@pytest.mark.parametrize("name", ["tiny", "mixtral", "qwen3", "dsv3", "decode"])
def test_weighted_workloads(ep, oracle_mod, name):
    w = wl.WORKLOADS[name]
    idx, _ = wl.routing(w)
    run_weighted(ep, oracle_mod, idx, w.E, w.H, w.A, seed=6000 + w.number, check_rows=4096)


@pytest.mark.parametrize("case", [
    (7, 3, 5, 200, 3, 0.2),      # ragged row, A not a power of two
    (600, 32, 64, 24, 4, 0.1),   # largest top-k
    (900, 1, 1, 8, 1, 0.0),      # one expert, top-1, smallest row
    (300, 4, 12, 32, 8, 1.0),    # every route masked
])
def test_weighted_edges(ep, oracle_mod, case):
    T, K, E, H, A, p_mask = case
    idx, _ = wl.random_routing(T, K, E, seed=7000 + T, p_mask=p_mask)
    run_weighted(ep, oracle_mod, idx, E, H, A, seed=7100 + T)


def test_unit_weights_equal_combine(ep, oracle_mod):
    """With every weight 1.0 the weighted combine is ep_combine, bit for bit."""
    w = wl.WORKLOADS["qwen3"]
    T = 1024
    idx, _ = wl.routing(w, T=T)
    layer = GpuLayer(ep, w.E, w.K, w.H, T, w.A)
    h = layer.handle()
    counts = torch.empty(w.E, dtype=torch.int32, device="cuda")
    ep.ep_prepare(h, idx.cuda(), counts, w.A)
    eo = wl.bf16_normal(layer.R, w.H, 8001).cuda()
    ones = torch.ones(layer.R, dtype=torch.float32, device="cuda")
    a = torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda")
    b = torch.empty(T, w.H, dtype=torch.bfloat16, device="cuda")
    ep.ep_combine(h, eo, a)
    ep.ep_combine_weighted(h, eo, ones, b)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
