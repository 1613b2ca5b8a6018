"""GPU parity for FP16 and FP32 payloads (layers registered with
EP_DTYPE_FP16 / EP_DTYPE_FP32): every output of the five calls and of the
weighted combine, bit for bit against the oracle; the weighted combine's
weight gradient within its float32 summation bound (exact products for fp16,
one rounding per product for fp32).

TransformerEngine PR #3034's C++ tests cover BF16, FP16 and FP32 payloads.
"""
import numpy as np
import pytest
import torch

from combine_ep_prepare_gb300 import workloads as wl
from ep_harness import (GpuLayer, assert_step_equal, bits, custom_inputs, gpu_step,
                        oracle_step, same, sentinel_tensor, untouched)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_ep_prepare_gb300 as ep
    return ep


CASES = [
    # name, T, K, E, H, A, p_mask, distinct
    ("tiny", 64, 2, 8, 128, 16, 0.0, True),
    ("qwen3_like", 1024, 8, 128, 2048, 128, 0.0, True),
    ("dsv3_like", 512, 8, 256, 7168, 128, 0.0, True),
    ("masked", 128, 8, 256, 7168, 1, 0.5, True),
    ("ragged_row", 37, 3, 5, 200, 3, 0.2, False),
    ("large_chunked", 9000, 4, 37, 24, 5, 0.1, False),
]


@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_step_parity(ep, oracle_mod, dtype, case):
    name, T, K, E, H, A, p_mask, distinct = case
    idx, wts = wl.random_routing(T, K, E, seed=8100 + T, p_mask=p_mask, distinct=distinct)
    inp = custom_inputs(idx, wts, E, H, A, oracle_mod, seed=8200 + T, dtype=dtype)
    layer = GpuLayer(ep, E, K, H, T, A, dtype=dtype)
    g = gpu_step(ep, layer, inp)
    o = oracle_step(inp, oracle_mod, layer.R)
    assert_step_equal(g, o, layer.R)


@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
@pytest.mark.parametrize("case", CASES[:5], ids=[c[0] for c in CASES[:5]])
def test_weighted_parity(ep, oracle_mod, dtype, case):
    name, T, K, E, H, A, p_mask, distinct = case
    idx, _ = wl.random_routing(T, K, E, seed=8300 + T, p_mask=p_mask, distinct=distinct)
    rt = oracle_mod.prepare(idx.numpy(), E, A)
    rows = max(rt.P, 1)
    y = wl.payload_normal(rows, H, 8400 + T, dtype)
    gr = wl.payload_normal(T, H, 8500 + T, dtype)
    w = wl.f32_normal(rows, 8600 + T)
    layer = GpuLayer(ep, E, K, H, T, A, dtype=dtype)
    R = layer.R
    h = layer.handle()
    eo = sentinel_tensor((R, H), dtype, "cuda")
    eo[:rows] = y.cuda()
    wd = torch.zeros(R, dtype=torch.float32, device="cuda")
    wd[:rows] = w.cuda()
    res = sentinel_tensor((T, H), dtype, "cuda")
    gexp = sentinel_tensor((R, H), dtype, "cuda")
    gw = torch.full((R,), -7.0, dtype=torch.float32, device="cuda")
    ep.ep_prepare(h, idx.cuda(), torch.empty(E, dtype=torch.int32, device="cuda"), A)
    ep.ep_combine_weighted(h, eo, wd, res)
    ep.ep_combine_weighted_bwd(h, gr.cuda(), eo, wd, gexp, gw)
    torch.cuda.synchronize()
    P = rt.P
    o_res = oracle_mod.combine_weighted(rt, bits(y), w.numpy(), dtype)
    o_gexp, o_gw = oracle_mod.combine_bwd_weighted(rt, bits(gr), w.numpy(), bits(y), dtype)
    assert same(bits(res), o_res)
    gb = bits(gexp)
    assert same(gb[:P], o_gexp) and untouched(gb[P:])
    gwh = gw.cpu().numpy()
    pad = rt.inv < 0
    assert np.all(gwh[:P][pad] == 0) and np.all(gwh[P:] == -7.0)
    valid = np.nonzero(~pad)[0]
    tok = rt.inv[valid] // K
    mag = (gr.double()[torch.from_numpy(tok)] * y.double()[torch.from_numpy(valid)]).abs().sum(1).numpy()
    bound = (H + (1 if dtype == "fp32" else -1)) * 2.0 ** -24 * mag + 1e-30
    assert np.all(np.abs(gwh[valid].astype(np.float64) - o_gw[valid]) <= bound)


def test_payload_dtype_checked_by_binding(ep):
    lid, size = ep.ep_register_layer(4, 2, 16, 8, 2, dtype="fp16")
    h = ep.alloc_handle(lid, size)
    bad = torch.zeros(8, 16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(TypeError):
        ep.ep_combine(h, torch.zeros(ep.ep_recv_capacity(lid), 16, dtype=torch.float16, device="cuda"), bad)
