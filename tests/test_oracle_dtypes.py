"""Pins for the oracle's FP16 and FP32 payload paths.

TransformerEngine PR #3034 ("Expert Parallelism: common C API + NCCL EP
backend", Greptile summary of tests/cpp_distributed/test_ep.cu) covers BF16,
FP16 and FP32 payloads; the sums accumulate in float32, in k order from +0.0f,
and round once to the payload type (FP32: the float32 sum itself).

Pinned by: binary16 conversions against torch's (library routine) on every
bit pattern and on random floats with all tie patterns; hand-worked FP16
sums (overflow, ties, subnormals); the dense 0/1 routing matrix and adjoint
identities on small integers (exact in every type); FP32 combine against the
fp64 sum within K float32 roundings; the FP16 identity round trip.
"""
import numpy as np
import pytest
import torch

from combine_ep_prepare_gb300 import workloads as wl


def f16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_f16_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.float16)


def rows_of(t: torch.Tensor, dtype: str) -> np.ndarray:
    if dtype == "fp32":
        return t.to(torch.float32).numpy()
    if dtype == "fp16":
        return f16_bits(t.to(torch.float16))
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def as_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "fp32":
        return a.astype(np.float64)
    if dtype == "fp16":
        return from_f16_bits(a).to(torch.float64).numpy()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def test_f16_widening_every_pattern(oracle_mod):
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = from_f16_bits(allb).to(torch.float32).numpy()
    ours = np.array([oracle_mod.f16_to_f32(int(b)) for b in allb], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f16_rounding_matches_torch(oracle_mod):
    g = torch.Generator().manual_seed(17)
    raw = torch.randint(-2**31, 2**31 - 1, (300_000,), generator=g, dtype=torch.int64).to(torch.int32)
    # values around the binary16 range, including subnormals and overflow
    near = (torch.randn(200_000, generator=g) * torch.exp2(torch.randint(-30, 18, (200_000,), generator=g).float()))
    # every tie: binary32 values halfway between neighbouring halves
    halves = torch.arange(0, 0x7C00, 3, dtype=torch.int32).to(torch.int16).view(torch.float16).float()
    nxt = (torch.arange(0, 0x7C00, 3, dtype=torch.int32) + 1).to(torch.int16).view(torch.float16).float()
    ties = ((halves.double() + nxt.double()) / 2).float()
    f = torch.cat([raw.view(torch.float32), near, ties, -ties])
    ours = oracle_mod.round_to_f16(f.numpy())
    ref = f16_bits(f.to(torch.float16))
    nan = torch.isnan(f).numpy()
    assert np.array_equal(ours[~nan], ref[~nan])
    assert torch.isnan(from_f16_bits(ours[nan]).float()).all()


def test_f16_boundaries_match_torch(oracle_mod):
    """The edges of binary16 rounding against torch's conversion (a library
    routine): the largest finite value and the overflow tie at 65520, the
    smallest normal 2^-14, the subnormal grid 2^-24 with its ties, and the
    flush to zero at and below 2^-25."""
    u = 2.0 ** -24
    vals = [65504.0, 65505.0, 65519.0, np.nextafter(np.float32(65520), np.float32(0)), 65520.0,
            65535.0, 65536.0, 1e6, 2.0 ** -14, np.nextafter(np.float32(2.0 ** -14), np.float32(0)),
            2.0 ** -14 - 0.5 * u, u, 0.5 * u, np.nextafter(np.float32(0.5 * u), np.float32(1)),
            0.25 * u, 1.5 * u, 2.5 * u, 3.5 * u, 1023.5 * u, 1022.5 * u, 0.0]
    f = torch.tensor(vals, dtype=torch.float32)
    f = torch.cat([f, -f])
    assert np.array_equal(oracle_mod.round_to_f16(f.numpy()), f16_bits(f.to(torch.float16)))


@pytest.mark.parametrize("name,rows,expected", [
    ("overflow_to_inf", [0x7BFF, 0x7BFF], 0x7C00),       # 65504 + 65504
    ("tie_down", [0x3C00, 0x1000], 0x3C00),              # 1 + 2^-11: tie, to even 1
    ("tie_up", [0x3C00, 0x1600], 0x3C02),                # 1 + 3*2^-11: tie, to even 1 + 2^-9
    ("subnormals_add", [0x0001, 0x0001], 0x0002),        # 2^-24 + 2^-24
    ("cancel", [0x4200, 0xC200], 0x0000),                # 3 - 3 = +0
    ("neg_zeros", [0x8000, 0x8000], 0x0000),             # +0 + -0 + -0
])
def test_f16_combine_golden(oracle_mod, name, rows, expected):
    idx = np.array([[0, 1]], np.int64)
    rt = oracle_mod.prepare(idx, 2, 1)
    out = oracle_mod.combine(rt, np.array(rows, np.uint16).reshape(2, 1), "fp16")
    assert int(out[0, 0]) == expected, name


ROUTINGS = [
    ("uniform", *wl.random_routing(120, 2, 6, seed=301, distinct=True), 6, 4),
    ("masked_dups", *wl.random_routing(90, 4, 9, seed=302, p_mask=0.25), 9, 3),
]


@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
@pytest.mark.parametrize("name,idx,wts,E,A", ROUTINGS, ids=[r[0] for r in ROUTINGS])
def test_dense_matrix_and_adjoints(oracle_mod, dtype, name, idx, wts, E, A):
    idx = idx.numpy()
    T, K = idx.shape
    rt = oracle_mod.prepare(idx, E, A)
    flat = idx.ravel()
    S = np.zeros((rt.P, T))
    for e in range(E):
        for j, r in enumerate(np.nonzero(flat == e)[0]):
            S[rt.offsets[e] + j, r // K] = 1.0
    H = 10
    x = wl.small_int_bf16(T, H, seed=311).float()
    y = wl.small_int_bf16(rt.P, H, seed=312).float()
    g = wl.small_int_bf16(T, H, seed=313).float()
    G = wl.small_int_bf16(rt.P, H, seed=314).float()
    recv, recv_w = oracle_mod.dispatch(rt, rows_of(x, dtype), wts.numpy(), dtype)
    assert np.array_equal(as_f64(recv, dtype), S @ x.double().numpy())
    out = oracle_mod.combine(rt, rows_of(y, dtype), dtype)
    assert np.array_equal(as_f64(out, dtype), S.T @ y.double().numpy())
    gb = oracle_mod.combine_bwd(rt, rows_of(g, dtype), dtype)
    assert np.array_equal(as_f64(gb, dtype), S @ g.double().numpy())
    gt, _ = oracle_mod.dispatch_bwd(rt, rows_of(G, dtype), None, dtype)
    assert np.array_equal(as_f64(gt, dtype), S.T @ G.double().numpy())
    # weighted, small integer weights: exact, and adjoint to its backward
    w = np.random.default_rng(315).integers(-2, 3, rt.P).astype(np.float32)
    fw = as_f64(oracle_mod.combine_weighted(rt, rows_of(y, dtype), w, dtype), dtype)
    assert np.array_equal(fw, S.T @ (w[:, None].astype(np.float64) * y.double().numpy()))
    gexp, gw = oracle_mod.combine_bwd_weighted(rt, rows_of(g, dtype), w, rows_of(y, dtype), dtype)
    assert (fw * g.double().numpy()).sum() == (y.double().numpy() * as_f64(gexp, dtype)).sum()
    assert np.array_equal(gw, ((S @ g.double().numpy()) * y.double().numpy()).sum(1))


def test_fp32_combine_within_rounding(oracle_mod):
    idx, _ = wl.random_routing(200, 8, 16, seed=321, p_mask=0.1)
    rt = oracle_mod.prepare(idx.numpy(), 16, 4)
    y = (torch.randn(rt.P, 24, generator=torch.Generator().manual_seed(322)) * 100).numpy()
    out = oracle_mod.combine(rt, y, "fp32").astype(np.float64)
    slot = rt.slot
    exact = np.zeros((200, 24))
    mag = np.zeros((200, 24))
    for k in range(8):
        ok = slot[:, k] >= 0
        term = np.where(ok[:, None], y[np.maximum(slot[:, k], 0)].astype(np.float64), 0.0)
        exact += term
        mag += np.abs(term)
    assert np.all(np.abs(out - exact) <= 8 * 2.0 ** -24 * mag)


def test_fp16_identity_round_trip(oracle_mod):
    idx, wts = wl.random_routing(150, 4, 7, seed=331, p_mask=0.2)
    rt = oracle_mod.prepare(idx.numpy(), 7, 8)
    x = torch.randn(150, 32, generator=torch.Generator().manual_seed(332)).to(torch.float16)
    recv, _ = oracle_mod.dispatch(rt, f16_bits(x), wts.numpy(), "fp16")
    y = oracle_mod.combine(rt, recv, "fp16")
    n = ((idx.numpy() >= 0).sum(1)).astype(np.float32)
    expect = (x.float() * torch.from_numpy(n)[:, None] + 0.0).to(torch.float16)
    assert np.array_equal(y, f16_bits(expect))
