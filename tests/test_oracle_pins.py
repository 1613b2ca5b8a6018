"""Pins for the CPU oracle, against things other than the oracle itself.

Each test fixes part of the oracle by a source independent of its C loops:
hand-worked golden cases (tests/golden/), library routines (numpy bincount,
stable argsort, matrix products, torch's bf16 rounding), closed forms (the
identity round trip), adjoint identities and brute force on tiny inputs.

What they pin comes from TransformerEngine PR #3034, "Expert Parallelism:
common C API + NCCL EP backend", section "Per-step (allocation-free,
CUDA-graph capturable)" (prepare counts and alignment, dispatch, unweighted
combine, the two backward passes, zeroed padded slots of grad_expert_out),
and from the test list of TransformerEngine PR #3035, "[PyTorch] Expert
Parallelism: PyTorch wrapper + autograd ops with symm-mem zero-copy", section
"Testing" (prepare correctness, identity round trip, VJP).
"""
import itertools

import numpy as np
import pytest
import torch

from combine_ep_prepare_gb300 import workloads as wl
from golden_io import prepare_cases, rounding_cases

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


def as_f64(b: np.ndarray) -> np.ndarray:
    return from_bits(b).to(torch.float64).numpy()


# ----------------------------------------------------------------------------
# Golden, hand-worked cases
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("case", prepare_cases(), ids=lambda c: c["name"])
def test_prepare_golden(oracle_mod, case):
    idx = np.array(case["topk_idx"], np.int64).reshape(case["T"], case["K"])
    rt = oracle_mod.prepare(idx, case["E"], case["A"], case["R"])
    assert rt.token_counts.tolist() == case["counts"]
    assert rt.offsets.tolist() == case["offsets"]
    assert rt.P == case["P"]
    assert rt.slot.ravel().tolist() == case["slot"]
    assert rt.inv.tolist() == case["inv"]
    assert rt.status == case["status"]


@pytest.mark.parametrize("case", rounding_cases(), ids=lambda c: c[0])
def test_combine_rounding_golden(oracle_mod, case):
    name, K, rows, expected = case
    idx = np.arange(K, dtype=np.int64).reshape(1, K)
    rt = oracle_mod.prepare(idx, K, 1)
    expert_out = np.array(rows, np.uint16).reshape(K, 1)
    out = oracle_mod.combine(rt, expert_out)
    assert int(out[0, 0]) == expected, name
    # dispatch_bwd's token half is the same gather-sum
    gt, _ = oracle_mod.dispatch_bwd(rt, expert_out, None)
    assert int(gt[0, 0]) == expected, name


# ----------------------------------------------------------------------------
# bf16 conversions against torch's rounding (library routine)
# ----------------------------------------------------------------------------

def test_bf16_round_matches_torch(oracle_mod):
    g = torch.Generator().manual_seed(7)
    raw = torch.randint(-2**31, 2**31 - 1, (400_000,), generator=g, dtype=torch.int64)
    u = raw.to(torch.int32)
    special = torch.tensor([0, 0x80000000 - 2**32, 0x7F800000, 0xFF800000 - 2**32,
                            0x7F7FFFFF, 0x7F7F8000, 0x7F7F7FFF, 0x00000001, 0x00008000,
                            0x00018000, 0x3F808000, 0x3F818000, 0x3F807FFF, 0x3F800001,
                            0x00800000, 0x007FFFFF, 0x807FFFFF - 2**32], dtype=torch.int64).to(torch.int32)
    # every tie pattern around a range of kept halves
    ties = (torch.arange(0, 65536, 7, dtype=torch.int64) << 16 | 0x8000).to(torch.int32)
    u = torch.cat([u, special, ties])
    f = u.view(torch.float32)
    ours = oracle_mod.round_to_bf16(f.numpy())
    ref_t = f.to(torch.bfloat16)
    ref = bits(ref_t)
    nan = torch.isnan(f).numpy()
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN stays NaN (payload bits are not compared)
    ours_f = from_bits(ours[nan]).to(torch.float32)
    assert torch.isnan(ours_f).all()


def test_bf16_widen_is_exact(oracle_mod):
    for b in [0x0000, 0x8000, 0x3F80, 0xC2F7, 0x7F7F, 0x0001, 0x7F80, 0xFF80]:
        ref = from_bits(np.array([b], np.uint16)).to(torch.float32).item()
        assert oracle_mod.bf16_to_f32(b) == ref or (np.isnan(ref))


# ----------------------------------------------------------------------------
# Prepare: library routines and invariants
# ----------------------------------------------------------------------------

def _routings():
    yield "tiny", *wl.routing(wl.WORKLOADS["tiny"]), 8, 16
    w = wl.WORKLOADS["qwen3"]
    idx, wts = wl.routing(w, T=512)
    yield "qwen3_512", idx, wts, w.E, w.A
    w = wl.WORKLOADS["dsv3"]
    idx, wts = wl.routing(w, T=256)
    yield "dsv3_256", idx, wts, w.E, w.A
    w = wl.WORKLOADS["decode"]
    idx, wts = wl.routing(w)
    yield "decode", idx, wts, w.E, w.A
    idx, wts = wl.random_routing(300, 4, 13, seed=11, p_mask=0.2)
    yield "dups_masked", idx, wts, 13, 5
    idx, wts = wl.random_routing(200, 3, 6, seed=12, p_mask=0.1, p_bad=0.05)
    yield "bad", idx, wts, 6, 3


ROUTINGS = list(_routings())


@pytest.mark.parametrize("name,idx,wts,E,A", ROUTINGS, ids=[r[0] for r in ROUTINGS])
def test_prepare_against_library(oracle_mod, name, idx, wts, E, A):
    idx = idx.numpy()
    rt = oracle_mod.prepare(idx, E, A)
    flat = idx.ravel()
    valid = (flat >= 0) & (flat < E)
    # a1: counts are numpy's bincount of the valid routes
    assert np.array_equal(rt.token_counts, np.bincount(flat[valid], minlength=E))
    assert rt.token_counts.sum() == valid.sum()
    # status: BAD_INDEX exactly when some index lies outside [-1, E)
    bad = ((flat < -1) | (flat >= E)).any()
    assert bool(rt.status & oracle_mod.STATUS_BAD_INDEX) == bool(bad)
    # a2: each block is the count rounded up to the alignment, blocks are contiguous
    pe = np.diff(rt.offsets.astype(np.int64))
    assert rt.offsets[0] == 0
    assert np.all(pe % A == 0) and np.all(pe >= rt.token_counts)
    assert np.all(pe - rt.token_counts < A)
    assert np.all((rt.token_counts > 0) | (pe == 0))
    assert rt.P == rt.offsets[-1]
    # a3: slots agree with numpy's stable argsort of the expert ids:
    # routes of one expert keep their (t, k) order
    slot = rt.slot.ravel()
    assert np.all(slot[~valid] == -1)
    routes = np.nonzero(valid)[0]
    order = routes[np.argsort(flat[routes], kind="stable")]
    rank_in_expert = np.empty(len(order), np.int64)
    starts = np.searchsorted(flat[order], np.arange(E))
    for e in range(E):
        lo = starts[e]
        hi = starts[e + 1] if e + 1 < E else len(order)
        rank_in_expert[lo:hi] = np.arange(hi - lo)
    expect = rt.offsets[flat[order]].astype(np.int64) + rank_in_expert
    assert np.array_equal(slot[order], expect)
    # slots are a bijection from valid routes onto the non-padding rows
    inv = rt.inv
    assert len(inv) == rt.P
    assert np.array_equal(np.sort(slot[valid]), np.nonzero(inv >= 0)[0])
    assert np.all(inv[slot[valid]] == np.nonzero(valid)[0])
    assert (inv < 0).sum() == (pe - rt.token_counts).sum()


def test_prepare_brute_force_tiny(oracle_mod):
    """All routings of 2 tokens x 2 routes over 3 experts (values -1..2), A in {1,2,3}:
    slots equal the rank of the route among the routes of the same expert
    counted by brute force over all earlier routes."""
    E = 3
    for vals in itertools.product(range(-1, E), repeat=4):
        idx = np.array(vals, np.int64).reshape(2, 2)
        for A in (1, 2, 3):
            rt = oracle_mod.prepare(idx, E, A)
            flat = list(vals)
            counts = [sum(1 for v in flat if v == e) for e in range(E)]
            padded = [((c + A - 1) // A) * A for c in counts]
            starts = [sum(padded[:e]) for e in range(E)]
            for r, e in enumerate(flat):
                if e < 0:
                    assert rt.slot.ravel()[r] == -1
                else:
                    earlier = sum(1 for q in range(r) if flat[q] == e)
                    assert rt.slot.ravel()[r] == starts[e] + earlier
            assert rt.P == sum(padded)


def test_zero_tokens(oracle_mod):
    rt = oracle_mod.prepare(np.zeros((0, 4), np.int64), 5, 8)
    assert rt.P == 0 and rt.token_counts.sum() == 0 and rt.status == 0
    assert oracle_mod.combine(rt, np.zeros((0, 16), np.uint16)).shape == (0, 16)


def test_overflow_writes_nothing(oracle_mod):
    idx, _ = wl.random_routing(50, 2, 4, seed=3)
    rt = oracle_mod.prepare(idx.numpy(), 4, 8, recv_capacity=10)
    assert rt.status & oracle_mod.STATUS_OVERFLOW
    assert oracle_mod.dispatch(rt, np.zeros((50, 8), np.uint16), np.zeros((50, 2), np.float32)) == (None, None)
    assert oracle_mod.combine(rt, np.zeros((200, 8), np.uint16)) is None
    rt2 = oracle_mod.prepare(idx.numpy(), 4, 8, recv_capacity=rt.P)
    assert rt2.status == 0


# ----------------------------------------------------------------------------
# Row operations: closed forms, adjoints, library products
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("name,idx,wts,E,A", ROUTINGS, ids=[r[0] for r in ROUTINGS])
def test_identity_round_trip(oracle_mod, name, idx, wts, E, A):
    """combine(dispatch(x))[t] = bf16(n_valid(t) * x[t]) exactly: n_valid <= 8
    equal bf16 terms sum exactly in binary32, then round once.  A token with
    no valid route gives +0 (the sum starts at +0), hence the "+ 0.0"."""
    T, K = idx.shape
    x = wl.bf16_normal(T, 40, seed=5)
    rt = oracle_mod.prepare(idx.numpy(), E, A)
    recv, recv_w = oracle_mod.dispatch(rt, bits(x), wts.numpy())
    y = oracle_mod.combine(rt, recv)
    flat = idx.numpy()
    n_valid = ((flat >= 0) & (flat < E)).sum(1)
    expect = (x.to(torch.float32) * torch.from_numpy(n_valid).to(torch.float32)[:, None] + 0.0).to(torch.bfloat16)
    assert np.array_equal(y, bits(expect))
    # weights land at their route's slot; padding weights are zero
    slot = rt.slot.ravel()
    ok = slot >= 0
    assert np.array_equal(recv_w[slot[ok]], wts.numpy().ravel()[ok])
    assert np.all(recv_w[rt.inv < 0] == 0)
    assert np.all(recv[rt.inv < 0] == 0)


@pytest.mark.parametrize("name,idx,wts,E,A", ROUTINGS, ids=[r[0] for r in ROUTINGS])
def test_scaled_dispatch_then_combine_matches_fp64(oracle_mod, name, idx, wts, E, A):
    """The MoE use: expert_out = recv_tokens * recv_topk_weights (bf16), then
    combine.  Compared with the fp64 textbook sum_k w_k x_t: two bf16
    roundings (per term and at the end) bound the error."""
    T, K = idx.shape
    x = wl.bf16_normal(T, 24, seed=6)
    rt = oracle_mod.prepare(idx.numpy(), E, A)
    recv, recv_w = oracle_mod.dispatch(rt, bits(x), wts.numpy())
    eo = (from_bits(recv).to(torch.float32) * torch.from_numpy(recv_w)[:, None]).to(torch.bfloat16)
    y = as_f64(oracle_mod.combine(rt, bits(eo)))
    flat = idx.numpy()
    valid = ((flat >= 0) & (flat < E)).astype(np.float64)
    w64 = wts.numpy().astype(np.float64) * valid
    x64 = x.to(torch.float64).numpy()
    exact = (w64.sum(1))[:, None] * x64
    mag = (np.abs(w64).sum(1))[:, None] * np.abs(x64)
    assert np.all(np.abs(y - exact) <= 2.0 ** -8 * mag + 2.0 ** -8 * np.abs(exact) + 1e-30)


def _dense_S(rt, idx, E):
    """0/1 matrix S [P, T]: S[s, t] = 1 when receive row s holds token t,
    built from numpy's stable sort of the routes by expert (not from the
    oracle's slot map)."""
    flat = idx.ravel()
    T, K = idx.shape
    valid = (flat >= 0) & (flat < E)
    S = np.zeros((rt.P, T))
    for e in range(E):
        routes = np.nonzero(valid & (flat == e))[0]  # ascending (t, k)
        for j, r in enumerate(routes):
            S[rt.offsets[e] + j, r // K] = 1.0
    return S


@pytest.mark.parametrize("name,idx,wts,E,A", ROUTINGS[:5], ids=[r[0] for r in ROUTINGS[:5]])
def test_dense_routing_matrix(oracle_mod, name, idx, wts, E, A):
    """dispatch = S x and combine = S^T y (matrix products, on small integers
    so that every sum is exact)."""
    idx = idx.numpy()
    T, K = idx.shape
    rt = oracle_mod.prepare(idx, E, A)
    S = _dense_S(rt, idx, E)
    x = wl.small_int_bf16(T, 16, seed=21)
    recv, _ = oracle_mod.dispatch(rt, bits(x), np.zeros((T, K), np.float32))
    assert np.array_equal(as_f64(recv), S @ x.to(torch.float64).numpy())
    y = wl.small_int_bf16(rt.P, 16, seed=22)
    out = oracle_mod.combine(rt, bits(y))
    assert np.array_equal(as_f64(out), S.T @ y.to(torch.float64).numpy())
    # combine_bwd is the transpose of combine: S g
    g = wl.small_int_bf16(T, 16, seed=23)
    gb = oracle_mod.combine_bwd(rt, bits(g))
    assert np.array_equal(as_f64(gb), S @ g.to(torch.float64).numpy())
    # dispatch_bwd's token half is the transpose of dispatch: S^T G
    G = wl.small_int_bf16(rt.P, 16, seed=24)
    gt, _ = oracle_mod.dispatch_bwd(rt, bits(G), None)
    assert np.array_equal(as_f64(gt), S.T @ G.to(torch.float64).numpy())


@pytest.mark.parametrize("name,idx,wts,E,A", ROUTINGS, ids=[r[0] for r in ROUTINGS])
def test_adjoint_identities(oracle_mod, name, idx, wts, E, A):
    """<combine(y), g> = <y, combine_bwd(g)> and <dispatch(x), G> =
    <x, dispatch_bwd(G)>, including the weight half, on small integers
    (all products and sums exact in fp64)."""
    idx = idx.numpy()
    T, K = idx.shape
    rt = oracle_mod.prepare(idx, E, A)
    H = 12
    y = wl.small_int_bf16(rt.P, H, seed=31)
    g = wl.small_int_bf16(T, H, seed=32)
    lhs = (as_f64(oracle_mod.combine(rt, bits(y))) * g.double().numpy()).sum()
    rhs = (y.double().numpy() * as_f64(oracle_mod.combine_bwd(rt, bits(g)))).sum()
    assert lhs == rhs
    x = wl.small_int_bf16(T, H, seed=33)
    w = np.random.default_rng(34).integers(-3, 4, (T, K)).astype(np.float32)
    G = wl.small_int_bf16(rt.P, H, seed=35)
    Gw = np.random.default_rng(36).integers(-3, 4, rt.P).astype(np.float32)
    recv, recv_w = oracle_mod.dispatch(rt, bits(x), w)
    gt, gw = oracle_mod.dispatch_bwd(rt, bits(G), Gw)
    assert (as_f64(recv) * G.double().numpy()).sum() == (x.double().numpy() * as_f64(gt)).sum()
    assert (recv_w.astype(np.float64) * Gw).sum() == (w.astype(np.float64) * gw).sum()
    # a missing weight gradient gives zeros
    _, gw0 = oracle_mod.dispatch_bwd(rt, bits(G), None)
    assert np.all(gw0 == 0)


@pytest.mark.parametrize("name,idx,wts,E,A", ROUTINGS, ids=[r[0] for r in ROUTINGS])
def test_weight_gradient_gather(oracle_mod, name, idx, wts, E, A):
    """Weight half of dispatch_bwd: route (t,k) takes the receive row's weight
    gradient (numpy fancy indexing, bit for bit); a masked or invalid route,
    and every route when no weight gradient is given, gets +0.0 (all bits
    zero, the value of a zero-filled buffer)."""
    idx = idx.numpy()
    rt = oracle_mod.prepare(idx, E, A)
    P = max(rt.P, 1)
    G = wl.bf16_normal(P, 4, seed=37)
    Gw = wl.f32_normal(P, seed=38).numpy()
    _, gw = oracle_mod.dispatch_bwd(rt, bits(G), Gw)
    ok = rt.slot >= 0
    assert np.array_equal(gw[ok].view(np.uint32), Gw[rt.slot[ok]].view(np.uint32))
    assert np.all(gw[~ok].view(np.uint32) == 0)
    _, gw0 = oracle_mod.dispatch_bwd(rt, bits(G), None)
    assert np.all(gw0.view(np.uint32) == 0)


def test_padding_rows_zero(oracle_mod):
    idx, _ = wl.random_routing(100, 3, 7, seed=41, p_mask=0.1)
    rt = oracle_mod.prepare(idx.numpy(), 7, 16)
    g = wl.bf16_normal(100, 32, seed=42)
    gb = oracle_mod.combine_bwd(rt, bits(g))
    pad = rt.inv < 0
    assert pad.sum() > 0
    assert np.all(gb[pad] == 0)
    assert np.array_equal(gb[~pad], bits(g)[rt.inv[~pad] // 3])


def test_masked_equals_extra_discarded_expert(oracle_mod):
    """A masked route behaves like a route to an extra expert E whose output
    is discarded: counts, offsets and slots of experts 0..E-1 agree, and
    combine agrees when that extra expert's rows are zero."""
    w = wl.WORKLOADS["decode"]
    idx, _ = wl.routing(w)
    idx = idx.numpy()
    E = w.E
    rt = oracle_mod.prepare(idx, E, 4)
    idx2 = np.where(idx < 0, E, idx)
    rt2 = oracle_mod.prepare(idx2, E + 1, 4)
    assert (idx < 0).sum() > 0
    assert np.array_equal(rt.token_counts, rt2.token_counts[:E])
    assert np.array_equal(rt.offsets, rt2.offsets[:E + 1])
    m = idx.ravel() >= 0
    assert np.array_equal(rt.slot.ravel()[m], rt2.slot.ravel()[m])
    y = wl.bf16_normal(rt2.P, 64, seed=51)
    yz = bits(y).copy()
    yz[rt.P:] = 0
    assert np.array_equal(oracle_mod.combine(rt, yz[: rt.P]), oracle_mod.combine(rt2, yz))


def test_repeat_calls_bit_identical(oracle_mod):
    w = wl.WORKLOADS["tiny"]
    idx, wts = wl.routing(w)
    x = bits(wl.tokens(w))
    a = oracle_mod.prepare(idx.numpy(), w.E, w.A)
    b = oracle_mod.prepare(idx.numpy(), w.E, w.A)
    assert np.array_equal(a.slot, b.slot) and np.array_equal(a.inv, b.inv)
    r1 = oracle_mod.dispatch(a, x, wts.numpy())[0]
    r2 = oracle_mod.dispatch(b, x, wts.numpy())[0]
    assert np.array_equal(r1, r2)


# ----------------------------------------------------------------------------
# Weighted combine (fused weight multiply) and its backward
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("name,idx,wts,E,A", ROUTINGS, ids=[r[0] for r in ROUTINGS])
def test_weighted_combine_unit_weights_is_combine(oracle_mod, name, idx, wts, E, A):
    """With every weight 1.0 the weighted combine is the unweighted one, bit for bit."""
    T, K = idx.shape
    rt = oracle_mod.prepare(idx.numpy(), E, A)
    y = bits(wl.bf16_normal(max(rt.P, 1), 24, seed=61))
    ones = np.ones(max(rt.P, 1), np.float32)
    assert np.array_equal(oracle_mod.combine_weighted(rt, y, ones), oracle_mod.combine(rt, y))


@pytest.mark.parametrize("name,idx,wts,E,A", ROUTINGS, ids=[r[0] for r in ROUTINGS])
def test_weighted_combine_matches_fp64(oracle_mod, name, idx, wts, E, A):
    """Against the fp64 textbook sum_k w_k y_k: float32 products and sums (K of
    each) plus one bf16 rounding bound the error."""
    rt = oracle_mod.prepare(idx.numpy(), E, A)
    P = max(rt.P, 1)
    y = wl.bf16_normal(P, 24, seed=62)
    w = wl.f32_normal(P, seed=63)
    out = as_f64(oracle_mod.combine_weighted(rt, bits(y), w.numpy()))
    slot = rt.slot
    T, K = slot.shape
    y64 = y.double().numpy()
    w64 = w.double().numpy()
    exact = np.zeros((T, 24))
    mag = np.zeros((T, 24))
    for k in range(K):
        s = slot[:, k]
        ok = s >= 0
        term = np.where(ok[:, None], w64[np.maximum(s, 0)][:, None] * y64[np.maximum(s, 0)], 0.0)
        exact += term
        mag += np.abs(term)
    assert np.all(np.abs(out - exact) <= 2.0 ** -8 * np.abs(exact) + 2.0 ** -21 * K * mag + 1e-30)


def test_weighted_golden(oracle_mod):
    """Hand-worked: one token, K=2, H=1, A=1 (rows 0 and 1)."""
    idx = np.array([[0, 1]], np.int64)
    rt = oracle_mod.prepare(idx, 2, 1)
    cases = [
        # rows (bf16 bits), weights, expected (bf16 bits)
        ([0x3F80, 0x4000], [0.5, 0.25], 0x3F80),    # 0.5*1 + 0.25*2 = 1
        ([0x3FC0, 0x4090], [3.0, -1.0], 0x0000),    # 3*1.5 - 4.5 = +0
        ([0x3F80, 0x3F80], [1.0, 2.0 ** -8], 0x3F80),  # 1 + 2^-8: tie, to even
        ([0x3F80, 0x3F80], [1.0, 3 * 2.0 ** -8], 0x3F82),  # 1 + 3*2^-8: tie, to even
    ]
    for rows, w, expected in cases:
        out = oracle_mod.combine_weighted(rt, np.array(rows, np.uint16).reshape(2, 1),
                                          np.array(w, np.float32))
        assert int(out[0, 0]) == expected, (rows, w)


def test_weighted_not_fused_golden(oracle_mod):
    """Hand-worked: the product is rounded to float32 before it is added.
    y1 = 3*2^-10 (bf16 0x3B40), w1 = 11184982 * 2^-23 (float32 0x3FAAAB56):
    w1*y1 = 33554946 * 2^-33 = 2^-8 + 2^-24 + 2^-32 exactly, a float32 tie that
    goes to the even 2^-8 + 2^-24.  Then 1 + (2^-8 + 2^-24) is again a tie and
    goes to 1 + 2^-8, a bf16 tie that goes to the even 1.0 (0x3F80).  A fused
    multiply-add would keep the 2^-32 and end at 1 + 2^-7 (0x3F81)."""
    idx = np.array([[0, 1]], np.int64)
    rt = oracle_mod.prepare(idx, 2, 1)
    w = np.array([0x3F800000, 0x3FAAAB56], np.uint32).view(np.float32)
    assert float(w[1]) * 3 * 2.0 ** -10 == 2.0 ** -8 + 2.0 ** -24 + 2.0 ** -32
    out = oracle_mod.combine_weighted(rt, np.array([[0x3F80], [0x3B40]], np.uint16), w)
    assert int(out[0, 0]) == 0x3F80


@pytest.mark.parametrize("case", rounding_cases(), ids=lambda c: c[0])
def test_weighted_unit_weights_rounding_golden(oracle_mod, case):
    """With weights 1.0 every product is exact, so the hand-worked combine
    cases (summation order, ties, signed zeros, overflow) hold for the
    weighted combine too."""
    name, K, rows, expected = case
    idx = np.arange(K, dtype=np.int64).reshape(1, K)
    rt = oracle_mod.prepare(idx, K, 1)
    out = oracle_mod.combine_weighted(rt, np.array(rows, np.uint16).reshape(K, 1), np.ones(K, np.float32))
    assert int(out[0, 0]) == expected, name


@pytest.mark.parametrize("name,idx,wts,E,A", ROUTINGS[:5], ids=[r[0] for r in ROUTINGS[:5]])
def test_weighted_adjoint_and_weight_gradient(oracle_mod, name, idx, wts, E, A):
    """On small integers and small integer weights (all exact):
    <combine_w(y), g> = <y, combine_bwd_w(g)>, and the weight gradient equals
    the change of <combine_w(y), g> when one receive row's weight grows by 1."""
    idx = idx.numpy()
    rt = oracle_mod.prepare(idx, E, A)
    T, K = idx.shape
    P = max(rt.P, 1)
    H = 6
    y = wl.small_int_bf16(P, H, seed=71)
    g = wl.small_int_bf16(T, H, seed=72)
    w = np.random.default_rng(73).integers(-2, 3, P).astype(np.float32)
    fwd = as_f64(oracle_mod.combine_weighted(rt, bits(y), w))
    gexp, gw = oracle_mod.combine_bwd_weighted(rt, bits(g), w, bits(y))
    lhs = (fwd * g.double().numpy()).sum()
    rhs = (y.double().numpy()[: rt.P] * as_f64(gexp)).sum()
    assert lhs == rhs
    for s in range(0, rt.P, max(1, rt.P // 7)):
        w2 = w.copy()
        w2[s] += 1.0
        lhs2 = (as_f64(oracle_mod.combine_weighted(rt, bits(y), w2)) * g.double().numpy()).sum()
        assert lhs2 - lhs == gw[s]
    pad = rt.inv < 0
    assert np.all(gexp[pad] == 0) and np.all(gw[pad] == 0)


def test_weighted_bwd_products_round_once(oracle_mod):
    """grad_expert_out = bf16(float32(w * g)): against torch's float32 multiply
    and bf16 rounding (library routines)."""
    idx, _ = wl.random_routing(50, 3, 5, seed=81, p_mask=0.1)
    rt = oracle_mod.prepare(idx.numpy(), 5, 4)
    g = wl.bf16_normal(50, 16, seed=82)
    w = wl.f32_normal(rt.P, seed=83)
    y = wl.bf16_normal(rt.P, 16, seed=84)
    gexp, gw = oracle_mod.combine_bwd_weighted(rt, bits(g), w.numpy(), bits(y))
    ok = rt.inv >= 0
    t = rt.inv[ok] // 3
    expect = (w[torch.from_numpy(np.nonzero(ok)[0])][:, None] * g.float()[torch.from_numpy(t)]).to(torch.bfloat16)
    assert np.array_equal(gexp[ok], bits(expect))
    dots = (g.double()[torch.from_numpy(t)] * y.double()[torch.from_numpy(np.nonzero(ok)[0])]).sum(1).numpy()
    assert np.allclose(gw[ok], dots, rtol=0, atol=1e-9)
