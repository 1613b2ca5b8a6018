"""Pins of the sharded oracle (expert parallelism over N ranks), CPU only.

The sharded functions of oracle/ep_oracle.c follow TransformerEngine PR #3035,
"Sequence Diagram" (prepare all-gathers the routing table; dispatch pushes
token rows to the owners of the chosen experts; combine pulls the expert rows
back; the backward pass runs the reverse scatter and the reverse gather), with
rank q owning experts [q*E/N, (q+1)*E/N).  They are pinned by
  - hand-worked cases (tests/golden/shard_hand_worked.txt);
  - the partition identity: stacking the owners' receive buffers in rank
    order gives the single-buffer receive buffer of the concatenated batch,
    and every rank's token-side outputs are the matching slice of the
    single-buffer outputs, bit for bit (the single-buffer oracle is pinned
    independently in test_oracle_pins.py);
  - invariants: per owner, the slots are a bijection onto [0, P_q) minus the
    padding rows, each block lists its routes in (rank, t, k) order, every
    block is a multiple of A long; bad indices flag their own rank only;
    overflow of any owner flags every rank.
"""
import numpy as np
import pytest

import golden_io
import oracle
from combine_ep_prepare_gb300 import workloads as wl


@pytest.mark.parametrize("case", golden_io.shard_cases(), ids=lambda c: c["name"])
def test_shard_golden(case, oracle_mod=oracle):
    N, K = case["N"], case["K"]
    idx = [np.array(case["idx%d" % r], np.int64).reshape(-1, K) for r in range(N)]
    sr = oracle_mod.shard_prepare(idx, case["E"], case["A"], N, case["R"])
    assert sr.counts.tolist() == case["counts"]
    assert sr.offsets[:case["E"]].tolist() == case["offsets"]
    assert sr.P.tolist() == case["P"]
    for r in range(N):
        assert sr.slot[r].reshape(-1).tolist() == case["slot%d" % r]
        assert sr.dest[r].reshape(-1).tolist() == case["dest%d" % r]
    for q in range(N):
        assert sr.inv[q].tolist() == case["inv%d" % q]
    assert sr.status.tolist() == case["status"]


def _ranks(N, K, E, seed, p_mask=0.0, p_bad=0.0, tmax=40):
    g = np.random.default_rng(seed)
    out = []
    for r in range(N):
        T = int(g.integers(0, tmax + 1)) if r % 3 != 2 else 0 if seed % 2 else int(g.integers(1, tmax))
        idx, _ = wl.random_routing(T, K, E, seed=seed * 31 + r, p_mask=p_mask, p_bad=p_bad)
        out.append(idx.numpy())
    return out


def _rows(n, H, seed):
    return wl.bf16_normal(max(n, 1), H, seed).view(__import__("torch").int16).numpy().view(np.uint16)[:n]


CONFIGS = [(2, 2, 4, 2, 1), (2, 3, 8, 4, 2), (4, 4, 8, 3, 3), (4, 1, 4, 1, 4), (8, 8, 16, 5, 5),
           (3, 2, 6, 7, 6), (2, 6, 2, 2, 7)]


@pytest.mark.parametrize("N,K,E,A,seed", CONFIGS)
def test_shard_reassembles_the_single_buffer_step(N, K, E, A, seed, oracle_mod=oracle):
    idx = _ranks(N, K, E, seed, p_mask=0.2, p_bad=0.05)
    cat = np.concatenate([a.reshape(-1, K) for a in idx])
    T = cat.shape[0]
    single = oracle_mod.prepare(cat, E, A)
    sr = oracle_mod.shard_prepare(idx, E, A, N)
    el = E // N
    base = [int(single.offsets[q * el]) for q in range(N)]
    # map: counts, offsets, P, slots, owners, inverse
    assert np.array_equal(sr.counts, single.token_counts)
    for q in range(N):
        assert sr.P[q] == single.offsets[(q + 1) * el] - base[q]
        assert np.array_equal(sr.offsets[q * el:(q + 1) * el], single.offsets[q * el:(q + 1) * el] - base[q])
        assert np.array_equal(sr.inv[q], single.inv[base[q]:base[q] + sr.P[q]])
    s_slot, s_dest = sr._cat(sr.slot), sr._cat(sr.dest)
    valid = single.slot >= 0
    owner = np.where(valid, np.clip(cat, 0, E - 1) // el, -1)
    assert np.array_equal(s_dest, owner)
    assert np.array_equal(s_slot[valid], single.slot[valid] - np.array(base)[owner[valid]])
    assert np.all(s_slot[~valid] == -1)
    bad = [bool(((a < -1) | (a >= E)).any()) for a in idx]
    assert [(int(x) & oracle.STATUS_BAD_INDEX) != 0 for x in sr.status] == bad
    assert ((single.status & oracle.STATUS_BAD_INDEX) != 0) == any(bad)
    # rows: every operation equals the single-buffer one, sliced
    H = 16
    tok = _rows(T, H, seed + 1)
    wts = np.random.default_rng(seed).random((T, K)).astype(np.float32)
    cuts = np.cumsum([0] + [a.shape[0] for a in idx])
    tok_r = [tok[cuts[r]:cuts[r + 1]] for r in range(N)]
    w_r = [wts[cuts[r]:cuts[r + 1]] for r in range(N)]
    recv, recv_w = oracle_mod.dispatch(single, tok, wts)
    for q, (rows, rw) in enumerate(oracle_mod.shard_dispatch(sr, tok_r, w_r)):
        assert np.array_equal(rows, recv[base[q]:base[q] + sr.P[q]])
        assert np.array_equal(rw.view(np.uint32), recv_w[base[q]:base[q] + sr.P[q]].view(np.uint32))
    eo = _rows(single.P, H, seed + 2)
    eo_q = [eo[base[q]:base[q] + sr.P[q]] for q in range(N)]
    res = oracle_mod.combine(single, eo)
    for r, out in enumerate(oracle_mod.shard_combine(sr, eo_q)):
        assert np.array_equal(out, res[cuts[r]:cuts[r + 1]])
    gres = _rows(T, H, seed + 3)
    gexp = oracle_mod.combine_bwd(single, gres)
    for q, rows in enumerate(oracle_mod.shard_combine_bwd(sr, [gres[cuts[r]:cuts[r + 1]] for r in range(N)])):
        assert np.array_equal(rows, gexp[base[q]:base[q] + sr.P[q]])
    grecv = _rows(single.P, H, seed + 4)
    gw = np.random.default_rng(seed + 5).standard_normal(max(single.P, 1)).astype(np.float32)
    gtok, gtw = oracle_mod.dispatch_bwd(single, grecv, gw)
    outs = oracle_mod.shard_dispatch_bwd(sr, [grecv[base[q]:base[q] + sr.P[q]] for q in range(N)],
                                         [gw[base[q]:base[q] + max(sr.P[q], 1)] for q in range(N)])
    for r, (gt, gk) in enumerate(outs):
        assert np.array_equal(gt, gtok[cuts[r]:cuts[r + 1]])
        assert np.array_equal(gk.view(np.uint32), gtw[cuts[r]:cuts[r + 1]].view(np.uint32))
    for r, (_, gk) in enumerate(oracle_mod.shard_dispatch_bwd(sr, [grecv[base[q]:base[q] + sr.P[q]]
                                                                   for q in range(N)], None)):
        assert np.all(gk.view(np.uint32) == 0)


@pytest.mark.parametrize("N,K,E,A,seed", CONFIGS)
def test_shard_invariants(N, K, E, A, seed, oracle_mod=oracle):
    idx = _ranks(N, K, E, seed + 100, p_mask=0.1)
    sr = oracle_mod.shard_prepare(idx, E, A, N)
    el = E // N
    cat = np.concatenate([a.reshape(-1, K) for a in idx]).reshape(-1)
    s_slot, s_dest = sr._cat(sr.slot).reshape(-1), sr._cat(sr.dest).reshape(-1)
    for q in range(N):
        mine = np.nonzero(s_dest == q)[0]
        rows = s_slot[mine]
        assert len(set(rows.tolist())) == len(rows)           # one route per row
        assert np.all((rows >= 0) & (rows < sr.P[q]))
        npad = int(sr.P[q]) - len(rows)
        assert int((sr.inv[q] < 0).sum()) == npad
        for e in range(q * el, (q + 1) * el):
            lo = sr.offsets[e]
            hi = sr.offsets[e + 1] if e + 1 < (q + 1) * el else sr.P[q]
            assert (hi - lo) % A == 0
            routes = sr.inv[q][lo:hi]
            routes = routes[routes >= 0]
            assert np.all(cat[routes] == e)
            assert np.all(np.diff(routes) > 0)                   # (rank, t, k) ascending
            assert len(routes) == sr.counts[e] and hi - lo - len(routes) < A


def test_shard_overflow_flags_every_rank(oracle_mod=oracle):
    N, K, E = 4, 2, 8
    idx = [np.full((10, K), 7, np.int64), np.zeros((3, K), np.int64), np.zeros((0, K), np.int64),
           np.full((2, K), -1, np.int64)]
    sr = oracle_mod.shard_prepare(idx, E, 1, N, recv_capacity=19)
    assert sr.P.tolist() == [6, 0, 0, 20]
    assert sr.status.tolist() == [oracle.STATUS_OVERFLOW] * N
    assert oracle_mod.shard_dispatch(sr, [np.zeros((a.shape[0], 8), np.uint16) for a in idx],
                                     [np.zeros(a.shape, np.float32) for a in idx]) is None
    sr = oracle_mod.shard_prepare(idx, E, 1, N, recv_capacity=20)
    assert sr.status.tolist() == [0] * N


@pytest.mark.parametrize("case", golden_io.rounding_cases(), ids=lambda c: c[0])
def test_shard_combine_rounding_golden(case, oracle_mod=oracle):
    """The combine rounding cases (tests/golden/combine_rounding.txt) with each
    of the token's K experts on a rank of its own (N = E = K): the token's
    rows come from K owners and are still summed in ascending k."""
    name, K, rows, expected = case
    idx = [np.arange(K, dtype=np.int64).reshape(1, K)] + [np.zeros((0, K), np.int64)] * (K - 1)
    sr = oracle_mod.shard_prepare(idx, K, 1, K)
    assert sr.P.tolist() == [1] * K
    per_owner = [np.array([[rows[k]]], np.uint16) for k in range(K)]
    out = oracle_mod.shard_combine(sr, per_owner)
    assert int(out[0][0, 0]) == expected, name
    gt, _ = oracle_mod.shard_dispatch_bwd(sr, per_owner, None)[0]
    assert int(gt[0, 0]) == expected, name
