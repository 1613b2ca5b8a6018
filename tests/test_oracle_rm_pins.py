"""Pins of the rank-major oracle (expert parallelism over N ranks with a
rank-major receive layout), CPU only.

TransformerEngine PR #3035's review thread on the receive buffers sets a
rank-major buffer (at most max_tokens_per_rank x num_ranks rows per owner)
against the expert-major one, with the owner permuting the received rows
locally.  The readings are in the header of oracle/ep_oracle.c.  Pinned by
  - hand-worked cases (tests/golden/rank_major_hand_worked.txt), including a
    combine whose float32 order decides the result;
  - brute force on small batches: every map, the dispatch and the whole
    two-stage step (rank-major dispatch, the owner's local single-buffer
    prepare / dispatch / combine, rank-major combine) recomputed per token
    from the definitions in numpy float32;
  - identities with the single-buffer oracle (pinned on its own in
    test_oracle_pins.py): with one rank, and whenever every token's routes
    have distinct owners, the two-stage step equals the single-buffer step
    bit for bit; the backward passes are the adjoints of the forward ones.
"""
import numpy as np
import pytest

import golden_io
import oracle
from combine_ep_prepare_gb300 import workloads as wl


def _bf16(vals):
    return np.array([oracle.f32_to_bf16(float(v)) for v in vals], np.uint16)


def _f32(bits):
    return np.array([oracle.bf16_to_f32(int(b)) for b in np.asarray(bits).reshape(-1)], np.float32)


@pytest.mark.parametrize("case", golden_io.rank_major_cases(), ids=lambda c: c["name"])
def test_rank_major_golden(case, oracle_mod=oracle):
    N, K, E = case["N"], case["K"], case["E"]
    idx = [np.array(case["idx%d" % r], np.int64).reshape(-1, K) for r in range(N)]
    w = [np.array(case["w%d" % r], np.float32).reshape(-1, K) for r in range(N)]
    rr = oracle_mod.rm_prepare(idx, E, N, case["R"])
    assert rr.counts.reshape(-1).tolist() == case["counts"]
    assert rr.M.tolist() == case["M"]
    for r in range(N):
        assert rr.row[r].reshape(-1).tolist() == case["row%d" % r]
        assert rr.dest[r].reshape(-1).tolist() == case["dest%d" % r]
        assert rr.first[r].reshape(-1).astype(int).tolist() == case["first%d" % r]
    for q in range(N):
        assert rr.src[q].tolist() == case["src%d" % q]
    assert rr.status.tolist() == case["status"]
    if "ids0" not in case:
        return
    tokens = [np.zeros((a.shape[0], 8), np.uint16) + np.arange(8, dtype=np.uint16) for a in idx]
    out = oracle_mod.rm_dispatch(rr, idx, tokens, w)
    for q in range(N):
        rows, ids, rw = out[q]
        assert ids.reshape(-1).tolist() == case["ids%d" % q]
        assert rw.reshape(-1).tolist() == case["rw%d" % q]
    if "part0" in case:
        parts = [_bf16(case["part%d" % q]).reshape(-1, 1) for q in range(N)]
        res = oracle_mod.rm_combine(rr, parts)
        for r in range(N):
            assert _f32(res[r]).tolist() == case["out%d" % r]
    if "gw0" in case:
        gws = [np.array(case["gw%d" % q], np.float32).reshape(-1, K) for q in range(N)]
        back = oracle_mod.rm_dispatch_bwd(rr, [np.zeros((int(m), 1), np.uint16) for m in rr.M], gws)
        for r in range(N):
            assert back[r][1].reshape(-1).tolist() == case["gout%d" % r]


def _ranks(N, K, E, seed, p_mask=0.2, p_bad=0.0, tmax=24, distinct=False):
    g = np.random.default_rng(seed)
    idx, wts = [], []
    for r in range(N):
        T = int(g.integers(0, tmax + 1)) if r % 3 != 2 else int(g.integers(0, 3))
        i, w = wl.random_routing(T, K, E, seed=seed * 37 + r, p_mask=p_mask, p_bad=p_bad,
                                 distinct=distinct)
        idx.append(i.numpy())
        wts.append(w.numpy())
    return idx, wts


def _rows(n, H, seed):
    import torch
    return wl.bf16_normal(max(n, 1), H, seed).view(torch.int16).numpy().view(np.uint16)[:n].copy()


CONFIGS = [(2, 2, 4, 1), (2, 3, 8, 2), (4, 4, 8, 3), (4, 1, 4, 4), (8, 8, 16, 5), (3, 2, 6, 6),
           (2, 6, 2, 7), (4, 8, 32, 8)]


@pytest.mark.parametrize("N,K,E,seed", CONFIGS)
def test_rank_major_maps_brute_force(N, K, E, seed, oracle_mod=oracle):
    """Every map recomputed per token from the definitions."""
    idx, w = _ranks(N, K, E, seed, p_bad=0.05)
    rr = oracle_mod.rm_prepare(idx, E, N)
    el = E // N
    cat = np.concatenate([a.reshape(-1, K) for a in idx])
    rank_of = np.concatenate([np.full(a.shape[0], r) for r, a in enumerate(idx)]).astype(int)
    rows_of = [[] for _ in range(N)]
    counts = np.zeros((N, N), int)
    exp_row, exp_dest, exp_first = [], [], []
    for g, toks in enumerate(cat):
        seen = {}
        for e in toks:
            if 0 <= e < E and e // el not in seen:
                q = int(e // el)
                seen[q] = len(rows_of[q])
                rows_of[q].append(g)
                counts[rank_of[g], q] += 1
        done = set()
        for e in toks:
            if 0 <= e < E:
                q = int(e // el)
                exp_row.append(seen[q])
                exp_dest.append(q)
                exp_first.append(q not in done)
                done.add(q)
            else:
                exp_row.append(-1)
                exp_dest.append(-1)
                exp_first.append(False)
    assert np.array_equal(rr.counts, counts)
    assert rr.M.tolist() == [len(x) for x in rows_of]
    for q in range(N):
        assert rr.src[q].tolist() == rows_of[q]
    assert rr._cat(rr.row).reshape(-1).tolist() == exp_row
    assert rr._cat(rr.dest).reshape(-1).tolist() == exp_dest
    assert rr._cat(rr.first).reshape(-1).tolist() == exp_first
    bad = [bool(((a < -1) | (a >= E)).any()) for a in idx]
    assert [bool(s & oracle.STATUS_BAD_INDEX) for s in rr.status] == bad
    # rank-major bound: a token sends at most one row per owner
    assert all(int(rr.M[q]) <= cat.shape[0] for q in range(N))


@pytest.mark.parametrize("N,K,E,seed", CONFIGS)
def test_rank_major_dispatch_brute_force(N, K, E, seed, oracle_mod=oracle):
    idx, w = _ranks(N, K, E, seed, p_bad=0.05)
    H = 24
    toks = [_rows(a.shape[0], H, 500 + seed * 10 + r) for r, a in enumerate(idx)]
    rr = oracle_mod.rm_prepare(idx, E, N)
    out = oracle_mod.rm_dispatch(rr, idx, toks, w)
    cat, tcat = np.concatenate([a.reshape(-1, K) for a in idx]), np.concatenate(toks)
    wcat = np.concatenate([x.reshape(-1, K) for x in w])
    el = E // N
    for q in range(N):
        rows, ids, rw = out[q]
        for s, g in enumerate(rr.src[q]):
            assert np.array_equal(rows[s], tcat[g])
            mine = (cat[g] >= 0) & (cat[g] < E) & (np.clip(cat[g], 0, E - 1) // el == q)
            assert np.array_equal(ids[s], np.where(mine, cat[g] - q * el, -1))
            assert np.array_equal(rw[s], np.where(mine, wcat[g], 0.0).astype(np.float32))


def _two_stage(idx, w, E, N, A, H, seed, oracle_mod):
    """The whole rank-major step: push, the owner's local single-buffer step
    on the received rows, pull.  Expert output of route (g, k) = f(g, k)."""
    K = idx[0].shape[1]
    cat = np.concatenate([a.reshape(-1, K) for a in idx])
    T = cat.shape[0]
    f = _rows(T * K, H, seed).reshape(T, K, H)
    rr = oracle_mod.rm_prepare(idx, E, N)
    toks = [np.zeros((a.shape[0], H), np.uint16) for a in idx]
    pushed = oracle_mod.rm_dispatch(rr, idx, toks, w)
    partials = []
    for q in range(N):
        _, ids, _ = pushed[q]
        local = oracle_mod.prepare(ids, E // N, A)
        eo = np.zeros((max(local.P, 1), H), np.uint16)
        for s, g in enumerate(rr.src[q]):
            for k in range(K):
                if local.slot[s, k] >= 0:
                    eo[local.slot[s, k]] = f[g, k]
        partials.append(oracle_mod.combine(local, eo))
    return rr, f, oracle_mod.rm_combine(rr, partials)


@pytest.mark.parametrize("N,K,E,seed", CONFIGS)
def test_two_stage_combine_brute_force(N, K, E, seed, oracle_mod=oracle):
    """result[g] = bf16(sum over owners in first-route order of
    f32(bf16(sum over that owner's routes, k ascending, of f32(f(g, k)))))."""
    idx, w = _ranks(N, K, E, seed)
    H = 16
    rr, f, res = _two_stage(idx, w, E, N, 3, H, 900 + seed, oracle_mod)
    cat = np.concatenate([a.reshape(-1, K) for a in idx])
    got = np.concatenate(res)
    el = E // N
    for g, toks in enumerate(cat):
        order = []
        for e in toks:
            if 0 <= e < E and e // el not in order:
                order.append(int(e // el))
        acc = np.zeros(H, np.float32)
        for q in order:
            part = np.zeros(H, np.float32)
            for k, e in enumerate(toks):
                if 0 <= e < E and e // el == q:
                    part = (part + _f32(f[g, k])).astype(np.float32)
            acc = (acc + _f32(oracle.round_to_bf16(part))).astype(np.float32)
        assert np.array_equal(got[g], oracle.round_to_bf16(acc)), g


@pytest.mark.parametrize("N,K,E,seed", [(1, 2, 4, 1), (1, 8, 16, 2), (1, 3, 5, 3)])
def test_one_rank_equals_single_buffer_step(N, K, E, seed, oracle_mod=oracle):
    idx, w = _ranks(N, K, E, seed, tmax=60)
    H = 8
    rr, f, res = _two_stage(idx, w, E, N, 4, H, 700 + seed, oracle_mod)
    cat = idx[0].reshape(-1, K)
    single = oracle_mod.prepare(cat, E, 4)
    eo = np.zeros((max(single.P, 1), H), np.uint16)
    for g in range(cat.shape[0]):
        for k in range(K):
            if single.slot[g, k] >= 0:
                eo[single.slot[g, k]] = f[g, k]
    assert np.array_equal(res[0], oracle_mod.combine(single, eo))


@pytest.mark.parametrize("N,K,E,seed", [(4, 4, 8, 11), (8, 8, 16, 12), (4, 2, 4, 13)])
def test_distinct_owners_equal_single_buffer_step(N, K, E, seed, oracle_mod=oracle):
    """One expert per owner and distinct experts per token: every partial row
    is a single expert row, so the two roundings collapse into one."""
    el = E // N
    idx = []
    for r in range(N):
        i, _ = wl.random_routing(7 + r, K, N, seed=seed * 5 + r, p_mask=0.2, distinct=True)
        i = i.numpy()
        idx.append(np.where(i >= 0, i * el, -1))  # expert q*el of owner q
    w = [np.ones(a.shape, np.float32) for a in idx]
    H = 8
    rr, f, res = _two_stage(idx, w, E, N, 2, H, 300 + seed, oracle_mod)
    cat = np.concatenate(idx)
    single = oracle_mod.prepare(cat, E, 2)
    eo = np.zeros((max(single.P, 1), H), np.uint16)
    for g in range(cat.shape[0]):
        for k in range(K):
            if single.slot[g, k] >= 0:
                eo[single.slot[g, k]] = f[g, k]
    assert np.array_equal(np.concatenate(res), oracle_mod.combine(single, eo))


@pytest.mark.parametrize("N,K,E,seed", CONFIGS[:5])
def test_backward_passes_are_adjoints(N, K, E, seed, oracle_mod=oracle):
    """<push(x), y> = <x, pull(y)> in exact arithmetic: rows of small
    integers, so the float32 sums and bf16 roundings are exact."""
    idx, w = _ranks(N, K, E, seed)
    H = 4
    rr = oracle_mod.rm_prepare(idx, E, N)
    g = np.random.default_rng(seed)
    x = [_bf16(g.integers(-4, 5, size=a.shape[0] * H)).reshape(-1, H) for a in idx]
    y = [_bf16(g.integers(-4, 5, size=int(m) * H)).reshape(-1, H) for m in rr.M]
    pushed = oracle_mod.rm_combine_bwd(rr, x)
    pulled = oracle_mod.rm_combine(rr, y)
    lhs = sum(float((_f32(p).reshape(-1, H) * _f32(b).reshape(-1, H)).sum()) for p, b in zip(pushed, y))
    rhs = sum(float((_f32(a).reshape(-1, H) * _f32(c).reshape(-1, H)).sum()) for a, c in zip(x, pulled))
    assert lhs == rhs
    # the combine backward sends the token's gradient to every row holding it
    cat = np.concatenate(x)
    for q in range(N):
        assert np.array_equal(pushed[q], cat[rr.src[q]])
    # dispatch_bwd's token half is the combine of the row gradients
    back = oracle_mod.rm_dispatch_bwd(rr, y, None)
    for r in range(N):
        assert np.array_equal(back[r][0], pulled[r])
        assert not back[r][1].any()


def test_overflow_writes_nothing(oracle_mod=oracle):
    idx, w = _ranks(2, 2, 4, 21, p_mask=0.0, tmax=10)
    rr = oracle_mod.rm_prepare(idx, 4, 2, recv_capacity=0)
    assert all(s & oracle.STATUS_OVERFLOW for s in rr.status) == (rr.M.max() > 0)
    if rr.M.max() > 0:
        assert oracle_mod.rm_dispatch(rr, idx, [np.zeros((a.shape[0], 8), np.uint16) for a in idx], w) is None
        assert oracle_mod.rm_combine(rr, [np.zeros((1, 8), np.uint16)] * 2) is None
