"""Rank-major sharded layers through the C ABI, against the rank-major oracle.

N ranks are emulated on one GPU, as in test_shard_gpu.py: each rank has its
own registered layer, handle memory and receive-side buffers, and the row
calls address the ranks' buffers through device pointer tables.  Compared
bit for bit with oracle.rm_*: counts per owner, received rows per owner,
status, the first-route row map, every owner's received rows, expert ids and
weights [0, M_q) (rows at or beyond M_q untouched), every rank's combine
result, token gradients and weight gradients.  One test runs the whole
two-stage step: push, the owner's local single-buffer prepare / dispatch /
combine (libep's own single-buffer calls) on the received rows, pull.
"""
import numpy as np
import pytest
import torch

from combine_ep_prepare_gb300 import workloads as wl
from ep_harness import bits, same, sentinel_tensor, untouched

pytestmark = pytest.mark.gpu

IDX_FILL = -77


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_ep_prepare_gb300 as ep
    return ep


def _routing(T_per_rank, K, E, seed, p_mask=0.1, p_bad=0.0, dsv3=False):
    out = []
    for r, T in enumerate(T_per_rank):
        if dsv3:
            w = wl.WORKLOADS["dsv3"]
            g = wl.Workload("dsv3_r%d" % r, 60 + r + seed, T=T, H=w.H, E=E, K=K, A=w.A, routing="grouped")
            idx, wts = wl.routing(g, T=T)
        else:
            idx, wts = wl.random_routing(T, K, E, seed=seed * 100 + r, p_mask=p_mask, p_bad=p_bad)
        out.append((idx, wts))
    return out


class Ranks:
    """N emulated ranks of one rank-major layer on the current GPU."""

    def __init__(self, ep, N, E, K, H, T_max, dtype="bf16", recv_capacity=0):
        self.ep, self.N, self.E, self.K, self.H, self.dtype = ep, N, E, K, H, dtype
        self.layers = [ep.ep_register_layer_rank_major(E, K, H, T_max, N, r, recv_capacity=recv_capacity,
                                                       dtype=dtype) for r in range(N)]
        self.R = ep.ep_recv_capacity(self.layers[0][0])
        self.h = [ep.alloc_handle(lid, size) for lid, size in self.layers]

    def prepare(self, idx, corrupt_counts_of=None):
        ep, N, dev = self.ep, self.N, "cuda"
        local = [torch.full((N,), -7, dtype=torch.int32, device=dev) for _ in range(N)]
        for r in range(N):
            ep.ep_rank_major_count(self.h[r], idx[r], local[r])
        all_counts = torch.stack(local).contiguous()  # the all-gather of the counts
        if corrupt_counts_of is not None:
            all_counts[corrupt_counts_of, 0] += 1
        rows = [torch.full((1,), -5, dtype=torch.int32, device=dev) for _ in range(N)]
        for r in range(N):
            ep.ep_rank_major_prepare(self.h[r], idx[r], all_counts, rows[r])
        return local, rows

    def step(self, routing, pay, corrupt_counts_of=None, null_owner_in_tables=None, weights=True):
        ep, N, K, H, R, dt, dev = self.ep, self.N, self.K, self.H, self.R, self.dtype, "cuda"
        idx = [i.to(dev) for i, _ in routing]
        wts = [w.to(dev) for _, w in routing]
        local, rows = self.prepare(idx, corrupt_counts_of)

        def owner_buf(src):
            b = sentinel_tensor((R, H), dt, dev)
            n = min(src.shape[0], R)
            b[:n] = src[:n].to(dev)
            return b

        recv = [sentinel_tensor((R, H), dt, dev) for _ in range(N)]
        recv_idx = [torch.full((R, K), IDX_FILL, dtype=torch.int64, device=dev) for _ in range(N)]
        recv_w = [torch.full((R, K), -3.0, dtype=torch.float32, device=dev) for _ in range(N)]
        grecv = [sentinel_tensor((R, H), dt, dev) for _ in range(N)]
        part = [owner_buf(x[0]) for x in pay["rows"]]
        gpart = [owner_buf(x[1]) for x in pay["rows"]]
        gw = []
        for x in pay["rows"]:
            b = torch.full((R, K), float("nan"), dtype=torch.float32, device=dev)
            n = min(x[2].shape[0], R)
            b[:n] = x[2][:n].to(dev)
            gw.append(b)

        def tab(ts):
            ts = list(ts)
            if null_owner_in_tables is not None:
                ts[null_owner_in_tables] = None
            return ep.pointer_table(ts, dev)

        t_recv, t_idx, t_w, t_grecv = tab(recv), tab(recv_idx), tab(recv_w), tab(grecv)
        t_part, t_gpart, t_gw = tab(part), tab(gpart), tab(gw)
        for r in range(N):
            ep.ep_rank_major_dispatch(self.h[r], idx[r], pay["tokens"][r].to(dev), wts[r] if weights else None,
                                      t_recv, t_idx, t_w if weights else None)
            ep.ep_rank_major_combine_bwd(self.h[r], pay["grad_result"][r].to(dev), t_grecv)
        res, gtok, gtw, slots = [], [], [], []
        for r in range(N):
            T = idx[r].shape[0]
            res.append(sentinel_tensor((T, H), dt, dev))
            gtok.append(sentinel_tensor((T, H), dt, dev))
            gtw.append(torch.full((T, K), -3.0, dtype=torch.float32, device=dev))
            ep.ep_rank_major_combine(self.h[r], t_part, res[r])
            ep.ep_rank_major_dispatch_bwd(self.h[r], t_gpart, t_gw if weights else None, gtok[r], gtw[r])
            sl = torch.full((T, K), -9, dtype=torch.int32, device=dev)
            ep.ep_token_slots(self.h[r], sl)
            slots.append(sl)
        info = [ep.ep_read_info(self.h[r]) for r in range(N)]
        torch.cuda.synchronize()
        return {"local": [x.cpu().numpy() for x in local], "rows": [int(x.item()) for x in rows],
                "slot": [x.cpu().numpy() for x in slots], "info": info,
                "recv": [bits(x) for x in recv], "recv_idx": [x.cpu().numpy() for x in recv_idx],
                "recv_w": [x.cpu().numpy() for x in recv_w], "grecv": [bits(x) for x in grecv],
                "result": [bits(x) for x in res], "grad_tokens": [bits(x) for x in gtok],
                "grad_topk_weights": [x.cpu().numpy() for x in gtw]}


def _payloads(rr, routing, H, K, dtype, seed):
    tokens = [wl.payload_normal(i.shape[0], H, seed + 10 + r, dtype) for r, (i, _) in enumerate(routing)]
    gres = [wl.payload_normal(i.shape[0], H, seed + 20 + r, dtype) for r, (i, _) in enumerate(routing)]
    rows = []
    for q in range(rr.N):
        M = max(int(rr.M[q]), 1)
        rows.append((wl.payload_normal(M, H, seed + 30 + q, dtype), wl.payload_normal(M, H, seed + 40 + q, dtype),
                     wl.f32_normal(M * K, seed + 50 + q).reshape(M, K)))
    return {"tokens": tokens, "grad_result": gres, "rows": rows}


def _check(g, rr, routing, pay, oracle_mod, dtype, weights=True):
    N = rr.N
    first = rr.first_rows()
    cuts = np.cumsum([0] + rr.tokens_per_rank)
    for r in range(N):
        assert np.array_equal(g["local"][r], rr.counts[r])
        assert g["info"][r]["status"] == int(rr.status[r]), (r, g["info"][r], rr.status)
        assert g["rows"][r] == int(rr.M[r])
        assert g["info"][r]["used_rows"] == int(rr.M[r]) and g["info"][r]["padding_rows"] == 0
        assert np.array_equal(g["slot"][r], first[cuts[r]:cuts[r + 1]])
    if rr.overflow:
        for q in range(N):
            assert untouched(g["recv"][q]) and untouched(g["grecv"][q])
            assert np.all(g["recv_idx"][q] == IDX_FILL)
        for r in range(N):
            assert untouched(g["result"][r]) and untouched(g["grad_tokens"][r])
        return
    idx = [i.numpy() for i, _ in routing]
    disp = oracle_mod.rm_dispatch(rr, idx, [bits(t) for t in pay["tokens"]], [w.numpy() for _, w in routing],
                                  dtype)
    cbwd = oracle_mod.rm_combine_bwd(rr, [bits(t) for t in pay["grad_result"]], dtype)
    comb = oracle_mod.rm_combine(rr, [bits(x[0])[:max(int(rr.M[q]), 1)] for q, x in enumerate(pay["rows"])],
                                 dtype)
    dbwd = oracle_mod.rm_dispatch_bwd(rr, [bits(x[1]) for x in pay["rows"]],
                                      [x[2].numpy() for x in pay["rows"]] if weights else None, dtype)
    for q in range(N):
        M = int(rr.M[q])
        assert same(g["recv"][q][:M], disp[q][0])
        assert np.array_equal(g["recv_idx"][q][:M], disp[q][1])
        if weights:
            assert np.array_equal(g["recv_w"][q][:M].view(np.uint32), disp[q][2].view(np.uint32))
        assert np.all(g["recv_w"][q][M if weights else 0:] == -3.0)
        assert same(g["grecv"][q][:M], cbwd[q])
        assert untouched(g["recv"][q][M:]) and untouched(g["grecv"][q][M:])
        assert np.all(g["recv_idx"][q][M:] == IDX_FILL)
    for r in range(N):
        assert same(g["result"][r], comb[r])
        assert same(g["grad_tokens"][r], dbwd[r][0])
        assert np.array_equal(g["grad_topk_weights"][r].view(np.uint32), dbwd[r][1].view(np.uint32))


CASES = [
    # N, E, K, H, tokens per rank, seed
    (1, 8, 2, 64, [100], 1),
    (2, 8, 2, 64, [100, 37], 2),
    (2, 4, 3, 200, [0, 50], 3),
    (4, 32, 4, 128, [70, 0, 129, 33], 4),
    (4, 16, 8, 72, [64, 64, 64, 64], 5),
    (8, 256, 8, 256, [128, 96, 0, 128, 17, 128, 128, 64], 6),
    (8, 64, 6, 40, [33, 1, 2, 3, 5, 8, 13, 21], 7),
    (16, 32, 32, 16, [9] * 16, 8),
    (3, 12, 3, 48, [20, 0, 33], 9),
]


@pytest.mark.parametrize("N,E,K,H,tpr,seed", CASES)
def test_rank_major_step_matches_oracle(ep, oracle_mod, N, E, K, H, tpr, seed):
    routing = _routing(tpr, K, E, seed, p_mask=0.15, p_bad=0.02 if seed % 2 else 0.0)
    ranks = Ranks(ep, N, E, K, H, max(tpr))
    rr = oracle_mod.rm_prepare([i.numpy() for i, _ in routing], E, N, ranks.R)
    pay = _payloads(rr, routing, H, K, "bf16", seed)
    g = ranks.step(routing, pay)
    _check(g, rr, routing, pay, oracle_mod, "bf16")


def test_rank_major_dsv3_shaped_ranks(ep, oracle_mod):
    """8 ranks of a DeepSeek-V3-shaped layer (E=256, K=8, group-limited
    routing, H=7168): the owners receive at most one row per token."""
    N, E, K, H = 8, 256, 8, 7168
    tpr = [256, 200, 256, 0, 256, 31, 256, 128]
    routing = _routing(tpr, K, E, 13, dsv3=True)
    ranks = Ranks(ep, N, E, K, H, max(tpr))
    rr = oracle_mod.rm_prepare([i.numpy() for i, _ in routing], E, N, ranks.R)
    assert int(rr.M.sum()) < sum(tpr) * K  # rows shared by routes to one owner
    pay = _payloads(rr, routing, H, K, "bf16", 13)
    g = ranks.step(routing, pay)
    _check(g, rr, routing, pay, oracle_mod, "bf16")


@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
def test_rank_major_payload_types(ep, oracle_mod, dtype):
    N, E, K, H, tpr = 4, 16, 4, 48, [40, 9, 0, 64]
    routing = _routing(tpr, K, E, 21, p_mask=0.2)
    ranks = Ranks(ep, N, E, K, H, max(tpr), dtype=dtype)
    rr = oracle_mod.rm_prepare([i.numpy() for i, _ in routing], E, N, ranks.R)
    pay = _payloads(rr, routing, H, K, dtype, 21)
    g = ranks.step(routing, pay)
    _check(g, rr, routing, pay, oracle_mod, dtype)


def test_rank_major_without_weights(ep, oracle_mod):
    """No weight tables: ids only on dispatch, zero weight gradients."""
    N, E, K, H, tpr = 2, 8, 4, 32, [30, 20]
    routing = _routing(tpr, K, E, 23)
    ranks = Ranks(ep, N, E, K, H, max(tpr))
    rr = oracle_mod.rm_prepare([i.numpy() for i, _ in routing], E, N, ranks.R)
    pay = _payloads(rr, routing, H, K, "bf16", 23)
    g = ranks.step(routing, pay, weights=False)
    _check(g, rr, routing, pay, oracle_mod, "bf16", weights=False)


def test_rank_major_overflow_writes_nothing(ep, oracle_mod):
    N, E, K, H = 2, 4, 2, 16
    routing = [(torch.full((20, K), 3, dtype=torch.int64), torch.rand(20, K)),
               (torch.zeros((5, K), dtype=torch.int64), torch.rand(5, K))]
    ranks = Ranks(ep, N, E, K, H, 20, recv_capacity=19)
    rr = oracle_mod.rm_prepare([i.numpy() for i, _ in routing], E, N, ranks.R)
    assert rr.overflow and rr.M.tolist() == [5, 20]
    pay = _payloads(rr, routing, H, K, "bf16", 3)
    g = ranks.step(routing, pay)
    _check(g, rr, routing, pay, oracle_mod, "bf16")


def test_rank_major_counts_mismatch_writes_nothing_on_that_rank(ep, oracle_mod):
    N, E, K, H = 2, 8, 2, 32
    routing = _routing([30, 30], K, E, 31, p_mask=0.0)
    ranks = Ranks(ep, N, E, K, H, 30)
    rr = oracle_mod.rm_prepare([i.numpy() for i, _ in routing], E, N, ranks.R)
    pay = _payloads(rr, routing, H, K, "bf16", 31)
    g = ranks.step(routing, pay, corrupt_counts_of=1)
    assert g["info"][1]["status"] & ep.EP_ST_COUNTS_MISMATCH
    assert not g["info"][0]["status"] & ep.EP_ST_COUNTS_MISMATCH
    assert untouched(g["result"][1]) and untouched(g["grad_tokens"][1])
    assert np.all(g["grad_topk_weights"][1] == -3.0)


def test_rank_major_null_table_entry_is_skipped_and_flagged(ep, oracle_mod):
    N, E, K, H = 2, 8, 2, 32
    routing = _routing([24, 24], K, E, 41, p_mask=0.0)
    ranks = Ranks(ep, N, E, K, H, 24)
    rr = oracle_mod.rm_prepare([i.numpy() for i, _ in routing], E, N, ranks.R)
    pay = _payloads(rr, routing, H, K, "bf16", 41)
    g = ranks.step(routing, pay, null_owner_in_tables=1)
    for r in range(N):
        assert g["info"][r]["status"] & ep.EP_ST_BAD_POINTER
    idx = [i.numpy() for i, _ in routing]
    disp = oracle_mod.rm_dispatch(rr, idx, [bits(t) for t in pay["tokens"]], [w.numpy() for _, w in routing])
    M0 = int(rr.M[0])
    assert same(g["recv"][0][:M0], disp[0][0])  # owner 0's rows arrive
    assert np.array_equal(g["recv_idx"][0][:M0], disp[0][1])


def test_rank_major_two_stage_step(ep, oracle_mod):
    """The whole step: push; on each owner libep's single-buffer prepare,
    dispatch and combine over the received rows and ids (an expert that
    returns its input rows); pull.  Equal, bit for bit, to the oracle's
    rank-major combine of the oracle's local single-buffer combine."""
    N, E, K, H, A = 4, 32, 4, 64, 8
    tpr = [70, 0, 129, 33]
    routing = _routing(tpr, K, E, 61, p_mask=0.1)
    ranks = Ranks(ep, N, E, K, H, max(tpr))
    dev = "cuda"
    R = ranks.R
    idx = [i.to(dev) for i, _ in routing]
    wts = [w.to(dev) for _, w in routing]
    _, rows = ranks.prepare(idx)
    recv = [torch.zeros((R, H), dtype=torch.bfloat16, device=dev) for _ in range(N)]
    recv_idx = [torch.full((R, K), -1, dtype=torch.int64, device=dev) for _ in range(N)]
    recv_w = [torch.zeros((R, K), dtype=torch.float32, device=dev) for _ in range(N)]
    tok = [wl.bf16_normal(T, H, seed=800 + r).to(dev) for r, T in enumerate(tpr)]
    for r in range(N):
        ep.ep_rank_major_dispatch(ranks.h[r], idx[r], tok[r], wts[r], ep.pointer_table(recv, dev),
                                  ep.pointer_table(recv_idx, dev), ep.pointer_table(recv_w, dev))
    torch.cuda.synchronize()
    M = [int(x.item()) for x in rows]
    partial = [torch.zeros((R, H), dtype=torch.bfloat16, device=dev) for _ in range(N)]
    for q in range(N):  # the owner's local expert-major step
        lid, size = ep.ep_register_layer(E // N, K, H, R, max_alignment=A)
        h = ep.alloc_handle(lid, size)
        RL = ep.ep_recv_capacity(lid)
        counts = torch.empty(E // N, dtype=torch.int32, device=dev)
        ep.ep_prepare(h, recv_idx[q][:M[q]], counts, A)
        lrecv = torch.zeros((RL, H), dtype=torch.bfloat16, device=dev)
        lrecv_w = torch.zeros(RL, dtype=torch.float32, device=dev)
        ep.ep_dispatch(h, recv_idx[q][:M[q]], recv[q][:M[q]], recv_w[q][:M[q]], lrecv, lrecv_w)
        ep.ep_combine(h, lrecv, partial[q][:M[q]])  # the expert returns its input rows
    res = [torch.zeros((T, H), dtype=torch.bfloat16, device=dev) for T in tpr]
    for r in range(N):
        ep.ep_rank_major_combine(ranks.h[r], ep.pointer_table(partial, dev), res[r])
    torch.cuda.synchronize()
    # oracle: the same two stages
    rr = oracle_mod.rm_prepare([i.numpy() for i, _ in routing], E, N, R)
    pushed = oracle_mod.rm_dispatch(rr, [i.numpy() for i, _ in routing], [bits(t) for t in tok],
                                    [w.numpy() for _, w in routing])
    parts = []
    for q in range(N):
        orows, oids, ow = pushed[q]
        assert same(bits(recv[q])[:M[q]], orows) and np.array_equal(recv_idx[q][:M[q]].cpu().numpy(), oids)
        local = oracle_mod.prepare(oids, E // N, A)
        lr, _ = oracle_mod.dispatch(local, orows, ow)
        parts.append(oracle_mod.combine(local, lr))
        assert same(bits(partial[q])[:M[q]], parts[q])
    want = oracle_mod.rm_combine(rr, parts)
    for r in range(N):
        assert same(bits(res[r]), want[r])


def test_rank_major_step_captures_in_a_cuda_graph(ep, oracle_mod):
    """Count, prepare and the four row calls of two ranks capture in one CUDA
    graph; a replay after new routing in the same buffers matches the oracle
    for that routing."""
    N, E, K, H, T = 2, 16, 4, 64, 96
    ranks = Ranks(ep, N, E, K, H, T)
    dev = "cuda"
    R = ranks.R
    idx = [torch.zeros((T, K), dtype=torch.int64, device=dev) for _ in range(N)]
    wts = [torch.zeros((T, K), dtype=torch.float32, device=dev) for _ in range(N)]
    local = [torch.empty(N, dtype=torch.int32, device=dev) for _ in range(N)]
    table = torch.empty(N, N, dtype=torch.int32, device=dev)
    rows = [torch.empty(1, dtype=torch.int32, device=dev) for _ in range(N)]
    recv = [torch.zeros((R, H), dtype=torch.bfloat16, device=dev) for _ in range(N)]
    recv_idx = [torch.full((R, K), -1, dtype=torch.int64, device=dev) for _ in range(N)]
    recv_w = [torch.zeros((R, K), dtype=torch.float32, device=dev) for _ in range(N)]
    part = [wl.bf16_normal(R, H, seed=900 + q).to(dev) for q in range(N)]
    tok = [wl.bf16_normal(T, H, seed=910 + r).to(dev) for r in range(N)]
    res = [torch.zeros((T, H), dtype=torch.bfloat16, device=dev) for _ in range(N)]
    tabs = [ep.pointer_table(x, dev) for x in (recv, recv_idx, recv_w, part)]
    s = torch.cuda.Stream()

    def step():
        for r in range(N):
            ep.ep_rank_major_count(ranks.h[r], idx[r], local[r], stream=s)
        for r in range(N):
            table[r].copy_(local[r])
        for r in range(N):
            ep.ep_rank_major_prepare(ranks.h[r], idx[r], table, rows[r], stream=s)
        for r in range(N):
            ep.ep_rank_major_dispatch(ranks.h[r], idx[r], tok[r], wts[r], tabs[0], tabs[1], tabs[2], stream=s)
        for r in range(N):
            ep.ep_rank_major_combine(ranks.h[r], tabs[3], res[r], stream=s)

    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    routing = _routing([T, T], K, E, 71, p_mask=0.1)
    for r in range(N):
        idx[r].copy_(routing[r][0].to(dev))
        wts[r].copy_(routing[r][1].to(dev))
    g.replay()
    torch.cuda.synchronize()
    rr = oracle_mod.rm_prepare([i.numpy() for i, _ in routing], E, N, R)
    pushed = oracle_mod.rm_dispatch(rr, [i.numpy() for i, _ in routing], [bits(t) for t in tok],
                                    [w.numpy() for _, w in routing])
    comb = oracle_mod.rm_combine(rr, [bits(p) for p in part])
    for q in range(N):
        M = int(rr.M[q])
        assert int(rows[q].item()) == M
        assert same(bits(recv[q])[:M], pushed[q][0])
        assert np.array_equal(recv_idx[q][:M].cpu().numpy(), pushed[q][1])
    for r in range(N):
        assert same(bits(res[r]), comb[r])
