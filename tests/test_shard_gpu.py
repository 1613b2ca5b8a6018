"""Sharded expert parallelism through the C ABI, against the sharded oracle.

N ranks are emulated on one GPU: each rank has its own registered layer, its
own handle memory and its own receive-side buffers, and the row calls address
the ranks' buffers through device pointer tables, exactly as they would
address peer-mapped buffers on a multi-GPU node.  The ranks' kernels never
wait on one another, so running them one after another on one stream is the
same computation.  Every output is compared bit for bit with
oracle.shard_*: counts, owner offsets, slot and owner maps, status, every
owner's receive rows [0, P_q) (rows at or beyond P_q untouched), every rank's
combine result and token gradients, and the weight gradients; one case also
checks the owners' buffers against the single-buffer step of all ranks'
tokens concatenated.
"""
import numpy as np
import pytest
import torch

from combine_ep_prepare_gb300 import workloads as wl
from ep_harness import SENTINEL32, bits, same, sentinel_tensor, untouched

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_ep_prepare_gb300 as ep
    return ep


def _routing(N, T_per_rank, K, E, seed, p_mask=0.1, p_bad=0.0, dsv3=False):
    out = []
    for r, T in enumerate(T_per_rank):
        if dsv3:
            w = wl.WORKLOADS["dsv3"]
            g = wl.Workload("dsv3_r%d" % r, 40 + r + seed, T=T, H=w.H, E=E, K=K, A=w.A, routing="grouped")
            idx, wts = wl.routing(g, T=T)
        else:
            idx, wts = wl.random_routing(T, K, E, seed=seed * 100 + r, p_mask=p_mask, p_bad=p_bad)
        out.append((idx, wts))
    return out


class Ranks:
    """N emulated ranks of one sharded layer on the current GPU."""

    def __init__(self, ep, N, E, K, H, T_max, A_max, dtype="bf16", recv_capacity=0):
        self.ep, self.N, self.E, self.K, self.H, self.dtype = ep, N, E, K, H, dtype
        self.layers = [ep.ep_register_layer_sharded(E, K, H, T_max, N, r, max_alignment=A_max,
                                                    recv_capacity=recv_capacity, dtype=dtype)
                       for r in range(N)]
        self.R = ep.ep_recv_capacity(self.layers[0][0])
        self.h = [ep.alloc_handle(lid, size) for lid, size in self.layers]

    def step(self, routing, A, payloads, corrupt_counts_of=None, null_owner_in_tables=None):
        ep, N, E, K, H, R, dt = self.ep, self.N, self.E, self.K, self.H, self.R, self.dtype
        dev = "cuda"
        idx = [i.to(dev) for i, _ in routing]
        wts = [w.to(dev) for _, w in routing]
        local = [torch.full((E,), -7, dtype=torch.int32, device=dev) for _ in range(N)]
        for r in range(N):
            ep.ep_shard_count(self.h[r], idx[r], local[r])
        all_counts = torch.stack(local).contiguous()  # the all-gather of the counts
        if corrupt_counts_of is not None:
            all_counts[corrupt_counts_of, 0] += 1
        tc = [torch.full((E // N,), -5, dtype=torch.int32, device=dev) for _ in range(N)]
        for r in range(N):
            ep.ep_shard_prepare(self.h[r], idx[r], all_counts, tc[r], A)
        # owners' receive-side buffers, sentinel beyond the rows the oracle fills
        rows_in = payloads["rows"]  # per owner: (expert_out, grad_recv, grad_recv_w)

        def owner_buf(src):
            b = sentinel_tensor((R, H), dt, dev)
            n = min(src.shape[0], R)
            b[:n] = src[:n].to(dev)
            return b

        recv = [sentinel_tensor((R, H), dt, dev) for _ in range(N)]
        recv_w = [torch.full((R,), -3.0, dtype=torch.float32, device=dev) for _ in range(N)]
        gexp = [sentinel_tensor((R, H), dt, dev) for _ in range(N)]
        eo = [owner_buf(x[0]) for x in rows_in]
        grecv = [owner_buf(x[1]) for x in rows_in]
        grecv_w = []
        for x in rows_in:
            b = torch.full((R,), float("nan"), dtype=torch.float32, device=dev)
            n = min(x[2].shape[0], R)
            b[:n] = x[2][:n].to(dev)
            grecv_w.append(b)

        def tab(ts):
            ts = list(ts)
            if null_owner_in_tables is not None:
                ts[null_owner_in_tables] = None
            return ep.pointer_table(ts, dev)

        t_recv, t_recv_w, t_gexp = tab(recv), tab(recv_w), tab(gexp)
        t_eo, t_grecv, t_grecv_w = tab(eo), tab(grecv), tab(grecv_w)
        res, gtok, gtw = [], [], []
        for r in range(N):
            T = idx[r].shape[0]
            tok = payloads["tokens"][r].to(dev)
            gres = payloads["grad_result"][r].to(dev)
            ep.ep_shard_dispatch(self.h[r], tok, wts[r], t_recv, t_recv_w)
            ep.ep_shard_combine_bwd(self.h[r], gres, t_gexp)
        for r in range(N):
            T = idx[r].shape[0]
            res.append(sentinel_tensor((T, H), dt, dev))
            gtok.append(sentinel_tensor((T, H), dt, dev))
            gtw.append(torch.full((T, K), -3.0, dtype=torch.float32, device=dev))
            ep.ep_shard_combine(self.h[r], t_eo, res[r])
            ep.ep_shard_dispatch_bwd(self.h[r], t_grecv, t_grecv_w, gtok[r], gtw[r])
        maps = []
        for r in range(N):
            T = idx[r].shape[0]
            off = torch.full((E // N + 1,), -9, dtype=torch.int32, device=dev)
            sl = torch.full((T, K), -9, dtype=torch.int32, device=dev)
            ow = torch.full((T, K), -9, dtype=torch.int32, device=dev)
            ep.ep_expert_offsets(self.h[r], off)
            ep.ep_token_slots(self.h[r], sl)
            ep.ep_shard_token_owners(self.h[r], ow)
            maps.append((off, sl, ow))
        info = [ep.ep_read_info(self.h[r]) for r in range(N)]
        torch.cuda.synchronize()
        return {"local": [x.cpu().numpy() for x in local], "token_counts": [x.cpu().numpy() for x in tc],
                "offsets": [m[0].cpu().numpy() for m in maps], "slot": [m[1].cpu().numpy() for m in maps],
                "owner": [m[2].cpu().numpy() for m in maps], "info": info,
                "recv": [bits(x) for x in recv], "recv_w": [x.cpu().numpy() for x in recv_w],
                "gexp": [bits(x) for x in gexp], "result": [bits(x) for x in res],
                "grad_tokens": [bits(x) for x in gtok], "grad_topk_weights": [x.cpu().numpy() for x in gtw]}


def _payloads(sr, routing, H, dtype, seed, oracle_mod):
    N = sr.N
    tokens = [wl.payload_normal(i.shape[0], H, seed + 10 + r, dtype) for r, (i, _) in enumerate(routing)]
    gres = [wl.payload_normal(i.shape[0], H, seed + 20 + r, dtype) for r, (i, _) in enumerate(routing)]
    rows = []
    for q in range(N):
        P = max(int(sr.P[q]), 1)
        rows.append((wl.payload_normal(P, H, seed + 30 + q, dtype), wl.payload_normal(P, H, seed + 40 + q, dtype),
                     wl.f32_normal(P, seed + 50 + q)))
    return {"tokens": tokens, "grad_result": gres, "rows": rows}


def _check(g, sr, routing, pay, oracle_mod, dtype, R):
    N, E = sr.N, sr.E
    for r in range(N):
        assert np.array_equal(g["local"][r], np.bincount(
            routing[r][0].numpy().reshape(-1)[(routing[r][0].numpy().reshape(-1) >= 0) &
                                              (routing[r][0].numpy().reshape(-1) < E)], minlength=E))
        assert g["info"][r]["status"] == int(sr.status[r]), (r, g["info"][r], sr.status)
        assert np.array_equal(g["token_counts"][r], sr.local_counts(r))
        assert np.array_equal(g["offsets"][r], sr.local_offsets(r))
        assert np.array_equal(g["slot"][r], sr.slot[r])
        assert np.array_equal(g["owner"][r], sr.dest[r])
        assert g["info"][r]["used_rows"] == int(sr.P[r])
        assert g["info"][r]["padding_rows"] == int((sr.inv[r] < 0).sum())
    if sr.overflow:
        for q in range(N):
            assert untouched(g["recv"][q]) and untouched(g["gexp"][q])
        return
    to_np = lambda ts: [bits(t) for t in ts]  # noqa: E731
    disp = oracle_mod.shard_dispatch(sr, to_np(pay["tokens"]), [w.numpy() for _, w in routing], dtype)
    cbwd = oracle_mod.shard_combine_bwd(sr, to_np(pay["grad_result"]), dtype)
    comb = oracle_mod.shard_combine(sr, [bits(x[0])[:max(int(sr.P[q]), 1)] for q, x in enumerate(pay["rows"])], dtype)
    dbwd = oracle_mod.shard_dispatch_bwd(sr, [bits(x[1]) for x in pay["rows"]],
                                         [x[2].numpy() for x in pay["rows"]], dtype)
    for q in range(N):
        P = int(sr.P[q])
        assert same(g["recv"][q][:P], disp[q][0])
        assert np.array_equal(g["recv_w"][q][:P].view(np.uint32), disp[q][1].view(np.uint32))
        assert same(g["gexp"][q][:P], cbwd[q])
        assert untouched(g["recv"][q][P:]) and untouched(g["gexp"][q][P:])
        assert np.all(g["recv_w"][q][P:] == -3.0)
    for r in range(N):
        assert same(g["result"][r], comb[r])
        assert same(g["grad_tokens"][r], dbwd[r][0])
        assert np.array_equal(g["grad_topk_weights"][r].view(np.uint32), dbwd[r][1].view(np.uint32))


CASES = [
    # N, E, K, H, tokens per rank, A, seed
    (1, 8, 2, 64, [100], 16, 1),
    (2, 8, 2, 64, [100, 37], 16, 2),
    (2, 4, 3, 200, [0, 50], 4, 3),
    (4, 32, 4, 128, [70, 0, 129, 33], 8, 4),
    (4, 16, 8, 72, [64, 64, 64, 64], 1, 5),
    (8, 256, 8, 256, [128, 96, 0, 128, 17, 128, 128, 64], 128, 6),
    (8, 64, 6, 40, [33, 1, 2, 3, 5, 8, 13, 21], 3, 7),
    (3, 12, 3, 48, [20, 0, 33], 4, 8),
]


@pytest.mark.parametrize("N,E,K,H,tpr,A,seed", CASES)
def test_shard_step_matches_oracle(ep, oracle_mod, N, E, K, H, tpr, A, seed):
    routing = _routing(N, tpr, K, E, seed, p_mask=0.15, p_bad=0.02 if seed % 2 else 0.0)
    sr = oracle_mod.shard_prepare([i.numpy() for i, _ in routing], E, A, N)
    ranks = Ranks(ep, N, E, K, H, max(tpr), 128)
    sr = oracle_mod.shard_prepare([i.numpy() for i, _ in routing], E, A, N, ranks.R)
    pay = _payloads(sr, routing, H, "bf16", seed, oracle_mod)
    g = ranks.step(routing, A, pay)
    _check(g, sr, routing, pay, oracle_mod, "bf16", ranks.R)


def test_shard_dsv3_shaped_ranks_reassemble_the_single_buffer_step(ep, oracle_mod):
    """8 ranks of a DeepSeek-V3-shaped layer (E=256, K=8, group-limited
    routing, A=128, H=7168): each owner's receive rows equal the matching
    rows of the single-buffer libep step over all ranks' tokens, bit for
    bit, and every rank's results the matching token slice."""
    N, E, K, H, A = 8, 256, 8, 7168, 128
    tpr = [256, 200, 256, 0, 256, 31, 256, 128]
    routing = _routing(N, tpr, K, E, 11, dsv3=True)
    ranks = Ranks(ep, N, E, K, H, max(tpr), A)
    sr = oracle_mod.shard_prepare([i.numpy() for i, _ in routing], E, A, N, ranks.R)
    pay = _payloads(sr, routing, H, "bf16", 11, oracle_mod)
    g = ranks.step(routing, A, pay)
    _check(g, sr, routing, pay, oracle_mod, "bf16", ranks.R)
    # the single-buffer library step on the concatenated batch
    from ep_harness import GpuLayer, StepInputs, gpu_step
    T = sum(tpr)
    cat_idx = torch.cat([i for i, _ in routing])
    cat_w = torch.cat([w for _, w in routing])
    single = oracle_mod.prepare(cat_idx.numpy(), E, A)
    base = [int(single.offsets[q * (E // N)]) for q in range(N)]
    eo = torch.cat([pay["rows"][q][0][:int(sr.P[q])] for q in range(N)])
    grecv = torch.cat([pay["rows"][q][1][:int(sr.P[q])] for q in range(N)])
    grecv_w = torch.cat([pay["rows"][q][2][:int(sr.P[q])] for q in range(N)])
    inp = StepInputs(E=E, K=K, H=H, A=A, topk_idx=cat_idx, topk_weights=cat_w,
                     tokens=torch.cat(pay["tokens"]), expert_out=eo, grad_result=torch.cat(pay["grad_result"]),
                     grad_recv=grecv, grad_recv_w=grecv_w)
    layer = GpuLayer(ep, E, K, H, T, A)
    s = gpu_step(ep, layer, inp)
    cuts = np.cumsum([0] + tpr)
    for q in range(N):
        P = int(sr.P[q])
        assert same(g["recv"][q][:P], s["recv_tokens"][base[q]:base[q] + P])
        assert same(g["gexp"][q][:P], s["grad_expert_out"][base[q]:base[q] + P])
    for r in range(N):
        assert same(g["result"][r], s["result"][cuts[r]:cuts[r + 1]])
        assert same(g["grad_tokens"][r], s["grad_tokens"][cuts[r]:cuts[r + 1]])


@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
def test_shard_payload_types(ep, oracle_mod, dtype):
    N, E, K, H, tpr, A = 4, 16, 4, 48, [40, 9, 0, 64], 8
    routing = _routing(N, tpr, K, E, 21, p_mask=0.2)
    ranks = Ranks(ep, N, E, K, H, max(tpr), 16, dtype=dtype)
    sr = oracle_mod.shard_prepare([i.numpy() for i, _ in routing], E, A, N, ranks.R)
    pay = _payloads(sr, routing, H, dtype, 21, oracle_mod)
    g = ranks.step(routing, A, pay)
    _check(g, sr, routing, pay, oracle_mod, dtype, ranks.R)


def test_shard_overflow_writes_nothing(ep, oracle_mod):
    """An owner whose rows exceed R: every rank sees EP_ST_OVERFLOW and no
    rank's row calls write anything."""
    N, E, K, H, A = 2, 4, 2, 16, 1
    routing = [(torch.full((20, K), 3, dtype=torch.int64), torch.rand(20, K)),
               (torch.zeros((5, K), dtype=torch.int64), torch.rand(5, K))]
    ranks = Ranks(ep, N, E, K, H, 20, 1, recv_capacity=39)
    sr = oracle_mod.shard_prepare([i.numpy() for i, _ in routing], E, A, N, ranks.R)
    assert sr.overflow and sr.P.tolist() == [10, 40]
    pay = _payloads(sr, routing, H, "bf16", 3, oracle_mod)
    g = ranks.step(routing, A, pay)
    _check(g, sr, routing, pay, oracle_mod, "bf16", ranks.R)
    for r in range(N):
        assert untouched(g["result"][r]) and untouched(g["grad_tokens"][r])


def test_shard_counts_mismatch_writes_nothing_on_that_rank(ep, oracle_mod):
    N, E, K, H, A = 2, 8, 2, 32, 4
    routing = _routing(N, [30, 30], K, E, 31, p_mask=0.0)
    ranks = Ranks(ep, N, E, K, H, 30, 4)
    sr = oracle_mod.shard_prepare([i.numpy() for i, _ in routing], E, A, N, ranks.R)
    pay = _payloads(sr, routing, H, "bf16", 31, oracle_mod)
    g = ranks.step(routing, A, pay, corrupt_counts_of=1)
    assert g["info"][1]["status"] & ep.EP_ST_COUNTS_MISMATCH
    assert not g["info"][0]["status"] & ep.EP_ST_COUNTS_MISMATCH
    assert untouched(g["result"][1]) and untouched(g["grad_tokens"][1])
    assert np.all(g["grad_topk_weights"][1] == -3.0)


def test_shard_null_table_entry_is_skipped_and_flagged(ep, oracle_mod):
    """A NULL address in the pointer tables: rows it would address are
    skipped, EP_ST_BAD_POINTER is set, everything else is written."""
    N, E, K, H, A = 2, 8, 2, 32, 4
    routing = _routing(N, [24, 24], K, E, 41, p_mask=0.0)
    ranks = Ranks(ep, N, E, K, H, 24, 4)
    sr = oracle_mod.shard_prepare([i.numpy() for i, _ in routing], E, A, N, ranks.R)
    pay = _payloads(sr, routing, H, "bf16", 41, oracle_mod)
    g = ranks.step(routing, A, pay, null_owner_in_tables=1)
    for r in range(N):
        assert g["info"][r]["status"] & ep.EP_ST_BAD_POINTER
    disp = oracle_mod.shard_dispatch(sr, [bits(t) for t in pay["tokens"]], [w.numpy() for _, w in routing])
    P0 = int(sr.P[0])
    assert same(g["recv"][0][:P0], disp[0][0])   # owner 0's rows arrive
    # routes whose rows live on owner 1 contribute nothing to combine
    comb = oracle_mod.shard_combine(sr, [bits(pay["rows"][0][0]), np.zeros_like(bits(pay["rows"][1][0]))])
    for r in range(N):
        ok = ~(sr.dest[r] == 1).any(axis=1)  # tokens with no route on owner 1
        assert same(g["result"][r][ok], comb[r][ok])


def test_shard_step_captures_in_a_cuda_graph(ep, oracle_mod):
    """The sharded calls allocate nothing and only enqueue work, so two
    ranks' whole step (count, prepare, the four row calls) captures in one
    CUDA graph; replays reproduce the eager results bit for bit, and a replay
    after new routing in the same buffers matches the oracle for that
    routing."""
    N, E, K, H, A, T = 2, 16, 4, 64, 8, 96
    ranks = Ranks(ep, N, E, K, H, T, 8)
    dev = "cuda"
    routing = _routing(N, [T, T], K, E, 51, p_mask=0.1)
    idx = [i.to(dev) for i, _ in routing]
    wts = [w.to(dev) for _, w in routing]
    R = ranks.R
    table = torch.empty(N, E, dtype=torch.int32, device=dev)
    tc = [torch.empty(E // N, dtype=torch.int32, device=dev) for _ in range(N)]
    bufs = {k: [sentinel_tensor((R, H), "bf16", dev) for _ in range(N)] for k in ("recv", "eo", "gexp", "gr")}
    for q in range(N):
        bufs["eo"][q].copy_(wl.bf16_normal(R, H, seed=700 + q).to(dev))
        bufs["gr"][q].copy_(wl.bf16_normal(R, H, seed=710 + q).to(dev))
    rw = [torch.zeros(R, dtype=torch.float32, device=dev) for _ in range(N)]
    gw = [wl.f32_normal(R, 720 + q).to(dev) for q in range(N)]
    tab = {k: ep.pointer_table(v, dev) for k, v in list(bufs.items()) + [("rw", rw), ("gw", gw)]}
    tok = [wl.bf16_normal(T, H, seed=730 + r).to(dev) for r in range(N)]
    gres = [wl.bf16_normal(T, H, seed=740 + r).to(dev) for r in range(N)]
    res = [sentinel_tensor((T, H), "bf16", dev) for _ in range(N)]
    gtok = [sentinel_tensor((T, H), "bf16", dev) for _ in range(N)]
    gtw = [torch.full((T, K), -3.0, dtype=torch.float32, device=dev) for _ in range(N)]
    s = torch.cuda.Stream()

    def step():
        for r in range(N):
            ep.ep_shard_count(ranks.h[r], idx[r], table[r], stream=s)
        for r in range(N):
            ep.ep_shard_prepare(ranks.h[r], idx[r], table, tc[r], A, stream=s)
        for r in range(N):
            ep.ep_shard_dispatch(ranks.h[r], tok[r], wts[r], tab["recv"], tab["rw"], stream=s)
            ep.ep_shard_combine_bwd(ranks.h[r], gres[r], tab["gexp"], stream=s)
        for r in range(N):
            ep.ep_shard_combine(ranks.h[r], tab["eo"], res[r], stream=s)
            ep.ep_shard_dispatch_bwd(ranks.h[r], tab["gr"], tab["gw"], gtok[r], gtw[r], stream=s)

    def snapshot():
        torch.cuda.synchronize()
        return [bits(x) for x in bufs["recv"] + bufs["gexp"] + res + gtok] + [x.cpu().numpy() for x in gtw]

    with torch.cuda.stream(s):
        step()
    eager = snapshot()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for _ in range(2):
        for b in bufs["recv"] + bufs["gexp"] + res + gtok:  # back to the state before the eager step
            b.copy_(sentinel_tensor(tuple(b.shape), "bf16", dev))
        for x in gtw:
            x.fill_(-3.0)
        g.replay()
        assert all(np.array_equal(a, b) for a, b in zip(eager, snapshot()))
    # new routing in the same index buffers: the replay follows it
    routing2 = _routing(N, [T, T], K, E, 52, p_mask=0.2)
    for r in range(N):
        idx[r].copy_(routing2[r][0].to(dev))
        wts[r].copy_(routing2[r][1].to(dev))
    g.replay()
    torch.cuda.synchronize()
    sr = oracle_mod.shard_prepare([i.numpy() for i, _ in routing2], E, A, N, R)
    comb = oracle_mod.shard_combine(sr, [bits(bufs["eo"][q])[:max(int(sr.P[q]), 1)] for q in range(N)])
    disp = oracle_mod.shard_dispatch(sr, [bits(t) for t in tok], [w.numpy() for _, w in routing2])
    for r in range(N):
        assert same(bits(res[r]), comb[r])
    for q in range(N):
        assert same(bits(bufs["recv"][q])[:int(sr.P[q])], disp[q][0])


def test_shard_large_batches_on_the_wide_cluster(ep, oracle_mod):
    """Two ranks of up to 16,384 tokens at E=256, K=8 (131,072 routes on the
    first: the 16-CTA routing cluster of the sharded modes): maps and rows
    bit-exact against the oracle."""
    N, E, K, H, A, T = 2, 256, 8, 16, 128, 16384
    routing = _routing(N, [T, T - 5], K, E, 61, p_mask=0.05)
    ranks = Ranks(ep, N, E, K, H, T, A)
    sr = oracle_mod.shard_prepare([i.numpy() for i, _ in routing], E, A, N, ranks.R)
    pay = _payloads(sr, routing, H, "bf16", 61, oracle_mod)
    g = ranks.step(routing, A, pay)
    _check(g, sr, routing, pay, oracle_mod, "bf16", ranks.R)


def test_exchange_counts_over_nccl_single_rank(ep):
    """The binding's counts exchange on the production collective: an NCCL
    group of one rank on this GPU gathers the device counts into [1, E]."""
    import socket
    import torch.distributed as dist
    if dist.is_initialized():
        pytest.skip("a process group is already initialised")
    sock = socket.socket()
    sock.bind(("127.0.0.1", 0))
    port = sock.getsockname()[1]
    sock.close()
    store = dist.TCPStore("127.0.0.1", port, 1, True)
    dist.init_process_group("nccl", store=store, rank=0, world_size=1)
    try:
        E = 16
        lid, size = ep.ep_register_layer_sharded(E, 2, 32, 64, 1, 0)
        h = ep.alloc_handle(lid, size)
        idx, _ = wl.random_routing(64, 2, E, seed=71, p_mask=0.1)
        local = torch.empty(E, dtype=torch.int32, device="cuda")
        ep.ep_shard_count(h, idx.cuda(), local)
        table = ep.exchange_counts(local)
        v = idx.numpy().reshape(-1)
        assert table.shape == (1, E) and table.device.type == "cuda"
        assert table.cpu().numpy()[0].tolist() == np.bincount(v[v >= 0], minlength=E).tolist()
    finally:
        dist.destroy_process_group()
