"""GPU parity: libep's CUDA path against the CPU oracle, bit for bit.

Every output of the five calls is compared element by element with the
oracle on the same seeded inputs: token_counts, padded offsets, the slot map,
recv_tokens / recv_topk_weights rows [0, P), result, grad_expert_out rows
[0, P), grad_tokens and grad_topk_weights; rows at or beyond P must stay
untouched.  All five workload shapes run at full size, through the same
calls (and so the same launch configuration) that bench.py times.

Operations: TransformerEngine PR #3034, "Expert Parallelism: common C API +
NCCL EP backend", section "Per-step (allocation-free, CUDA-graph
capturable)".  Test list modelled on TransformerEngine PR #3035, section
"Testing" (prepare correctness, round trip, bit stability over iterations,
CUDA graph capture, several buffers in flight, index validation).
"""
import numpy as np
import pytest
import torch

from combine_ep_prepare_gb300 import workloads as wl
from ep_harness import (GpuLayer, assert_step_equal, bits, custom_inputs, gpu_step,
                        oracle_step, workload_inputs, SENTINEL)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_ep_prepare_gb300 as ep
    return ep


@pytest.mark.parametrize("name", ["tiny", "mixtral", "qwen3", "dsv3", "decode"])
def test_workload_parity(ep, oracle_mod, name):
    w = wl.WORKLOADS[name]
    inp = workload_inputs(w, oracle_mod)
    layer = GpuLayer(ep, w.E, w.K, w.H, w.T, w.A)
    assert layer.R == w.worst_case_rows()
    g = gpu_step(ep, layer, inp)
    o = oracle_step(inp, oracle_mod, layer.R)
    assert o["status"] == 0
    assert_step_equal(g, o, layer.R)


@pytest.mark.parametrize("case", [
    # (T, K, E, H, A, p_mask, p_bad, distinct, seed)
    (1, 1, 1, 8, 1, 0.0, 0.0, False, 1),          # smallest everything
    (3, 2, 5, 200, 3, 0.2, 0.0, False, 2),        # ragged row (25 vectors), A not a power of 2
    (1100, 1, 7, 64, 3, 0.1, 0.0, False, 18),     # two-CTA cluster prepare, ragged chunk
    (4097, 1, 7, 64, 5, 0.0, 0.0, False, 3),      # five-CTA cluster, one route in the last
    (5000, 3, 37, 136, 7, 0.1, 0.0, False, 4),    # eight-CTA cluster, duplicates allowed
    # Prepare runs as one cluster launch up to 65,536 routes, above that as one
    # grid-wide cooperative launch of G CTAs x W warps x up to 512 routes
    # (W = 16 up to 256 experts, 6 at 1024; G at most one per SM, 152 on a
    # GB300, and at most 65,536 / E rounded up to 4), else as three kernels.
    # Where the grid-wide launch is not available, the cluster takes up to
    # C x W x 512 routes (C = 16 CTAs where the device runs a 16-CTA cluster,
    # else 8).
    (9001, 4, 37, 16, 5, 0.1, 0.01, False, 11),   # wide cluster, ragged last CTA
    (40000, 1, 3, 8, 2, 0.0, 0.0, False, 12),     # wide cluster, few experts
    (32769, 1, 128, 8, 2, 0.05, 0.0, False, 15),  # past 256 routes per warp at 8 CTAs
    (8192, 8, 128, 16, 4, 0.0, 0.0, True, 16),    # 65,536 routes: the last cluster batch
    (65537, 1, 128, 8, 4, 0.05, 0.0, False, 17),  # one route more: grid-wide, ragged last CTA
    (33000, 4, 37, 16, 5, 0.1, 0.01, False, 13),  # grid-wide, invalid indices
    (140001, 1, 3, 8, 2, 0.0, 0.0, False, 14),    # grid-wide, few experts
    (16384, 8, 128, 8, 4, 0.0, 0.0, True, 19),    # grid-wide, 131,072 routes
    (131073, 1, 128, 8, 4, 0.05, 0.0, False, 20), # grid-wide, ragged
    (40000, 4, 1024, 8, 16, 0.1, 0.0, False, 24), # grid-wide at 1024 experts: 60 CTAs of 6 warps
    (1245184, 1, 3, 8, 2, 0.0, 0.0, False, 25),   # 152 x 16 x 512: the last grid-wide batch on a GB300
    (1245185, 1, 3, 8, 2, 0.0, 0.0, False, 26),   # one route more: three kernels
    (2048, 8, 1024, 16, 16, 0.3, 0.0, True, 5),   # largest expert count
    (300, 32, 64, 24, 4, 0.1, 0.0, False, 6),     # largest top-k
    (700, 4, 9, 40, 1000, 0.0, 0.0, False, 7),    # alignment larger than any count
    (1500, 4, 12, 32, 8, 1.0, 0.0, False, 8),     # every route masked
    (900, 3, 6, 48, 4, 0.1, 0.05, False, 9),      # invalid indices: flagged, treated as masked
    (64, 8, 3, 8, 2, 0.0, 0.0, False, 10),        # heavy repeats of few experts
    (700, 2, 9, 4608, 8, 0.1, 0.0, False, 21),    # rows over 8 KB: 4 KB scatter items, 2.25 per row
    (400, 3, 11, 4112, 4, 0.1, 0.0, False, 22),   # last 4 KB item of a row holds one 32-byte vector
])
def test_edge_parity(ep, oracle_mod, case):
    T, K, E, H, A, p_mask, p_bad, distinct, seed = case
    idx, wts = wl.random_routing(T, K, E, seed=100 + seed, p_mask=p_mask, p_bad=p_bad,
                                 distinct=distinct)
    inp = custom_inputs(idx, wts, E, H, A, oracle_mod, seed=200 + 10 * seed)
    layer = GpuLayer(ep, E, K, H, T, max(A, 1))
    g = gpu_step(ep, layer, inp)
    o = oracle_step(inp, oracle_mod, layer.R)
    if p_bad > 0:
        assert o["status"] & ep.EP_ST_BAD_INDEX
    assert_step_equal(g, o, layer.R)


def test_zero_tokens(ep, oracle_mod):
    E, K, H = 6, 2, 32
    idx = torch.zeros((0, K), dtype=torch.int64)
    wts = torch.zeros((0, K), dtype=torch.float32)
    inp = custom_inputs(idx, wts, E, H, 4, oracle_mod, seed=900)
    layer = GpuLayer(ep, E, K, H, 16, 4)
    g = gpu_step(ep, layer, inp)
    o = oracle_step(inp, oracle_mod, layer.R)
    assert_step_equal(g, o, layer.R)
    assert g["info"]["used_rows"] == 0


def test_no_weight_gradient(ep, oracle_mod):
    w = wl.WORKLOADS["tiny"]
    inp = workload_inputs(w, oracle_mod, with_weight_grad=False)
    layer = GpuLayer(ep, w.E, w.K, w.H, w.T, w.A)
    g = gpu_step(ep, layer, inp)
    o = oracle_step(inp, oracle_mod, layer.R)
    assert np.all(o["grad_topk_weights"] == 0)
    assert_step_equal(g, o, layer.R)


def test_overflow_writes_nothing(ep, oracle_mod):
    E, K, H, A, T = 5, 2, 64, 8, 200
    idx, wts = wl.random_routing(T, K, E, seed=31)
    inp = custom_inputs(idx, wts, E, H, A, oracle_mod, seed=310)
    P = oracle_mod.prepare(idx.numpy(), E, A).P
    layer = GpuLayer(ep, E, K, H, T, A, recv_capacity=P - 1)
    g = gpu_step(ep, layer, inp)
    assert g["info"]["status"] & ep.EP_ST_OVERFLOW
    o = oracle_step(inp, oracle_mod, layer.R)
    assert_step_equal(g, o, layer.R)  # counts / offsets / slots still exact
    assert np.all(g["recv_tokens"] == SENTINEL)
    assert np.all(g["grad_expert_out"] == SENTINEL)
    assert np.all(g["result"] == SENTINEL) and np.all(g["grad_tokens"] == SENTINEL)
    # exactly enough capacity: no overflow
    layer2 = GpuLayer(ep, E, K, H, T, A, recv_capacity=P)
    g2 = gpu_step(ep, layer2, inp)
    assert_step_equal(g2, oracle_step(inp, oracle_mod, layer2.R), layer2.R)


def test_token_count_mismatch_flagged(ep, oracle_mod):
    w = wl.WORKLOADS["tiny"]
    idx, wts = wl.routing(w)
    layer = GpuLayer(ep, w.E, w.K, w.H, w.T, w.A)
    h = layer.handle()
    counts = torch.empty(w.E, dtype=torch.int32, device="cuda")
    ep.ep_prepare(h, idx.cuda(), counts, w.A)
    eo = torch.zeros(layer.R, w.H, dtype=torch.bfloat16, device="cuda")
    res = torch.full((w.T - 1, w.H), 7.0, dtype=torch.bfloat16, device="cuda")
    ep.ep_combine(h, eo, res)  # one token fewer than prepared
    info = ep.ep_read_info(h)
    assert info["status"] & ep.EP_ST_TOKENS_MISMATCH
    assert torch.all(res == 7.0)


def test_repeat_bit_stable(ep, oracle_mod):
    w = wl.WORKLOADS["qwen3"]
    inp = workload_inputs(w, oracle_mod, T=1024)
    layer = GpuLayer(ep, w.E, w.K, w.H, 1024, w.A)
    h = layer.handle()
    a = gpu_step(ep, layer, inp, handle=h)
    for _ in range(3):
        b = gpu_step(ep, layer, inp, handle=h)
        for key in ("slot", "recv_tokens", "result", "grad_expert_out", "grad_tokens",
                    "grad_topk_weights"):
            assert np.array_equal(np.asarray(a[key]), np.asarray(b[key])), key


def test_interleaved_handles(ep, oracle_mod):
    """Three handles of one layer in flight (pipeline microbatches): prepare
    all three, then run the rest interleaved; each matches its own oracle."""
    E, K, H, A, T = 16, 4, 64, 8, 500
    layer = GpuLayer(ep, E, K, H, T, A)
    inps, hs, counts, idxs = [], [], [], []
    for i in range(3):
        idx, wts = wl.random_routing(T, K, E, seed=400 + i, p_mask=0.1 * i)
        inps.append(custom_inputs(idx, wts, E, H, A, oracle_mod, seed=4000 + 10 * i))
        hs.append(layer.handle())
        counts.append(torch.empty(E, dtype=torch.int32, device="cuda"))
        idxs.append(idx.cuda())
    for i in range(3):
        ep.ep_prepare(hs[i], idxs[i], counts[i], A)
    outs = []
    for i in (2, 0, 1):
        outs.append((i, gpu_step_after_prepare(ep, layer, inps[i], hs[i], idxs[i])))
    for i, g in outs:
        o = oracle_step(inps[i], oracle_mod, layer.R)
        P = o["P"]
        assert np.array_equal(g["recv_tokens"][:P], o["recv_tokens"])
        assert np.array_equal(g["result"], o["result"])
        assert np.array_equal(g["grad_tokens"], o["grad_tokens"])
        assert np.array_equal(g["grad_expert_out"][:P], o["grad_expert_out"])
        assert np.array_equal(counts[i].cpu().numpy(), o["counts"])


def gpu_step_after_prepare(ep, layer, inp, h, idx_dev):
    R, H, T, K = layer.R, inp.H, inp.T, inp.K
    recv = torch.empty(R, H, dtype=torch.bfloat16, device="cuda")
    recv_w = torch.empty(R, dtype=torch.float32, device="cuda")
    eo = torch.zeros(R, H, dtype=torch.bfloat16, device="cuda")
    eo[: inp.expert_out.shape[0]] = inp.expert_out.cuda()
    gr = torch.zeros(R, H, dtype=torch.bfloat16, device="cuda")
    gr[: inp.grad_recv.shape[0]] = inp.grad_recv.cuda()
    res = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    gexp = torch.empty(R, H, dtype=torch.bfloat16, device="cuda")
    gtok = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    gtw = torch.empty(T, K, dtype=torch.float32, device="cuda")
    ep.ep_dispatch(h, idx_dev, inp.tokens.cuda(), inp.topk_weights.cuda(), recv, recv_w)
    ep.ep_combine(h, eo, res)
    ep.ep_combine_bwd(h, inp.grad_result.cuda(), gexp)
    ep.ep_dispatch_bwd(h, gr, None, gtok, gtw)
    torch.cuda.synchronize()
    return {"recv_tokens": bits(recv), "result": bits(res), "grad_expert_out": bits(gexp),
            "grad_tokens": bits(gtok)}


def test_cuda_graph_decode(ep, oracle_mod):
    """The decode step captured whole in a CUDA graph: replays are bit-stable,
    and a replay after new routing and new token values is exact against the
    oracle for the new inputs (the routing map is rebuilt inside the graph)."""
    w = wl.WORKLOADS["decode"]
    inp = workload_inputs(w, oracle_mod)
    layer = GpuLayer(ep, w.E, w.K, w.H, w.T, w.A)
    R, T, H, K = layer.R, w.T, w.H, w.K
    h = layer.handle()
    d = {
        "idx": inp.topk_idx.cuda(), "wts": inp.topk_weights.cuda(), "tok": inp.tokens.cuda(),
        "eo": torch.zeros(R, H, dtype=torch.bfloat16, device="cuda"),
        "gres": inp.grad_result.cuda(),
        "grecv": torch.zeros(R, H, dtype=torch.bfloat16, device="cuda"),
        "counts": torch.empty(w.E, dtype=torch.int32, device="cuda"),
        "recv": torch.empty(R, H, dtype=torch.bfloat16, device="cuda"),
        "recv_w": torch.empty(R, dtype=torch.float32, device="cuda"),
        "res": torch.empty(T, H, dtype=torch.bfloat16, device="cuda"),
        "gexp": torch.empty(R, H, dtype=torch.bfloat16, device="cuda"),
        "gtok": torch.empty(T, H, dtype=torch.bfloat16, device="cuda"),
        "gtw": torch.empty(T, K, dtype=torch.float32, device="cuda"),
    }
    n = inp.expert_out.shape[0]
    d["eo"][:n] = inp.expert_out.cuda()
    d["grecv"][:n] = inp.grad_recv.cuda()
    s = torch.cuda.Stream()

    def step():
        ep.ep_prepare(h, d["idx"], d["counts"], w.A, stream=s)
        ep.ep_dispatch(h, d["idx"], d["tok"], d["wts"], d["recv"], d["recv_w"], stream=s)
        ep.ep_combine(h, d["eo"], d["res"], stream=s)
        ep.ep_combine_bwd(h, d["gres"], d["gexp"], stream=s)
        ep.ep_dispatch_bwd(h, d["grecv"], None, d["gtok"], d["gtw"], stream=s)

    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    snaps = []
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        snaps.append([bits(d["res"]), bits(d["gtok"]), bits(d["recv"]), d["counts"].cpu().numpy()])
    for a in snaps[1:]:
        for x, y in zip(snaps[0], a):
            assert np.array_equal(x, y)
    o = oracle_step(inp, oracle_mod, R)
    P = o["P"]
    assert np.array_equal(snaps[0][0], o["result"])
    assert np.array_equal(snaps[0][1], o["grad_tokens"])
    assert np.array_equal(snaps[0][2][:P], o["recv_tokens"])
    # new routing + new values, same shapes: the replay follows the inputs
    idx2, wts2 = wl.random_routing(T, K, w.E, seed=777, p_mask=0.5, distinct=True)
    inp2 = custom_inputs(idx2, wts2, w.E, H, w.A, oracle_mod, seed=7770, with_weight_grad=False)
    d["idx"].copy_(idx2.cuda())
    d["wts"].copy_(wts2.cuda())
    d["tok"].copy_(inp2.tokens.cuda())
    n2 = inp2.expert_out.shape[0]
    d["eo"][:n2] = inp2.expert_out.cuda()
    d["grecv"][:n2] = inp2.grad_recv.cuda()
    d["gres"].copy_(inp2.grad_result.cuda())
    g.replay()
    torch.cuda.synchronize()
    o2 = oracle_step(inp2, oracle_mod, R)
    assert np.array_equal(bits(d["res"]), o2["result"])
    assert np.array_equal(bits(d["gtok"]), o2["grad_tokens"])
    assert np.array_equal(bits(d["recv"])[: o2["P"]], o2["recv_tokens"])
    assert np.array_equal(bits(d["gexp"])[: o2["P"]], o2["grad_expert_out"])
    assert np.array_equal(d["counts"].cpu().numpy(), o2["counts"])


def test_arch_and_launches(ep):
    before = ep.ep_launch_count()
    w = wl.WORKLOADS["tiny"]
    layer = GpuLayer(ep, w.E, w.K, w.H, w.T, w.A)
    h = layer.handle()
    idx, _ = wl.routing(w)
    ep.ep_prepare(h, idx.cuda(), torch.empty(w.E, dtype=torch.int32, device="cuda"), w.A)
    torch.cuda.synchronize()
    assert ep.ep_launch_count() == before + 1  # tiny: the one-CTA prepare
    assert torch.cuda.get_device_capability() == (10, 3)


def test_payloads_16_byte_aligned_only(ep, oracle_mod):
    """Payload buffers that start 16 bytes past a 32-byte boundary (the
    kernels then use 16-byte vectors even though H % 16 == 0)."""
    w = wl.WORKLOADS["qwen3"]
    T, H = 512, w.H
    inp = workload_inputs(w, oracle_mod, T=T)
    layer = GpuLayer(ep, w.E, w.K, H, T, w.A)
    R = layer.R
    h = layer.handle()

    def off16(rows, cols, dtype=torch.bfloat16):
        raw = torch.zeros(rows * cols + 8, dtype=dtype, device="cuda")
        t = raw[8:].view(rows, cols)
        assert t.data_ptr() % 32 == 16
        return t

    tok = off16(T, H)
    tok.copy_(inp.tokens.cuda())
    recv = off16(R, H)
    gexp = off16(R, H)
    gres = off16(T, H)
    gres.copy_(inp.grad_result.cuda())
    idx = inp.topk_idx.cuda()
    counts = torch.empty(w.E, dtype=torch.int32, device="cuda")
    recv_w = torch.empty(R, dtype=torch.float32, device="cuda")
    ep.ep_prepare(h, idx, counts, w.A)
    ep.ep_dispatch(h, idx, tok, inp.topk_weights.cuda(), recv, recv_w)
    ep.ep_combine_bwd(h, gres, gexp)
    torch.cuda.synchronize()
    o = oracle_step(inp, oracle_mod, R)
    P = o["P"]
    assert np.array_equal(bits(recv)[:P], o["recv_tokens"])
    assert np.array_equal(bits(gexp)[:P], o["grad_expert_out"])


def test_large_full_step(ep, oracle_mod):
    """2^20 routes (65536 tokens x top-16 over 64 experts): the three-kernel
    prepare with many routes per lane, and every row call, bit for bit."""
    T, K, E, H, A = 65536, 16, 64, 8, 8
    idx, wts = wl.random_routing(T, K, E, seed=990, p_mask=0.05)
    inp = custom_inputs(idx, wts, E, H, A, oracle_mod, seed=9900)
    layer = GpuLayer(ep, E, K, H, T, A)
    g = gpu_step(ep, layer, inp)
    o = oracle_step(inp, oracle_mod, layer.R)
    assert_step_equal(g, o, layer.R)


def test_maximum_routes_prepare(ep, oracle_mod):
    """The registration limit: 2^24 routes (2^20 tokens x top-16)."""
    T, K, E, A = 1 << 20, 16, 64, 8
    idx, _ = wl.random_routing(T, K, E, seed=991, p_mask=0.05)
    layer = GpuLayer(ep, E, K, 8, T, A)
    h = layer.handle()
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    ep.ep_prepare(h, idx.cuda(), counts, A)
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    slots = torch.empty(T, K, dtype=torch.int32, device="cuda")
    ep.ep_expert_offsets(h, offsets)
    ep.ep_token_slots(h, slots)
    info = ep.ep_read_info(h)
    rt = oracle_mod.prepare(idx.numpy(), E, A, layer.R)
    assert info["status"] == 0 and info["used_rows"] == rt.P
    assert np.array_equal(counts.cpu().numpy(), rt.token_counts)
    assert np.array_equal(offsets.cpu().numpy(), rt.offsets)
    assert np.array_equal(slots.cpu().numpy(), rt.slot)


@pytest.mark.parametrize("fill", [0x00, 0xFF])
def test_unprepared_handle_writes_nothing(ep, fill):
    """Row calls on handle memory no prepare has written (zero-filled, or
    arbitrary bytes) write nothing, and ep_read_info reports it."""
    E, K, H, T = 8, 2, 64, 32
    layer = GpuLayer(ep, E, K, H, T, 4)
    h = layer.handle()
    h.mem.fill_(fill)
    idx, wts = wl.random_routing(T, K, E, seed=991)
    tok = wl.bf16_normal(T, H, seed=992).cuda()
    recv = torch.full((layer.R, H), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    recv_w = torch.full((layer.R,), -3.0, dtype=torch.float32, device="cuda")
    res = torch.full((T, H), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    eo = wl.bf16_normal(layer.R, H, seed=993).cuda()
    ep.ep_dispatch(h, idx.cuda(), tok, wts.cuda(), recv, recv_w)
    ep.ep_combine(h, eo, res)
    info = ep.ep_read_info(h)
    assert info["status"] == ep.EP_ST_NOT_PREPARED
    assert np.all(bits(recv) == SENTINEL) and np.all(bits(res) == SENTINEL)
    assert torch.all(recv_w == -3.0)


def test_two_streams_concurrently(ep, oracle_mod):
    """Two layers' steps enqueued on two streams at once, one on the
    one-launch prepare and one on the three-kernel prepare (each handle has
    its own state, the chunked scan's ticket included): each matches its own
    oracle bit for bit."""
    cases = [(5000, 2, 16, 64, 8, 0.1, 601), (140001, 1, 3, 8, 2, 0.0, 602)]  # T, K, E, H, A, p_mask, seed
    runs = []
    for T, K, E, H, A, p_mask, seed in cases:
        idx, wts = wl.random_routing(T, K, E, seed=seed, p_mask=p_mask)
        inp = custom_inputs(idx, wts, E, H, A, oracle_mod, seed=10 * seed)
        layer = GpuLayer(ep, E, K, H, T, A)
        R, rows = layer.R, inp.expert_out.shape[0]
        d = {"idx": idx.cuda(), "wts": wts.cuda(), "tok": inp.tokens.cuda(), "gres": inp.grad_result.cuda(),
             "counts": torch.empty(E, dtype=torch.int32, device="cuda"),
             "recv": torch.empty(R, H, dtype=torch.bfloat16, device="cuda"),
             "recv_w": torch.empty(R, dtype=torch.float32, device="cuda"),
             "eo": torch.zeros(R, H, dtype=torch.bfloat16, device="cuda"),
             "grecv": torch.zeros(R, H, dtype=torch.bfloat16, device="cuda"),
             "grecv_w": torch.zeros(R, dtype=torch.float32, device="cuda"),
             "res": torch.empty(T, H, dtype=torch.bfloat16, device="cuda"),
             "gexp": torch.empty(R, H, dtype=torch.bfloat16, device="cuda"),
             "gtok": torch.empty(T, H, dtype=torch.bfloat16, device="cuda"),
             "gtw": torch.empty(T, K, dtype=torch.float32, device="cuda")}
        d["eo"][:rows] = inp.expert_out.cuda()
        d["grecv"][:rows] = inp.grad_recv.cuda()
        d["grecv_w"][:rows] = inp.grad_recv_w.cuda()
        runs.append((inp, layer, layer.handle(), d, A))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    calls = []
    for (inp, layer, h, d, A), s in zip(runs, streams):
        calls.append([
            lambda h=h, d=d, A=A, s=s: ep.ep_prepare(h, d["idx"], d["counts"], A, stream=s),
            lambda h=h, d=d, s=s: ep.ep_dispatch(h, d["idx"], d["tok"], d["wts"], d["recv"], d["recv_w"], stream=s),
            lambda h=h, d=d, s=s: ep.ep_combine(h, d["eo"], d["res"], stream=s),
            lambda h=h, d=d, s=s: ep.ep_combine_bwd(h, d["gres"], d["gexp"], stream=s),
            lambda h=h, d=d, s=s: ep.ep_dispatch_bwd(h, d["grecv"], d["grecv_w"], d["gtok"], d["gtw"], stream=s)])
    for step in zip(*calls):  # interleave the two streams' launches
        for f in step:
            f()
    torch.cuda.synchronize()
    for inp, layer, h, d, A in runs:
        o = oracle_step(inp, oracle_mod, layer.R)
        P = o["P"]
        assert np.array_equal(d["counts"].cpu().numpy(), o["counts"])
        assert np.array_equal(bits(d["recv"])[:P], o["recv_tokens"])
        assert np.array_equal(d["recv_w"].cpu().numpy()[:P].view(np.uint32), o["recv_w"].view(np.uint32))
        assert np.array_equal(bits(d["res"]), o["result"])
        assert np.array_equal(bits(d["gexp"])[:P], o["grad_expert_out"])
        assert np.array_equal(bits(d["gtok"]), o["grad_tokens"])
        assert np.array_equal(d["gtw"].cpu().numpy().view(np.uint32), o["grad_topk_weights"].view(np.uint32))


# The timed-out marker a grid-wide prepare leaves in the handle header (word
# 6) when its wait gives up.  A valid cooperative launch cannot make the wait
# run out, so the test plants the marker from the host instead.
_TIMED_OUT_MARKER = 0x45505454


def _plant_marker(h):
    h.mem[24:28] = torch.tensor([_TIMED_OUT_MARKER], dtype=torch.int32).view(torch.uint8).to(h.mem.device)


def test_timed_out_handle_is_refused_until_zero_filled(ep, oracle_mod):
    """After a grid-wide wait gave up: ep_read_info reports EP_ST_TIMEOUT,
    the row calls write nothing, a grid-wide prepare does nothing on the
    handle, and once the memory is zero-filled the handle prepares again."""
    E, K, H, A, T = 3, 1, 8, 2, 100000  # 100,000 routes: the grid-wide routing map
    idx, wts = wl.random_routing(T, K, E, seed=951)
    layer = GpuLayer(ep, E, K, H, T, A)
    h = layer.handle()
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    ep.ep_prepare(h, idx.cuda(), counts, A)
    assert ep.ep_read_info(h)["status"] == 0
    _plant_marker(h)
    assert ep.ep_read_info(h)["status"] == ep.EP_ST_NOT_PREPARED | ep.EP_ST_TIMEOUT
    recv = torch.full((layer.R, H), SENTINEL, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    recv_w = torch.full((layer.R,), -3.0, dtype=torch.float32, device="cuda")
    tok = wl.bf16_normal(T, H, seed=952).cuda()
    ep.ep_dispatch(h, idx.cuda(), tok, wts.cuda(), recv, recv_w)
    ep.ep_prepare(h, idx.cuda(), counts, A)  # refused by the kernel: the marker stays
    info = ep.ep_read_info(h)
    assert info["status"] == ep.EP_ST_NOT_PREPARED | ep.EP_ST_TIMEOUT
    assert np.all(bits(recv) == SENTINEL) and torch.all(recv_w == -3.0)
    h.mem.zero_()
    ep.ep_prepare(h, idx.cuda(), counts, A)
    slots = torch.empty((T, K), dtype=torch.int32, device="cuda")
    ep.ep_token_slots(h, slots)
    rt = oracle_mod.prepare(idx.numpy(), E, A, layer.R)
    assert ep.ep_read_info(h)["status"] == 0
    assert np.array_equal(slots.cpu().numpy(), rt.slot)
