"""Time libep calls in isolation on a workload shape.

    python -m combine_ep_prepare_gb300.callbench --workload dsv3 --call prepare
    python -m combine_ep_prepare_gb300.callbench --workload dsv3 --tokens 2048 --tight --call all
    python -m combine_ep_prepare_gb300.callbench --workload mixtral --ranks 2 --call all

Allocates only the buffers the calls need (for a row call: one prepare is
run first, outside the timing), then times --iters launches of each call
with CUDA events on the launching stream, each after an L2 flush and a
short GPU spin (so the host's enqueue cost is not timed).  Prints one JSON
line per call: the average duration, the call's algorithmic bytes and the
achieved GB/s.

--tokens   a smaller batch of the workload's shape;
--tight    receive capacity = the rows the batch uses (a first prepare on a
           probe layer gives them), instead of the worst case: the same
           kernels on a smaller device footprint, for profiler captures;
--ranks N  a sharded layer: N ranks' handles and receive buffers on this
           GPU, the batch split evenly over them; the calls of rank 0 are
           timed (the sharded kernel instances); with --rank-major, a
           rank-major layer (its prepare runs the owners and routing kernels,
           dispatch the ids and rows kernels, dispatch_bwd the rows and
           weight-gradient kernels);
--call all the five step calls, in step order, each timed on its own.

Meant for per-kernel tuning and for ncu captures of single calls; the whole
step is timed by bench.py.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import workloads as wl

CALLS = ("prepare", "dispatch", "combine", "combine_bwd", "dispatch_bwd", "combine_weighted",
         "combine_weighted_bwd")
STEP = ("prepare", "dispatch", "combine", "combine_bwd", "dispatch_bwd")


def _single(ep, w, T, args, dev, s):
    E, K, H, A = w.E, w.K, w.H, w.A
    pt = wl.TORCH_PAYLOAD[args.dtype]
    idx_cpu, wts_cpu = wl.routing(w, T=T)
    idx, wts = idx_cpu.to(dev), wts_cpu.to(dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    cap = 0
    if args.tight:
        lid, size = ep.ep_register_layer(E, K, H, T, A, dtype=args.dtype)
        probe = ep.alloc_handle(lid, size, dev)
        ep.ep_prepare(probe, idx, counts, A, stream=s)
        cap = max(1, ep.ep_read_info(probe, stream=s)["used_rows"])
        del probe
    lid, size = ep.ep_register_layer(E, K, H, T, A, recv_capacity=cap, dtype=args.dtype)
    R = ep.ep_recv_capacity(lid)
    h = ep.alloc_handle(lid, size, dev)
    with torch.cuda.stream(s):
        ep.ep_prepare(h, idx, counts, A, stream=s)
    info = ep.ep_read_info(h, stream=s)
    P, npad = info["used_rows"], info["padding_rows"]
    fns = {}
    need = set(STEP) if args.call == "all" else {args.call}
    if "prepare" in need:
        fns["prepare"] = lambda: ep.ep_prepare(h, idx, counts, A, stream=s)
    if "dispatch" in need:
        tok = wl.tokens(w, T=T, device=dev).to(pt)
        recv = torch.empty(R, H, dtype=pt, device=dev)
        rw = torch.empty(R, dtype=torch.float32, device=dev)
        fns["dispatch"] = lambda: ep.ep_dispatch(h, idx, tok, wts, recv, rw, stream=s)
    if "combine" in need:
        eo = wl.expert_out(w, R, device=dev).to(pt)
        res = torch.empty(T, H, dtype=pt, device=dev)
        fns["combine"] = lambda: ep.ep_combine(h, eo, res, stream=s)
    if "combine_bwd" in need:
        g = wl.grad_result(w, T=T, device=dev).to(pt)
        gexp = torch.empty(R, H, dtype=pt, device=dev)
        fns["combine_bwd"] = lambda: ep.ep_combine_bwd(h, g, gexp, stream=s)
    if "dispatch_bwd" in need:
        gr = wl.grad_recv(w, R, device=dev).to(pt)
        gw = wl.grad_recv_weights(w, R, device=dev)
        gt = torch.empty(T, H, dtype=pt, device=dev)
        gtw = torch.empty(T, K, dtype=torch.float32, device=dev)
        fns["dispatch_bwd"] = lambda: ep.ep_dispatch_bwd(h, gr, gw, gt, gtw, stream=s)
    if "combine_weighted" in need:
        eo2 = wl.expert_out(w, R, device=dev).to(pt)
        rw2 = wl.grad_recv_weights(w, R, device=dev)
        res2 = torch.empty(T, H, dtype=pt, device=dev)
        fns["combine_weighted"] = lambda: ep.ep_combine_weighted(h, eo2, rw2, res2, stream=s)
    if "combine_weighted_bwd" in need:
        g3 = wl.grad_result(w, T=T, device=dev).to(pt)
        eo3 = wl.expert_out(w, R, device=dev).to(pt)
        rw3 = wl.grad_recv_weights(w, R, device=dev)
        gexp3 = torch.empty(R, H, dtype=pt, device=dev)
        gw3 = torch.empty(R, dtype=torch.float32, device=dev)
        fns["combine_weighted_bwd"] = lambda: ep.ep_combine_weighted_bwd(h, g3, eo3, rw3, gexp3, gw3, stream=s)
    return fns, P, npad, P - npad


def _sharded(ep, w, T, args, dev, s):
    """N ranks of a sharded layer on this GPU; rank 0's calls."""
    E, K, H, A, N = w.E, w.K, w.H, w.A, args.ranks
    pt = wl.TORCH_PAYLOAD[args.dtype]
    tpr = T // N
    hs, idxs, wtss = [], [], []
    for r in range(N):
        lid, size = ep.ep_register_layer_sharded(E, K, H, tpr, N, r, max_alignment=A, dtype=args.dtype)
        hs.append(ep.alloc_handle(lid, size, dev))
        idx_cpu, wts_cpu = wl.routing(w, T=T)
        idxs.append(idx_cpu[r * tpr:(r + 1) * tpr].contiguous().to(dev))
        wtss.append(wts_cpu[r * tpr:(r + 1) * tpr].contiguous().to(dev))
    R = ep.ep_recv_capacity(lid)
    local = [torch.empty(E, dtype=torch.int32, device=dev) for _ in range(N)]
    tcs = [torch.empty(E // N, dtype=torch.int32, device=dev) for _ in range(N)]
    for r in range(N):
        ep.ep_shard_count(hs[r], idxs[r], local[r], stream=s)
    table = torch.stack(local).contiguous()
    for r in range(N):
        ep.ep_shard_prepare(hs[r], idxs[r], table, tcs[r], A, stream=s)
    info = ep.ep_read_info(hs[0], stream=s)
    bufs = {k: [torch.empty(R, H, dtype=pt, device=dev) for _ in range(N)] for k in ("recv", "eo", "gexp", "gr")}
    wb = {k: [torch.empty(R, dtype=torch.float32, device=dev) for _ in range(N)] for k in ("rw", "gw")}
    tab = {k: ep.pointer_table(v, dev) for k, v in list(bufs.items()) + list(wb.items())}
    tok = wl.tokens(w, T=tpr, device=dev).to(pt)
    g = wl.grad_result(w, T=tpr, device=dev).to(pt)
    res = torch.empty(tpr, H, dtype=pt, device=dev)
    gt = torch.empty(tpr, H, dtype=pt, device=dev)
    gtw = torch.empty(tpr, K, dtype=torch.float32, device=dev)
    h, idx = hs[0], idxs[0]
    fns = {"prepare": lambda: ep.ep_shard_prepare(h, idx, table, tcs[0], A, stream=s),
           "dispatch": lambda: ep.ep_shard_dispatch(h, tok, wtss[0], tab["recv"], tab["rw"], stream=s),
           "combine": lambda: ep.ep_shard_combine(h, tab["eo"], res, stream=s),
           "combine_bwd": lambda: ep.ep_shard_combine_bwd(h, g, tab["gexp"], stream=s),
           "dispatch_bwd": lambda: ep.ep_shard_dispatch_bwd(h, tab["gr"], tab["gw"], gt, gtw, stream=s)}
    if args.call != "all":
        fns = {args.call: fns[args.call]}
    P, npad = info["used_rows"], info["padding_rows"]
    # rank 0's own rows: an estimate of the bytes its calls move (rows land on every owner)
    return fns, P, npad, P - npad


def _rank_major(ep, w, T, args, dev, s):
    """N ranks of a rank-major layer on this GPU; rank 0's calls.  Before
    them: every rank's count, then every rank's prepare (4N launches)."""
    E, K, H, N = w.E, w.K, w.H, args.ranks
    pt = wl.TORCH_PAYLOAD[args.dtype]
    tpr = T // N
    idx_cpu, wts_cpu = wl.routing(w, T=T)
    idxs = [idx_cpu[r * tpr:(r + 1) * tpr].contiguous().to(dev) for r in range(N)]
    wtss = [wts_cpu[r * tpr:(r + 1) * tpr].contiguous().to(dev) for r in range(N)]
    hs = []
    for r in range(N):
        lid, size = ep.ep_register_layer_rank_major(E, K, H, tpr, N, r, dtype=args.dtype)
        hs.append(ep.alloc_handle(lid, size, dev))
    R = ep.ep_recv_capacity(lid)
    table = torch.empty(N, N, dtype=torch.int32, device=dev)
    rows = [torch.empty(1, dtype=torch.int32, device=dev) for _ in range(N)]
    for r in range(N):
        ep.ep_rank_major_count(hs[r], idxs[r], table[r], stream=s)
    for r in range(N):
        ep.ep_rank_major_prepare(hs[r], idxs[r], table, rows[r], stream=s)
    M0 = ep.ep_read_info(hs[0], stream=s)["used_rows"]
    bufs = {k: [torch.empty(R, H, dtype=pt, device=dev) for _ in range(N)] for k in ("recv", "part", "grecv", "gpart")}
    ids = [torch.empty(R, K, dtype=torch.int64, device=dev) for _ in range(N)]
    wb = {k: [torch.empty(R, K, dtype=torch.float32, device=dev) for _ in range(N)] for k in ("rw", "gw")}
    tab = {k: ep.pointer_table(v, dev) for k, v in list(bufs.items()) + list(wb.items()) + [("ids", ids)]}
    tok = wl.tokens(w, T=tpr, device=dev).to(pt)
    g = wl.grad_result(w, T=tpr, device=dev).to(pt)
    res = torch.empty(tpr, H, dtype=pt, device=dev)
    gt = torch.empty(tpr, H, dtype=pt, device=dev)
    gtw = torch.empty(tpr, K, dtype=torch.float32, device=dev)
    h, idx = hs[0], idxs[0]
    fns = {"prepare": lambda: ep.ep_rank_major_prepare(h, idx, table, rows[0], stream=s),
           "dispatch": lambda: ep.ep_rank_major_dispatch(h, idx, tok, wtss[0], tab["recv"], tab["ids"], tab["rw"],
                                                         stream=s),
           "combine": lambda: ep.ep_rank_major_combine(h, tab["part"], res, stream=s),
           "combine_bwd": lambda: ep.ep_rank_major_combine_bwd(h, g, tab["grecv"], stream=s),
           "dispatch_bwd": lambda: ep.ep_rank_major_dispatch_bwd(h, tab["gpart"], tab["gw"], gt, gtw, stream=s)}
    if args.call != "all":
        fns = {args.call: fns[args.call]}
    # rank 0's own received rows stand in for its rows (an estimate, as for --ranks)
    return fns, M0, 0, M0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="mixtral", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--call", default="prepare", choices=CALLS + ("all",))
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--dtype", choices=sorted(wl.TORCH_PAYLOAD), default="bf16")
    ap.add_argument("--tokens", type=int, default=0,
                    help="a smaller batch of the workload's shape (0: the workload's T)")
    ap.add_argument("--tight", action="store_true",
                    help="receive capacity = the rows the batch uses (smaller footprint)")
    ap.add_argument("--ranks", type=int, default=0, help="a sharded layer over this many ranks")
    ap.add_argument("--rank-major", action="store_true", help="with --ranks: the rank-major layout")
    args = ap.parse_args(argv)

    import combine_ep_prepare_gb300 as ep
    w = wl.WORKLOADS[args.workload]
    dev = torch.device("cuda", torch.cuda.current_device())
    T = args.tokens if args.tokens > 0 else w.T
    H, E, K = w.H, w.E, w.K
    es = torch.empty(0, dtype=wl.TORCH_PAYLOAD[args.dtype]).element_size()
    s = torch.cuda.Stream(device=dev)
    if args.ranks > 0 and args.rank_major:
        fns, P, npad, V = _rank_major(ep, w, T, args, dev, s)
        T = T // args.ranks
    elif args.ranks > 0:
        fns, P, npad, V = _sharded(ep, w, T, args, dev, s)
        T = T // args.ranks
    else:
        fns, P, npad, V = _single(ep, w, T, args, dev, s)
    nbytes = {
        "prepare": 8 * T * K + 4 * T * K + 12 * E + 4 + 4 * npad,
        "dispatch": es * T * H + es * P * H + 8 * T * K + 4 * P + 4 * npad,
        "combine_bwd": es * T * H + es * P * H + 4 * T * K + 4 * npad,
        "combine": es * V * H + es * T * H + 4 * T * K,
        "combine_weighted": es * V * H + es * T * H + 4 * T * K + 4 * V,
        "combine_weighted_bwd": es * T * H + es * V * H + es * P * H + 4 * T * K + 4 * V + 4 * P,
        "dispatch_bwd": es * V * H + es * T * H + 8 * T * K + 4 * V,
    }
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.int32, device=dev)
    spin = int(0.1e-3 * 2.07e9)
    for name, fn in fns.items():
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.iters)]
        with torch.cuda.stream(s):
            for _ in range(args.warmup):
                flush.zero_()
                fn()
            for a, b in evs:
                flush.zero_()
                torch.cuda._sleep(spin)
                a.record(s)
                fn()
                b.record(s)
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in evs) / len(evs)
        line = {"workload": w.name, "T": T, "call": name, "dtype": args.dtype, "iters": args.iters,
                "ms": ms, "algorithmic_bytes": nbytes[name], "GB/s": nbytes[name] / (ms * 1e-3) / 1e9}
        if args.ranks:
            line["ranks"] = args.ranks
            line["layout"] = "rank-major" if args.rank_major else "expert-major"
            line["bytes_note"] = "rank 0's token side and its own receive rows"
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
