"""Time one libep call in isolation on a workload shape.

    python -m combine_ep_prepare_gb300.callbench --workload dsv3 --call prepare

Allocates only the buffers the call needs (for a row call: one prepare is
run first, outside the timing), then times --iters launches of the call with
CUDA events on the launching stream, each after an L2 flush and a short GPU
spin (so the host's enqueue cost is not timed).  Prints one JSON line: the
average duration, the call's algorithmic bytes and the achieved GB/s.

Meant for per-kernel tuning and for ncu captures of a single call; the whole
step is timed by bench.py.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import workloads as wl

CALLS = ("prepare", "dispatch", "combine", "combine_bwd", "dispatch_bwd", "combine_weighted",
         "combine_weighted_bwd")


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="mixtral", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--call", default="prepare", choices=CALLS)
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--dtype", choices=sorted(wl.TORCH_PAYLOAD), default="bf16")
    ap.add_argument("--tokens", type=int, default=0,
                    help="a smaller batch of the workload's shape (0: the workload's T)")
    args = ap.parse_args(argv)

    import combine_ep_prepare_gb300 as ep
    w = wl.WORKLOADS[args.workload]
    dev = torch.device("cuda", torch.cuda.current_device())
    T, H, E, K, A = w.T, w.H, w.E, w.K, w.A
    if args.tokens > 0:
        T = args.tokens
    lid, size = ep.ep_register_layer(E, K, H, T, A, dtype=args.dtype)
    pt = wl.TORCH_PAYLOAD[args.dtype]
    es = torch.empty(0, dtype=pt).element_size()
    R = ep.ep_recv_capacity(lid)
    h = ep.alloc_handle(lid, size, dev)
    idx_cpu, wts_cpu = wl.routing(w, T=T)
    idx, wts = idx_cpu.to(dev), wts_cpu.to(dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        ep.ep_prepare(h, idx, counts, A, stream=s)
    info = ep.ep_read_info(h, stream=s)
    P, npad = info["used_rows"], info["padding_rows"]
    V = P - npad

    if args.call == "prepare":
        fn = lambda: ep.ep_prepare(h, idx, counts, A, stream=s)  # noqa: E731
        nbytes = 8 * T * K + 4 * T * K + 12 * E + 4 + 4 * npad
    elif args.call == "dispatch":
        tok = wl.tokens(w, T=T, device=dev).to(pt)
        recv = torch.empty(R, H, dtype=pt, device=dev)
        rw = torch.empty(R, dtype=torch.float32, device=dev)
        fn = lambda: ep.ep_dispatch(h, idx, tok, wts, recv, rw, stream=s)  # noqa: E731
        nbytes = es * T * H + es * P * H + 8 * T * K + 4 * P + 4 * npad
    elif args.call == "combine_bwd":
        g = wl.grad_result(w, T=T, device=dev).to(pt)
        gexp = torch.empty(R, H, dtype=pt, device=dev)
        fn = lambda: ep.ep_combine_bwd(h, g, gexp, stream=s)  # noqa: E731
        nbytes = es * T * H + es * P * H + 4 * T * K + 4 * npad
    elif args.call == "combine":
        eo = wl.expert_out(w, R, device=dev).to(pt)
        res = torch.empty(T, H, dtype=pt, device=dev)
        fn = lambda: ep.ep_combine(h, eo, res, stream=s)  # noqa: E731
        nbytes = es * V * H + es * T * H + 4 * T * K
    elif args.call == "combine_weighted":
        eo = wl.expert_out(w, R, device=dev).to(pt)
        rw = wl.grad_recv_weights(w, R, device=dev)
        res = torch.empty(T, H, dtype=pt, device=dev)
        fn = lambda: ep.ep_combine_weighted(h, eo, rw, res, stream=s)  # noqa: E731
        nbytes = es * V * H + es * T * H + 4 * T * K + 4 * V
    elif args.call == "combine_weighted_bwd":
        g = wl.grad_result(w, T=T, device=dev).to(pt)
        eo = wl.expert_out(w, R, device=dev).to(pt)
        rw = wl.grad_recv_weights(w, R, device=dev)
        gexp = torch.empty(R, H, dtype=pt, device=dev)
        gw = torch.empty(R, dtype=torch.float32, device=dev)
        fn = lambda: ep.ep_combine_weighted_bwd(h, g, eo, rw, gexp, gw, stream=s)  # noqa: E731
        nbytes = es * T * H + es * V * H + es * P * H + 4 * T * K + 4 * V + 4 * P
    else:
        g = wl.grad_recv(w, R, device=dev).to(pt)
        gw = wl.grad_recv_weights(w, R, device=dev)
        gt = torch.empty(T, H, dtype=pt, device=dev)
        gtw = torch.empty(T, K, dtype=torch.float32, device=dev)
        fn = lambda: ep.ep_dispatch_bwd(h, g, gw, gt, gtw, stream=s)  # noqa: E731
        nbytes = es * V * H + es * T * H + 8 * T * K + 4 * V

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.int32, device=dev)
    spin = int(0.1e-3 * 2.07e9)
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
    print(json.dumps({"workload": w.name, "T": T, "call": args.call, "dtype": args.dtype, "iters": args.iters, "ms": ms,
                      "algorithmic_bytes": nbytes, "GB/s": nbytes / (ms * 1e-3) / 1e9}))


if __name__ == "__main__":
    main()
