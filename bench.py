#!/usr/bin/env python3
"""Benchmark of the MoE expert-parallel step on GB300 through libep.

One step = one pass of the whole path over one batch: ep_prepare,
ep_dispatch, ep_combine, ep_combine_bwd, ep_dispatch_bwd (forward and
backward of dispatch + combine), on seeded synthetic inputs shaped like the
workload named by --workload (default: the DeepSeek-V3-like layer, T=16384
tokens, H=7168, E=256 experts, top-8, group-limited routing, alignment 128,
the largest of the five workloads).

Prints ONE JSON line (rank 0), whose top level is the --workload step:
  value         tokens/s over all ranks, inputs resident in HBM, device-timed
                with CUDA events on the launching stream, L2 flushed between
                steps (the flush is outside the per-step events);
  roofline      the dominant kernel's algorithmic bytes per launch / its
                duration inside the chained step (the step's prefix through
                the call minus the prefix before it, both event-timed),
                against the measured HBM copy bandwidth; also the same over
                an event pair around the call alone;
  e2e           the same metric with every step's inputs copied from pinned
                host memory and the token-side outputs copied back, inside
                the timed region;
  cpu_baseline  the CPU oracle (single thread) on a bounded sample;
  gpu_launches  libep kernels launched in the timed region (library counter);
  workloads     the same device-timed measurements (step, graph replay,
                per-call durations and rooflines) for each workload of
                --also (default: Mixtral-like, Qwen3-MoE-like, decode, tiny),
                run after the headline in the same process, and for the
                DeepSeek-V3-like batch on a sharded layer of --sharded ranks
                emulated on this GPU, expert-major (dsv3_sharded8) and
                rank-major (dsv3_rank_major8).

--impl reference times the CPU oracle instead (the slow reference arm): same
metric, config and unit, each step a bounded sample of the workload.

Multi-GPU (torchrun): replicas only; each rank runs the same workload on its
own GPU with no data exchange (weak scaling); max step time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE dispatch+combine fwd+bwd tokens/s and achieved HBM GB/s vs ~8 TB/s"
UNIT = "tokens/s"
CALLS = ("prepare", "dispatch", "combine", "combine_bwd", "dispatch_bwd")
KERNEL_OF_CALL = {"prepare": "ep_route (prepare)", "dispatch": "ep_scatter_rows_kernel<weights>",
                  "combine": "ep_gather_sum_kernel", "combine_bwd": "ep_scatter_rows_kernel",
                  "dispatch_bwd": "ep_gather_sum_kernel<weights>"}
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["libep", "reference"], default="libep")
    ap.add_argument("--workload", default="dsv3",
                    choices=["tiny", "mixtral", "qwen3", "dsv3", "decode"])
    ap.add_argument("--also", default="mixtral,qwen3,decode,tiny",
                    help="comma-separated workloads measured after the headline and reported "
                         "under 'workloads' ('none' for none)")
    ap.add_argument("--sharded", type=int, default=8,
                    help="also time the DeepSeek-V3-like batch on a sharded layer of this many ranks "
                         "emulated on this GPU, under workloads (0: skip)")
    ap.add_argument("--dtype", choices=["bf16", "fp16", "fp32"], default="bf16",
                    help="payload type of the rows (the CPU-oracle legs run for bf16 only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="wall-clock budget of the CPU-baseline sample")
    return ap.parse_args()


# ----------------------------------------------------------------------------
# Algorithmic bytes per call (what the method must move)
# ----------------------------------------------------------------------------

def algorithmic_bytes(T, H, E, K, V, P, npad, es=2):
    """Bytes each call must move; es = payload element size (2 for bf16 / fp16, 4 for fp32)."""
    return {
        "prepare": 8 * T * K + 4 * T * K + 12 * E + 4 + 4 * npad,
        "dispatch": es * T * H + es * P * H + 4 * T * K * 2 + 4 * P + 4 * npad,
        "combine": es * V * H + es * T * H + 4 * T * K,
        "combine_bwd": es * T * H + es * P * H + 4 * T * K + 4 * npad,
        "dispatch_bwd": es * V * H + es * T * H + 4 * T * K * 2 + 4 * V,
    }


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_digest():
    """Digest of the kernel sources' code: comments and blank space are left
    out, so that a comment edit does not void the committed ncu counters."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "combine_ep_prepare_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(f.encode())
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def committed_traffic(call, workload, alg_bytes=None):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel sources changed since the counters were taken.

    A row for the workload itself is used as it is.  A row for a smaller
    batch of the same shape (workload field "<name>@T<tokens>", fifth field
    "alg=<algorithmic bytes of that launch>") is scaled to the full launch by
    the ratio of algorithmic bytes, alg_bytes / alg: the row kernels' DRAM
    traffic grows in proportion to the rows they move."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = source_digest()
    scaled = None
    with open(path) as f:
        for line in f:
            parts = line.split("#")[0].split()
            if len(parts) < 4 or parts[0] != call or parts[3] != digest:
                continue
            if parts[1] == workload:
                return float(parts[2])
            if (scaled is None and alg_bytes and parts[1].startswith(workload + "@")
                    and len(parts) >= 5 and parts[4].startswith("alg=")):
                scaled = float(parts[2]) * alg_bytes / float(parts[4][4:])
    return scaled


# ----------------------------------------------------------------------------
# Clocks
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ----------------------------------------------------------------------------

def oracle_inputs(w, T):
    import oracle
    from combine_ep_prepare_gb300 import workloads as wl
    idx, wts = wl.routing(w, T=T)
    rt = oracle.prepare(idx.numpy(), w.E, w.A)
    rows = max(rt.P, 1)

    def b(t):
        return t.contiguous().view(__import__("torch").int16).numpy().view("uint16")
    return {"idx": idx.numpy(), "wts": wts.numpy(), "tok": b(wl.tokens(w, T=T)),
            "eo": b(wl.expert_out(w, rows)), "gres": b(wl.grad_result(w, T=T)),
            "grecv": b(wl.grad_recv(w, rows)), "grecv_w": wl.grad_recv_weights(w, rows).numpy()}


def oracle_step(w, d):
    import oracle
    rt = oracle.prepare(d["idx"], w.E, w.A)
    oracle.dispatch(rt, d["tok"], d["wts"])
    oracle.combine(rt, d["eo"])
    oracle.combine_bwd(rt, d["gres"])
    oracle.dispatch_bwd(rt, d["grecv"], d["grecv_w"])


def oracle_sample_tokens(w, budget_s):
    """Largest token count (<= T) whose oracle step fits about budget_s / 4."""
    T = w.T
    d = oracle_inputs(w, min(T, 256))
    t0 = time.perf_counter()
    oracle_step(w, d)
    per_tok = (time.perf_counter() - t0) / min(T, 256)
    fit = int(max(64, min(T, (budget_s / 4) / max(per_tok, 1e-9))))
    return fit


def cpu_baseline(w, budget_s):
    import oracle
    oracle.build_oracle()
    Ts = oracle_sample_tokens(w, budget_s)
    d = oracle_inputs(w, Ts)
    n, t_total = 0, 0.0
    while t_total < budget_s and n < 100:
        t0 = time.perf_counter()
        oracle_step(w, d)
        t_total += time.perf_counter() - t0
        n += 1
    return {"value": n * Ts / t_total, "unit": UNIT, "cores": 1, "host_cores": os.cpu_count(),
            "kind": "oracle",
            "sample": "%d oracle steps of %d of the workload's %d tokens (same recipe), "
                      "single-threaded C, %.1f s" % (n, Ts, w.T, t_total)}


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.build_oracle()
    per_step_budget = 4.0
    Ts = oracle_sample_tokens(w, 4 * per_step_budget)
    d = oracle_inputs(w, Ts)
    for _ in range(args.warmup):
        oracle_step(w, d)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, d)
    dt = time.perf_counter() - t0
    value = args.steps * Ts / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(w, "none (CPU)"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "host_cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": "%d of %d tokens per step, single-threaded C oracle" % (Ts, w.T)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def reduce_max(x, device):
    """Max of a float over all ranks (timing only; no data-path exchange)."""
    import torch
    import torch.distributed as dist
    if not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_rank, world, ms_max):
    """Tokens/s of all ranks together, timed by the slowest rank."""
    return world * tokens_per_rank / (ms_max * 1e-3)


def workload_config(w, l2):
    return {"workload": "%s: T=%d H=%d E=%d K=%d A=%d (%s routing)" % (w.name, w.T, w.H, w.E, w.K, w.A, w.routing),
            "T": w.T, "H": w.H, "E": w.E, "K": w.K, "A": w.A, "l2": l2,
            "parallelism": "replicas (one independent step per GPU)"}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

class Step:
    """Device buffers of one workload's step and the five calls on them."""

    def __init__(self, torch, ep, w, dev, dtype):
        T, H, E, K, A = w.T, w.H, w.E, w.K, w.A
        self.w = w
        lid, mem_size = ep.ep_register_layer(E, K, H, T, A, dtype=dtype)
        self.R = R = ep.ep_recv_capacity(lid)
        self.h = h = ep.alloc_handle(lid, mem_size, dev)
        # Inputs: routing from the CPU recipe, payloads drawn on the device
        # (the same bf16 draws, converted for the fp16 / fp32 payload types).
        pt = wl_mod().TORCH_PAYLOAD[dtype]
        self.es = torch.empty(0, dtype=pt).element_size()
        wl = wl_mod()
        self.idx_cpu, self.wts_cpu = wl.routing(w)
        self.idx = idx = self.idx_cpu.to(dev)
        self.wts = wts = self.wts_cpu.to(dev)
        self.tok = tok = wl.tokens(w, device=dev).to(pt)
        self.eo = eo = wl.expert_out(w, R, device=dev).to(pt)
        self.gres = gres = wl.grad_result(w, device=dev).to(pt)
        self.grecv = grecv = wl.grad_recv(w, R, device=dev).to(pt)
        self.grecv_w = grecv_w = wl.grad_recv_weights(w, R, device=dev)
        self.counts = counts = torch.empty(E, dtype=torch.int32, device=dev)
        self.recv = recv = torch.empty(R, H, dtype=pt, device=dev)
        self.recv_w = recv_w = torch.empty(R, dtype=torch.float32, device=dev)
        self.res = res = torch.empty(T, H, dtype=pt, device=dev)
        self.gexp = gexp = torch.empty(R, H, dtype=pt, device=dev)
        self.gtok = gtok = torch.empty(T, H, dtype=pt, device=dev)
        self.gtw = gtw = torch.empty(T, K, dtype=torch.float32, device=dev)
        self.s = s = torch.cuda.Stream(device=dev)
        self.fns = (
            lambda: ep.ep_prepare(h, idx, counts, A, stream=s),
            lambda: ep.ep_dispatch(h, idx, tok, wts, recv, recv_w, stream=s),
            lambda: ep.ep_combine(h, eo, res, stream=s),
            lambda: ep.ep_combine_bwd(h, gres, gexp, stream=s),
            lambda: ep.ep_dispatch_bwd(h, grecv, grecv_w, gtok, gtw, stream=s),
        )


class ShardStep:
    """The same batch as Step, split evenly over `nranks` ranks of a sharded
    layer, all emulated on this GPU (each rank its own layer, handle and
    receive-side buffers; row calls through device tables of the ranks'
    buffer addresses).  Each of the five calls runs every rank's call; the
    counts exchange is each rank's ep_shard_count writing its row of one
    [N][E] table.  Receive buffers hold the rows this batch needs (the
    largest owner's P, from a first prepare)."""

    traffic_key = None  # the committed ncu rows are the single-buffer kernels'

    def __init__(self, torch, ep, w, dev, dtype, nranks):
        T, H, E, K, A = w.T, w.H, w.E, w.K, w.A
        N = nranks
        assert T % N == 0 and E % N == 0
        tpr = T // N
        self.w, self.N = w, N
        wl = wl_mod()
        pt = wl.TORCH_PAYLOAD[dtype]
        self.es = torch.empty(0, dtype=pt).element_size()
        idx_cpu, wts_cpu = wl.routing(w)
        idx = [idx_cpu[r * tpr:(r + 1) * tpr].contiguous().to(dev) for r in range(N)]
        wts = [wts_cpu[r * tpr:(r + 1) * tpr].contiguous().to(dev) for r in range(N)]
        table = torch.empty(N, E, dtype=torch.int32, device=dev)
        tc = [torch.empty(E // N, dtype=torch.int32, device=dev) for _ in range(N)]
        # a first prepare on worst-case layers gives every owner's P
        hs = []
        for r in range(N):
            lid, size = ep.ep_register_layer_sharded(E, K, H, tpr, N, r, max_alignment=A, dtype=dtype)
            hs.append(ep.alloc_handle(lid, size, dev))
        for r in range(N):
            ep.ep_shard_count(hs[r], idx[r], table[r])
        for r in range(N):
            ep.ep_shard_prepare(hs[r], idx[r], table, tc[r], A)
        infos = [ep.ep_read_info(h) for h in hs]
        R = max(1, max(i["used_rows"] for i in infos))
        self.P = sum(i["used_rows"] for i in infos)
        self.npad = sum(i["padding_rows"] for i in infos)
        self.h = []
        for r in range(N):
            lid, size = ep.ep_register_layer_sharded(E, K, H, tpr, N, r, max_alignment=A,
                                                     recv_capacity=R, dtype=dtype)
            self.h.append(ep.alloc_handle(lid, size, dev))
        self.R = R
        rows = lambda: [torch.empty(R, H, dtype=pt, device=dev) for _ in range(N)]  # noqa: E731
        recv, eo, gexp, grecv = rows(), rows(), rows(), rows()
        for q in range(N):
            eo[q].copy_(wl.expert_out(w, R, device=dev).to(pt))
            grecv[q].copy_(wl.grad_recv(w, R, device=dev).to(pt))
        recv_w = [torch.empty(R, dtype=torch.float32, device=dev) for _ in range(N)]
        grecv_w = [wl.grad_recv_weights(w, R, device=dev) for _ in range(N)]
        tab = {k: ep.pointer_table(v, dev) for k, v in
               (("recv", recv), ("recv_w", recv_w), ("eo", eo), ("gexp", gexp), ("grecv", grecv),
                ("grecv_w", grecv_w))}
        tok_all, gres_all = wl.tokens(w, device=dev).to(pt), wl.grad_result(w, device=dev).to(pt)
        tok = [tok_all[r * tpr:(r + 1) * tpr] for r in range(N)]
        gres = [gres_all[r * tpr:(r + 1) * tpr] for r in range(N)]
        res = [torch.empty(tpr, H, dtype=pt, device=dev) for _ in range(N)]
        gtok = [torch.empty(tpr, H, dtype=pt, device=dev) for _ in range(N)]
        gtw = [torch.empty(tpr, K, dtype=torch.float32, device=dev) for _ in range(N)]
        self.keep = (idx, wts, table, tc, recv, eo, gexp, grecv, recv_w, grecv_w, tab, tok_all,
                     gres_all, res, gtok, gtw)
        self.s = s = torch.cuda.Stream(device=dev)
        h = self.h

        def prepare():
            for r in range(N):
                ep.ep_shard_count(h[r], idx[r], table[r], stream=s)
            for r in range(N):
                ep.ep_shard_prepare(h[r], idx[r], table, tc[r], A, stream=s)

        self.fns = (
            prepare,
            lambda: [ep.ep_shard_dispatch(h[r], tok[r], wts[r], tab["recv"], tab["recv_w"], stream=s)
                     for r in range(N)],
            lambda: [ep.ep_shard_combine(h[r], tab["eo"], res[r], stream=s) for r in range(N)],
            lambda: [ep.ep_shard_combine_bwd(h[r], gres[r], tab["gexp"], stream=s) for r in range(N)],
            lambda: [ep.ep_shard_dispatch_bwd(h[r], tab["grecv"], tab["grecv_w"], gtok[r], gtw[r], stream=s)
                     for r in range(N)],
        )


class RankMajorStep:
    """The same batch as Step, split evenly over `nranks` ranks of a
    rank-major layer emulated on this GPU: a token goes once to each owner of
    its routes, with its ids relative to the owner and its weights.  The five
    calls are the rank-major ones (prepare = every rank's count, then every
    rank's prepare); the owners' local permutation, the single-buffer calls
    timed by the other workloads, is not part of this step.  Receive buffers
    hold the rows this batch needs (the largest owner's M)."""

    traffic_key = None  # no committed ncu rows for these launches

    def __init__(self, torch, ep, w, dev, dtype, nranks):
        T, H, E, K = w.T, w.H, w.E, w.K
        N = nranks
        assert T % N == 0 and E % N == 0
        tpr = T // N
        self.w, self.N = w, N
        wl = wl_mod()
        pt = wl.TORCH_PAYLOAD[dtype]
        self.es = torch.empty(0, dtype=pt).element_size()
        idx_cpu, wts_cpu = wl.routing(w)
        v = idx_cpu.reshape(-1)
        self.V = int(((v >= 0) & (v < E)).sum())
        idx = [idx_cpu[r * tpr:(r + 1) * tpr].contiguous().to(dev) for r in range(N)]
        wts = [wts_cpu[r * tpr:(r + 1) * tpr].contiguous().to(dev) for r in range(N)]
        table = torch.empty(N, N, dtype=torch.int32, device=dev)
        rows = [torch.empty(1, dtype=torch.int32, device=dev) for _ in range(N)]
        hs = []
        for r in range(N):
            lid, size = ep.ep_register_layer_rank_major(E, K, H, tpr, N, r, dtype=dtype)
            hs.append(ep.alloc_handle(lid, size, dev))
        for r in range(N):
            ep.ep_rank_major_count(hs[r], idx[r], table[r])
        for r in range(N):
            ep.ep_rank_major_prepare(hs[r], idx[r], table, rows[r])
        M = [int(x.item()) for x in rows]
        R = max(1, max(M))
        self.P, self.npad = sum(M), 0
        self.h = []
        for r in range(N):
            lid, size = ep.ep_register_layer_rank_major(E, K, H, tpr, N, r, recv_capacity=R, dtype=dtype)
            self.h.append(ep.alloc_handle(lid, size, dev))
        self.R = R
        prow = lambda: [torch.empty(R, H, dtype=pt, device=dev) for _ in range(N)]  # noqa: E731
        recv, part, grecv, gpart = prow(), prow(), prow(), prow()
        for q in range(N):
            part[q].copy_(wl.expert_out(w, R, device=dev).to(pt))
            gpart[q].copy_(wl.grad_recv(w, R, device=dev).to(pt))
        recv_idx = [torch.empty(R, K, dtype=torch.int64, device=dev) for _ in range(N)]
        recv_w = [torch.empty(R, K, dtype=torch.float32, device=dev) for _ in range(N)]
        gw = [wl.grad_recv_weights(w, R * K, device=dev).view(R, K) for _ in range(N)]
        tab = {k: ep.pointer_table(x, dev) for k, x in
               (("recv", recv), ("recv_idx", recv_idx), ("recv_w", recv_w), ("part", part),
                ("grecv", grecv), ("gpart", gpart), ("gw", gw))}
        tok_all, gres_all = wl.tokens(w, device=dev).to(pt), wl.grad_result(w, device=dev).to(pt)
        tok = [tok_all[r * tpr:(r + 1) * tpr] for r in range(N)]
        gres = [gres_all[r * tpr:(r + 1) * tpr] for r in range(N)]
        res = [torch.empty(tpr, H, dtype=pt, device=dev) for _ in range(N)]
        gtok = [torch.empty(tpr, H, dtype=pt, device=dev) for _ in range(N)]
        gtw = [torch.empty(tpr, K, dtype=torch.float32, device=dev) for _ in range(N)]
        self.keep = (idx, wts, table, rows, recv, part, grecv, gpart, recv_idx, recv_w, gw, tab, tok_all,
                     gres_all, res, gtok, gtw)
        self.s = s = torch.cuda.Stream(device=dev)
        h = self.h

        def prepare():
            for r in range(N):
                ep.ep_rank_major_count(h[r], idx[r], table[r], stream=s)
            for r in range(N):
                ep.ep_rank_major_prepare(h[r], idx[r], table, rows[r], stream=s)

        self.fns = (
            prepare,
            lambda: [ep.ep_rank_major_dispatch(h[r], idx[r], tok[r], wts[r], tab["recv"], tab["recv_idx"],
                                               tab["recv_w"], stream=s) for r in range(N)],
            lambda: [ep.ep_rank_major_combine(h[r], tab["part"], res[r], stream=s) for r in range(N)],
            lambda: [ep.ep_rank_major_combine_bwd(h[r], gres[r], tab["grecv"], stream=s) for r in range(N)],
            lambda: [ep.ep_rank_major_dispatch_bwd(h[r], tab["gpart"], tab["gw"], gtok[r], gtw[r], stream=s)
                     for r in range(N)],
        )

    def call_bytes(self):
        """Bytes each rank-major call must move over all ranks (M = rows over
        all owners): the routing map reads idx and writes the row map; the
        push reads each token once and writes M rows plus K ids and weights
        per row; the pulls read M rows and write T; the weight gradients
        read one entry per route."""
        w, es, M = self.w, self.es, self.P
        T, H, K = w.T, w.H, w.K
        return {
            "prepare": 8 * T * K + 4 * T * K + 4 * self.N * self.N,
            "dispatch": es * T * H + es * M * H + 8 * T * K + 4 * T * K * 2 + 12 * M * K,
            "combine": es * M * H + es * T * H + 4 * T * K,
            "combine_bwd": es * T * H + es * M * H + 4 * T * K,
            "dispatch_bwd": es * M * H + es * T * H + 4 * T * K * 4,
        }


def wl_mod():
    from combine_ep_prepare_gb300 import workloads
    return workloads


def measure_step(torch, ep, st, steps, warmup, flush, spin, world, dev, peak, peak_kind,
                 dtype, local):
    """Device-timed measurements of one workload's step: the step (events at
    its ends), every call alone between events, every prefix of the step (for
    the calls' marginal durations), and the step captured as a CUDA graph.
    Clocks are sampled over these timed regions."""
    w, s, fns = st.w, st.s, st.fns
    T, H, E, K = w.T, w.H, w.E, w.K
    with torch.cuda.stream(s):
        for _ in range(warmup):
            flush.zero_()
            torch.cuda._sleep(spin)
            for f in fns:
                f()
    torch.cuda.synchronize()
    if isinstance(st, (ShardStep, RankMajorStep)):
        for h in st.h:
            if ep.ep_read_info(h, stream=s)["status"] != 0:
                raise RuntimeError("libep status after warm-up (%s, sharded)" % w.name)
        P, npad = st.P, st.npad
    else:
        info = ep.ep_read_info(st.h, stream=s)
        if info["status"] != 0:
            raise RuntimeError("libep status %d after warm-up (%s)" % (info["status"], w.name))
        P, npad = info["used_rows"], info["padding_rows"]
    V = st.V if isinstance(st, RankMajorStep) else P - npad
    byts = st.call_bytes() if isinstance(st, RankMajorStep) else algorithmic_bytes(T, H, E, K, V, P, npad, st.es)

    # Timed region 1 (the step, as a user runs it): events only at the step
    # boundaries.  Timed region 2: the same steps with an event between calls,
    # for each kernel's own duration; events between calls serialise the
    # kernels, so region 2's step is a little longer.
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(CALLS) + 1)]
           for _ in range(steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clock = ClockSampler(local)
    time.sleep(0.3)
    launches0 = ep.ep_launch_count()
    with torch.cuda.stream(s):
        for i in range(steps):
            flush.zero_()
            torch.cuda._sleep(spin)
            ev_step[i][0].record(s)
            for f in fns:
                f()
            ev_step[i][1].record(s)
    torch.cuda.synchronize()
    launches = ep.ep_launch_count() - launches0
    with torch.cuda.stream(s):
        for i in range(steps):
            flush.zero_()
            torch.cuda._sleep(spin)
            evs[i][0].record(s)
            for j, f in enumerate(fns):
                f()
                evs[i][j + 1].record(s)
    torch.cuda.synchronize()
    # Timed region 3: prefixes of the step, calls 0..j, with events only at
    # the prefix's ends, so the kernels chain exactly as in the step.  A
    # call's marginal duration t(0..j) - t(0..j-1) is what it adds to the
    # chained step (the five add up to the step); an event pair around one
    # short launch (region 2) also times its launch and drain, which the
    # chain overlaps.  The roofline uses the marginal duration.
    prefix_ms = []
    for j in range(1, len(CALLS) + 1):
        evp = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        with torch.cuda.stream(s):
            for i in range(steps):
                flush.zero_()
                torch.cuda._sleep(spin)
                evp[i][0].record(s)
                for f in fns[:j]:
                    f()
                evp[i][1].record(s)
        torch.cuda.synchronize()
        prefix_ms.append(sum(a.elapsed_time(b) for a, b in evp) / len(evp))
    # Timed region 4: prepare run twice in a row.  The second one follows a
    # kernel in the chain, as prepare follows the router in a model step, so
    # its launch overlaps the first one's run: t(2 prepares) - t(1 prepare) is
    # prepare's cost inside a chain, without the wait from the step's first
    # event to its first kernel that the marginal duration above includes.
    evq = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    with torch.cuda.stream(s):
        for i in range(steps):
            flush.zero_()
            torch.cuda._sleep(spin)
            evq[i][0].record(s)
            fns[0]()
            fns[0]()
            evq[i][1].record(s)
    torch.cuda.synchronize()
    prepare_chained = sum(a.elapsed_time(b) for a, b in evq) / len(evq) - prefix_ms[0]
    graph = run_graph(torch, fns, s, flush, spin, steps, T, world, dev)
    clocks = clock.stop()

    per_call = {c: [] for c in CALLS}
    step_ms = [a.elapsed_time(b) for a, b in ev_step]
    for e in evs:
        for j, c in enumerate(CALLS):
            per_call[c].append(e[j].elapsed_time(e[j + 1]))
    ms = reduce_max(sum(step_ms) / len(step_ms), dev)
    value = whole_job_rate(T, world, ms)
    step_bytes = sum(byts.values())
    avg = {c: sum(v) / len(v) for c, v in per_call.items()}
    marginal = {c: prefix_ms[j] - (prefix_ms[j - 1] if j else 0.0) for j, c in enumerate(CALLS)}
    dom = max(CALLS, key=lambda c: marginal[c])
    achieved = byts[dom] / (marginal[dom] * 1e-3) / 1e9
    achieved_events = byts[dom] / (avg[dom] * 1e-3) / 1e9

    def rate(c, t_ms):
        return byts[c] / (t_ms * 1e-3) / 1e9 if t_ms > 0 else None

    kernels = {c: {"ms_marginal": round(marginal[c], 5), "ms_events": round(avg[c], 5),
                   "algorithmic_bytes": byts[c],
                   "GB/s_marginal": rate(c, marginal[c]) and round(rate(c, marginal[c]), 1),
                   "GB/s_events": round(rate(c, avg[c]), 1),
                   "frac_of_" + peak_kind + "_marginal":
                       rate(c, marginal[c]) and round(rate(c, marginal[c]) / peak, 4),
                   "frac_of_" + peak_kind + "_events": round(rate(c, avg[c]) / peak, 4)}
               for c in CALLS}
    kernels["prepare"]["ms_chained"] = round(prepare_chained, 5)
    # ncu DRAM bytes were captured for bf16 payloads
    key = getattr(st, "traffic_key", w.name)
    traffic = committed_traffic(dom, key, byts[dom]) if dtype == "bf16" and key else None
    graph["hbm_frac_step"] = step_bytes / (graph["ms_per_step"] * 1e-3) / 1e9 / peak
    return {
        "config": workload_config(w, None),
        "value": value, "unit": UNIT, "ms_per_step": ms,
        "hbm_gbs_step": step_bytes / (ms * 1e-3) / 1e9,
        "hbm_frac_step": step_bytes / (ms * 1e-3) / 1e9 / peak,
        "bytes_per_step": step_bytes,
        "routing": {"valid_routes": V, "used_rows": P, "padding_rows": npad, "recv_capacity": st.R},
        "roofline": {"bound": "hbm", "kernel": KERNEL_OF_CALL[dom] + " (" + dom + ")",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "traffic": traffic,
                     "duration": "marginal in the chained step, %.2f us" % (marginal[dom] * 1e3),
                     "achieved_events": achieved_events,
                     "frac_events": achieved_events / peak},
        "kernels": kernels,
        "graph_replay": graph,
        "gpu_launches": launches,
        "clocks": clocks,
        "steps": steps, "warmup": warmup,
    }


def main():
    args = parse_args()
    wl = wl_mod()
    w = wl.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)

    import torch
    import torch.distributed as dist
    import combine_ep_prepare_gb300 as ep

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.int32, device=dev)
    # Before each step the GPU spins for ~0.3 ms (outside the step's events)
    # so that the host has enqueued the whole step before it starts: the
    # events then time the device, not the host's per-call enqueue cost.
    spin = int(0.3e-3 * 2.07e9)
    peak, peak_kind = measured_peak()
    l2_note = ("flushed before every step (write of %d MB, outside the step's events); "
               "host enqueue hidden by a 0.3 ms GPU spin before each step" % (flush.numel() * 4 >> 20))

    st = Step(torch, ep, w, dev, args.dtype)
    head = measure_step(torch, ep, st, args.steps, args.warmup, flush, spin, world, dev, peak,
                        peak_kind, args.dtype, local)

    # End to end: host inputs -> device -> five calls -> host outputs.
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, torch, ep, w, st.h, dev, st.s, st.idx_cpu, st.wts_cpu, st.tok, st.eo,
                      st.gres, st.grecv, st.grecv_w, st.counts, st.recv, st.recv_w, st.res,
                      st.gexp, st.gtok, st.gtw, world)
    del st
    torch.cuda.empty_cache()

    # The other workloads, one after another in the same process (each
    # workload's buffers freed before the next is allocated).
    others = {}
    names = [n for n in args.also.split(",") if n and n != "none" and n != w.name]
    for name in names:
        ow = wl.WORKLOADS[name]
        ost = Step(torch, ep, ow, dev, args.dtype)
        r = measure_step(torch, ep, ost, min(args.steps, 20), max(3, min(args.warmup, 5)), flush,
                         spin, world, dev, peak, peak_kind, args.dtype, local)
        r["config"] = workload_config(ow, l2_note)
        others[name] = r
        del ost
        torch.cuda.empty_cache()

    if args.sharded > 0 and args.also != "none":
        sw = wl.WORKLOADS["dsv3"]
        sst = ShardStep(torch, ep, sw, dev, args.dtype, args.sharded)
        r = measure_step(torch, ep, sst, min(args.steps, 20), max(3, min(args.warmup, 5)), flush,
                         spin, world, dev, peak, peak_kind, args.dtype, local)
        r["config"] = workload_config(sw, l2_note)
        r["config"]["workload"] = ("dsv3, sharded: the same batch over %d ranks of a sharded layer "
                                   "emulated on this GPU (each call runs every rank's call)" % args.sharded)
        r["config"]["ranks"] = args.sharded
        others["dsv3_sharded%d" % args.sharded] = r
        del sst
        torch.cuda.empty_cache()
        rst = RankMajorStep(torch, ep, sw, dev, args.dtype, args.sharded)
        r = measure_step(torch, ep, rst, min(args.steps, 20), max(3, min(args.warmup, 5)), flush,
                         spin, world, dev, peak, peak_kind, args.dtype, local)
        r["config"] = workload_config(sw, l2_note)
        r["config"]["workload"] = ("dsv3, rank-major: the same batch over %d ranks of a rank-major layer "
                                   "emulated on this GPU (each call runs every rank's call; the owners' "
                                   "local permutation is not in the step)" % args.sharded)
        r["config"]["ranks"] = args.sharded
        others["dsv3_rank_major%d" % args.sharded] = r
        del rst
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and args.dtype == "bf16":
        cpu = cpu_baseline(w, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
            "data": "synthetic (seeded; shapes of the %s workload)" % w.name,
            "config": workload_config(w, l2_note),
            "hbm_gbs_step": head["hbm_gbs_step"],
            "hbm_frac_step": head["hbm_frac_step"],
            "bytes_per_step": head["bytes_per_step"],
            "routing": head["routing"],
            "roofline": head["roofline"],
            "kernels": head["kernels"],
            "cpu_baseline": cpu,
            "e2e": e2e,
            "graph_replay": head["graph_replay"],
            "gpu_launches": head["gpu_launches"],
            "clocks": head["clocks"],
            "workloads": others,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_e2e(args, torch, ep, w, h, dev, s, idx_cpu, wts_cpu, tok, eo, gres, grecv, grecv_w,
            counts, recv, recv_w, res, gexp, gtok, gtw, world):
    """End to end through the public API: every step copies all its inputs from
    pinned host memory (topk_idx, topk_weights, tokens, expert_out [R,H], the
    combine gradient [T,H], the dispatch gradient [R,H] and its weights [R]),
    runs the five calls, and copies the token-side outputs back (result,
    grad_tokens, grad_topk_weights, token_counts); recv_tokens and
    grad_expert_out stay in HBM for the expert GEMMs that consume them.
    Pipelined as a serving loop would be: step i+1's host-to-device copies
    run on a copy stream while step i computes, and step i's outputs come
    back on a third stream; inputs and outputs are double-buffered."""
    pin = lambda t: t.detach().to("cpu").pin_memory()  # noqa: E731
    h_in = {"idx": pin(idx_cpu), "wts": pin(wts_cpu), "tok": pin(tok), "eo": pin(eo),
            "gres": pin(gres), "grecv": pin(grecv), "grecv_w": pin(grecv_w)}
    d_in = [{k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in h_in.items()}
            for _ in range(2)]
    outs = {"res": res, "gtok": gtok, "gtw": gtw, "counts": counts}
    d_out = [{k: torch.empty_like(v) for k, v in outs.items()} for _ in range(2)]
    h_out = [{k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in outs.items()}
             for _ in range(2)]
    bi = sum(t.numel() * t.element_size() for t in h_in.values())
    bo = sum(t.numel() * t.element_size() for t in h_out[0].values())
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    comp_done = [ev(), ev()]
    out_done = [ev(), ev()]
    in_done = [ev(), ev()]
    started = [False, False]

    def step(i):
        b = i % 2
        di, do = d_in[b], d_out[b]
        with torch.cuda.stream(s_in):
            if started[b]:
                s_in.wait_event(comp_done[b])  # step i-2 has finished reading these inputs
            for k in h_in:
                di[k].copy_(h_in[k], non_blocking=True)
            in_done[b].record(s_in)
        with torch.cuda.stream(s):
            s.wait_event(in_done[b])
            if started[b]:
                s.wait_event(out_done[b])  # step i-2's outputs have been copied out
            ep.ep_prepare(h, di["idx"], do["counts"], w.A, stream=s)
            ep.ep_dispatch(h, di["idx"], di["tok"], di["wts"], recv, recv_w, stream=s)
            ep.ep_combine(h, di["eo"], do["res"], stream=s)
            ep.ep_combine_bwd(h, di["gres"], gexp, stream=s)
            ep.ep_dispatch_bwd(h, di["grecv"], di["grecv_w"], do["gtok"], do["gtw"], stream=s)
            comp_done[b].record(s)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            for k in do:
                h_out[b][k].copy_(do[k], non_blocking=True)
            out_done[b].record(s_out)
        started[b] = True

    for i in range(max(2, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    n = max(4, args.steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(n):
        step(i)
    e1.record(s_out)  # the last step's outputs are the last work of the pipeline
    torch.cuda.synchronize()
    ms = reduce_max(e0.elapsed_time(e1) / n, dev)
    return {"value": whole_job_rate(w.T, world, ms), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "pipeline": "copies of step i+1 overlap step i (3 streams, double-buffered)"}


def run_graph(torch, fns, s, flush, spin, steps, T, world, dev):
    """The five calls captured once as a CUDA graph and replayed (the API
    is allocation-free and stream-ordered, so the whole step captures); each
    replay after an L2 flush and a GPU spin, outside its events."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for f in fns:
            f()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    with torch.cuda.stream(s):
        for _ in range(3):
            flush.zero_()
            g.replay()
        for a, b in evs:
            flush.zero_()
            torch.cuda._sleep(spin)
            a.record(s)
            g.replay()
            b.record(s)
    torch.cuda.synchronize()
    ms = reduce_max(sum(a.elapsed_time(b) for a, b in evs) / len(evs), dev)
    del g
    return {"value": whole_job_rate(T, world, ms), "unit": UNIT, "ms_per_step": ms}


if __name__ == "__main__":
    sys.exit(main())
