"""Runs one expert-parallel step through libep (GPU) and through the CPU oracle
on the same seeded inputs, for the parity tests.

Inputs come from combine_ep_prepare_gb300.workloads (CPU, seeded); the oracle
never sees anything the GPU produced.  Receive-side inputs (expert_out, the
gradient rows) only matter in rows [0, P); their row count is taken from the
oracle's own prepare, and the GPU buffers hold R rows with a sentinel pattern
beyond P so that untouched rows can be checked.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

from combine_ep_prepare_gb300 import workloads as wl

SENTINEL = 0x7FC1          # a NaN bf16 / fp16 pattern no kernel writes
SENTINEL32 = 0x7FC1C0DE    # a NaN fp32 pattern no kernel writes
TORCH = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def bits(t: torch.Tensor) -> np.ndarray:
    """Payload tensor -> numpy: uint16 bit patterns for 16-bit types, float32
    for fp32 (compare those with same())."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def same(a, b) -> bool:
    """Bit-for-bit equality of two payload arrays."""
    a, b = np.ascontiguousarray(a), np.ascontiguousarray(b)
    if a.dtype == np.float32 or b.dtype == np.float32:
        return a.shape == b.shape and np.array_equal(a.view(np.uint32), b.view(np.uint32))
    return np.array_equal(a, b)


def untouched(a) -> bool:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return bool(np.all(a.view(np.uint32) == SENTINEL32))
    return bool(np.all(a == SENTINEL))


def sentinel_tensor(shape, dtype: str, device):
    if dtype == "fp32":
        return torch.full(shape, SENTINEL32, dtype=torch.int32, device=device).view(torch.float32)
    return torch.full(shape, SENTINEL, dtype=torch.int16, device=device).view(TORCH[dtype])


def from_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


@dataclasses.dataclass
class StepInputs:
    E: int
    K: int
    H: int
    A: int
    topk_idx: torch.Tensor        # int64 [T,K] (cpu)
    topk_weights: torch.Tensor    # f32 [T,K]
    tokens: torch.Tensor          # bf16 [T,H]
    expert_out: torch.Tensor      # bf16 [rows,H]
    grad_result: torch.Tensor     # bf16 [T,H]
    grad_recv: torch.Tensor       # bf16 [rows,H]
    grad_recv_w: Optional[torch.Tensor]  # f32 [rows] or None
    dtype: str = "bf16"

    @property
    def T(self):
        return self.topk_idx.shape[0]


def workload_inputs(w: wl.Workload, oracle_mod, T: Optional[int] = None,
                    with_weight_grad: bool = True) -> StepInputs:
    idx, wts = wl.routing(w, T=T)
    rt = oracle_mod.prepare(idx.numpy(), w.E, w.A)
    rows = max(rt.P, 1)
    return StepInputs(
        E=w.E, K=w.K, H=w.H, A=w.A, topk_idx=idx, topk_weights=wts,
        tokens=wl.tokens(w, T=idx.shape[0]),
        expert_out=wl.expert_out(w, rows),
        grad_result=wl.grad_result(w, T=idx.shape[0]),
        grad_recv=wl.grad_recv(w, rows),
        grad_recv_w=wl.grad_recv_weights(w, rows) if with_weight_grad else None)


def custom_inputs(idx, wts, E, H, A, oracle_mod, seed=0, with_weight_grad=True,
                  dtype="bf16") -> StepInputs:
    rt = oracle_mod.prepare(idx.numpy(), E, A)
    rows = max(rt.P, 1)
    T = idx.shape[0]
    return StepInputs(
        E=E, K=idx.shape[1], H=H, A=A, topk_idx=idx, topk_weights=wts,
        tokens=wl.payload_normal(T, H, seed + 1, dtype),
        expert_out=wl.payload_normal(rows, H, seed + 2, dtype),
        grad_result=wl.payload_normal(T, H, seed + 3, dtype),
        grad_recv=wl.payload_normal(rows, H, seed + 4, dtype),
        grad_recv_w=wl.f32_normal(rows, seed + 5) if with_weight_grad else None,
        dtype=dtype)


def oracle_step(inp: StepInputs, oracle_mod, R: Optional[int] = None) -> dict:
    rt = oracle_mod.prepare(inp.topk_idx.numpy(), inp.E, inp.A, R)
    out = {"rt": rt, "counts": rt.token_counts, "offsets": rt.offsets, "slot": rt.slot,
           "P": rt.P, "status": rt.status}
    if rt.overflow:
        return out
    dt = inp.dtype
    recv, recv_w = oracle_mod.dispatch(rt, bits(inp.tokens), inp.topk_weights.numpy(), dt)
    out["recv_tokens"], out["recv_w"] = recv, recv_w
    out["result"] = oracle_mod.combine(rt, bits(inp.expert_out), dt)
    out["grad_expert_out"] = oracle_mod.combine_bwd(rt, bits(inp.grad_result), dt)
    gw = None if inp.grad_recv_w is None else inp.grad_recv_w.numpy()
    out["grad_tokens"], out["grad_topk_weights"] = oracle_mod.dispatch_bwd(rt, bits(inp.grad_recv), gw, dt)
    return out


class GpuLayer:
    """A registered layer with its receive-side buffers (R rows) on the GPU."""

    def __init__(self, ep, E, K, H, max_tokens, max_alignment, recv_capacity=0, device="cuda",
                 dtype="bf16"):
        self.ep = ep
        self.E, self.K, self.H, self.dtype = E, K, H, dtype
        self.id, self.mem_size = ep.ep_register_layer(E, K, H, max_tokens, max_alignment, recv_capacity,
                                                      dtype=dtype)
        self.R = ep.ep_recv_capacity(self.id)
        self.device = device

    def handle(self):
        return self.ep.alloc_handle(self.id, self.mem_size, self.device)


def gpu_step(ep, layer: GpuLayer, inp: StepInputs, handle=None, stream=None) -> dict:
    """Upload inputs, run the five calls, download everything."""
    dev = layer.device
    T, K, H, R = inp.T, inp.K, inp.H, layer.R
    h = handle if handle is not None else layer.handle()
    idx = inp.topk_idx.to(dev)
    wts = inp.topk_weights.to(dev)
    tok = inp.tokens.to(dev)
    rows = inp.expert_out.shape[0]

    dt = inp.dtype

    def rbuf(src):
        b = sentinel_tensor((R, H), dt, dev)
        n = min(rows, R)
        b[:n] = src[:n].to(dev)
        return b

    eo = rbuf(inp.expert_out)
    grecv = rbuf(inp.grad_recv)
    grecv_w = None
    if inp.grad_recv_w is not None:
        grecv_w = torch.full((R,), float("nan"), dtype=torch.float32, device=dev)
        n = min(rows, R)
        grecv_w[:n] = inp.grad_recv_w[:n].to(dev)
    gres = inp.grad_result.to(dev)
    counts = torch.full((inp.E,), -5, dtype=torch.int32, device=dev)
    recv = sentinel_tensor((R, H), dt, dev)
    recv_w = torch.full((R,), -3.0, dtype=torch.float32, device=dev)
    result = sentinel_tensor((T, H), dt, dev)
    gexp = sentinel_tensor((R, H), dt, dev)
    gtok = sentinel_tensor((T, H), dt, dev)
    gtw = torch.full((T, K), -3.0, dtype=torch.float32, device=dev)
    offsets = torch.full((inp.E + 1,), -9, dtype=torch.int32, device=dev)
    slots = torch.full((T, K), -9, dtype=torch.int32, device=dev)

    ep.ep_prepare(h, idx, counts, inp.A, stream=stream)
    ep.ep_dispatch(h, idx, tok, wts, recv, recv_w, stream=stream)
    ep.ep_combine(h, eo, result, stream=stream)
    ep.ep_combine_bwd(h, gres, gexp, stream=stream)
    ep.ep_dispatch_bwd(h, grecv, grecv_w, gtok, gtw, stream=stream)
    ep.ep_expert_offsets(h, offsets, stream=stream)
    ep.ep_token_slots(h, slots, stream=stream)
    info = ep.ep_read_info(h, stream=stream)
    torch.cuda.synchronize()
    return {"counts": counts.cpu().numpy(), "offsets": offsets.cpu().numpy(),
            "slot": slots.cpu().numpy(), "info": info,
            "recv_tokens": bits(recv), "recv_w": recv_w.cpu().numpy(),
            "result": bits(result), "grad_expert_out": bits(gexp),
            "grad_tokens": bits(gtok), "grad_topk_weights": gtw.cpu().numpy(), "handle": h}


def assert_step_equal(g: dict, o: dict, R: int):
    """Bit-exact comparison of every output of the step."""
    P = o["P"]
    assert g["info"]["status"] == o["status"], (g["info"], o["status"])
    assert np.array_equal(g["counts"], o["counts"])
    assert np.array_equal(g["offsets"], o["offsets"])
    assert np.array_equal(g["slot"], o["slot"])
    assert g["info"]["used_rows"] == P
    assert g["info"]["padding_rows"] == int((o["rt"].inv < 0).sum())
    if o["rt"].overflow:
        return
    assert same(g["recv_tokens"][:P], o["recv_tokens"])
    assert np.array_equal(g["recv_w"][:P].view(np.uint32), o["recv_w"].view(np.uint32))
    assert same(g["result"], o["result"])
    assert same(g["grad_expert_out"][:P], o["grad_expert_out"])
    assert same(g["grad_tokens"], o["grad_tokens"])
    assert np.array_equal(g["grad_topk_weights"].view(np.uint32), o["grad_topk_weights"].view(np.uint32))
    # rows at or beyond P are never touched
    assert untouched(g["recv_tokens"][P:])
    assert untouched(g["grad_expert_out"][P:])
    assert np.all(g["recv_w"][P:] == -3.0)
