"""Seeded synthetic workloads for MoE expert-parallel dispatch / combine.

This module only draws random inputs.  It holds none of the routing,
dispatch or combine arithmetic: the routing *choice* made here (which experts a
token picks, with which weights) plays the part of a model's router, which
sits upstream of the expert-parallel path and is an input to it.

Shapes follow the MoE models the pages use as examples of expert-parallel
workloads (Mixtral, Qwen3-MoE, DeepSeek-V3, and a masked decode batch in the
style of the HF transformers all-reduce EP mode, "Expert-parallel
implementations for ep_dispatch_experts", section "AllReduceEP").  No weights
or datasets are involved: every tensor is drawn from a seeded generator.

Seeds: routing = 1000 + config number, tokens = 2000 + n, expert_out = 3000 + n,
gradients = 4000 + n.

Both the CUDA path (through the C ABI) and the CPU oracle read the same
tensors produced here; nothing in this file imports either of them.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One configuration of the expert-parallel step."""

    name: str
    number: int          # seed offset
    T: int               # tokens
    H: int               # hidden size (bf16 elements per row)
    E: int               # experts
    K: int               # top-k
    A: int               # dispatch_output_per_expert_alignment
    routing: str         # "uniform" | "zipf" | "grouped" | "grouped_masked"
    zipf_s: float = 1.2
    n_groups: int = 8
    topk_groups: int = 4
    local_experts: Optional[int] = None  # masked config: experts >= this become -1

    def worst_case_rows(self, max_alignment: Optional[int] = None) -> int:
        """Receive capacity that no routing of this shape can exceed."""
        a = self.A if max_alignment is None else max_alignment
        routes = self.T * self.K
        return routes + min(self.E, routes) * (a - 1)


WORKLOADS = {
    "tiny": Workload("tiny", 0, T=64, H=128, E=8, K=2, A=16, routing="uniform"),
    "mixtral": Workload("mixtral", 1, T=4096, H=4096, E=8, K=2, A=128, routing="uniform"),
    "qwen3": Workload("qwen3", 2, T=8192, H=2048, E=128, K=8, A=128, routing="zipf"),
    "dsv3": Workload("dsv3", 3, T=16384, H=7168, E=256, K=8, A=128, routing="grouped"),
    "decode": Workload("decode", 4, T=128, H=7168, E=256, K=8, A=1,
                       routing="grouped_masked", local_experts=128),
}


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def routing(w: Workload, T: Optional[int] = None, device="cpu"):
    """Return (topk_idx int64 [T,K], topk_weights float32 [T,K]).

    uniform : K distinct experts per token, uniformly at random (argsort of
              U(0,1)[E], first K); weights softmax of K N(0,1) logits.
    zipf    : expert popularity p proportional to rank^-s over a seeded
              permutation of experts; K distinct experts per token by
              Gumbel-top-K on log p; weights softmax of K N(0,1) logits.
    grouped : per token z ~ N(0,1)[E] and group scores g ~ N(0,1)[n_groups];
              keep the top groups by g, then the top-K experts by z inside
              them; weights sigmoid(z_sel) / sum sigmoid(z_sel).
    grouped_masked : as grouped, then experts >= local_experts become -1.
    """
    T = w.T if T is None else T
    g = _gen(1000 + w.number, device)
    E, K = w.E, w.K
    if w.routing == "uniform":
        u = torch.rand(T, E, generator=g, device=device)
        idx = torch.argsort(u, dim=1)[:, :K].contiguous()
        logits = torch.randn(T, K, generator=g, device=device)
        wts = torch.softmax(logits, dim=1)
    elif w.routing == "zipf":
        perm = torch.randperm(E, generator=g, device=device)
        ranks = torch.empty(E, dtype=torch.float64, device=device)
        ranks[perm] = torch.arange(1, E + 1, dtype=torch.float64, device=device)
        logp = -w.zipf_s * torch.log(ranks)
        u = torch.rand(T, E, generator=g, device=device, dtype=torch.float64)
        gumbel = -torch.log(-torch.log(u.clamp_min(1e-300)))
        idx = torch.topk(logp[None, :] + gumbel, K, dim=1).indices.contiguous()
        logits = torch.randn(T, K, generator=g, device=device)
        wts = torch.softmax(logits, dim=1)
    elif w.routing in ("grouped", "grouped_masked"):
        z = torch.randn(T, E, generator=g, device=device)
        gs = torch.randn(T, w.n_groups, generator=g, device=device)
        per_group = E // w.n_groups
        top_groups = torch.topk(gs, w.topk_groups, dim=1).indices
        keep = torch.zeros(T, w.n_groups, dtype=torch.bool, device=device)
        keep.scatter_(1, top_groups, True)
        keep = keep.repeat_interleave(per_group, dim=1)
        zm = z.masked_fill(~keep, float("-inf"))
        sel = torch.topk(zm, K, dim=1)
        idx = sel.indices.contiguous()
        sig = torch.sigmoid(sel.values)
        wts = sig / sig.sum(dim=1, keepdim=True)
        if w.routing == "grouped_masked":
            idx = idx.masked_fill(idx >= w.local_experts, -1)
    else:
        raise ValueError(w.routing)
    return idx.to(torch.int64).contiguous(), wts.to(torch.float32).contiguous()


def bf16_normal(rows: int, cols: int, seed: int, device="cpu") -> torch.Tensor:
    """bf16 [rows, cols] drawn from N(0,1), seeded."""
    g = _gen(seed, device)
    return torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


TORCH_PAYLOAD = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def payload_normal(rows: int, cols: int, seed: int, dtype: str = "bf16", device="cpu") -> torch.Tensor:
    """[rows, cols] of the payload type drawn from N(0,1), seeded (bf16 draws
    are bit-identical to bf16_normal)."""
    g = _gen(seed, device)
    x = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32)
    return x.to(TORCH_PAYLOAD[dtype])


def f32_normal(n: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randn(n, generator=g, device=device, dtype=torch.float32)


def tokens(w: Workload, T: Optional[int] = None, device="cpu") -> torch.Tensor:
    return bf16_normal(w.T if T is None else T, w.H, 2000 + w.number, device)


def expert_out(w: Workload, rows: int, device="cpu") -> torch.Tensor:
    """Stand-in for the expert MLP output: rows x H bf16 N(0,1)."""
    return bf16_normal(rows, w.H, 3000 + w.number, device)


def grad_result(w: Workload, T: Optional[int] = None, device="cpu") -> torch.Tensor:
    """Upstream gradient of combine's result: [T,H] bf16 N(0,1)."""
    return bf16_normal(w.T if T is None else T, w.H, 4000 + w.number, device)


def grad_recv(w: Workload, rows: int, device="cpu") -> torch.Tensor:
    """Upstream gradient of dispatch's recv_tokens: [rows,H] bf16 N(0,1)."""
    return bf16_normal(rows, w.H, 4500 + w.number, device)


def grad_recv_weights(w: Workload, rows: int, device="cpu") -> torch.Tensor:
    """Upstream gradient of dispatch's recv_topk_weights: [rows] float32 N(0,1)."""
    return f32_normal(rows, 4800 + w.number, device)


def small_int_bf16(rows: int, cols: int, seed: int, lo: int = -4, hi: int = 5) -> torch.Tensor:
    """bf16 tensor of small integers: sums of a few of them are exact in fp32."""
    g = _gen(seed)
    return torch.randint(lo, hi, (rows, cols), generator=g).to(torch.bfloat16)


def random_routing(T: int, K: int, E: int, seed: int, p_mask: float = 0.0,
                   p_bad: float = 0.0, distinct: bool = False):
    """Unstructured routing for edge cases: repeats allowed unless distinct,
    a fraction p_mask of routes set to -1 and p_bad set to out-of-range values."""
    g = _gen(seed)
    if distinct:
        idx = torch.argsort(torch.rand(T, E, generator=g), dim=1)[:, :K]
    else:
        idx = torch.randint(0, E, (T, K), generator=g)
    if p_mask > 0:
        m = torch.rand(T, K, generator=g) < p_mask
        idx = idx.masked_fill(m, -1)
    if p_bad > 0:
        b = torch.rand(T, K, generator=g) < p_bad
        bad_vals = torch.where(torch.rand(T, K, generator=g) < 0.5,
                               torch.full((T, K), E, dtype=torch.int64),
                               torch.full((T, K), -7, dtype=torch.int64))
        idx = torch.where(b, bad_vals, idx)
    wts = torch.softmax(torch.randn(T, K, generator=g), dim=1)
    return idx.to(torch.int64).contiguous(), wts.to(torch.float32).contiguous()
