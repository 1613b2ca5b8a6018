"""CPU oracle for MoE expert-parallel prepare / dispatch / combine and backward.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
path (``combine_ep_prepare_gb300``) never imports it, and it never imports
the product.

The arithmetic lives in ``ep_oracle.c`` (plain single-threaded C, one loop per
definition); this module only marshals numpy arrays into it.  bf16 data is
passed as raw ``uint16`` bit patterns.

The operations follow TransformerEngine PR #3034, "Expert Parallelism: common
C API + NCCL EP backend", section "Per-step (allocation-free, CUDA-graph
capturable)": prepare, dispatch, combine (unweighted), dispatch_bwd and
combine_bwd, with the readings listed in the header of ``ep_oracle.c``.

Every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (hand-worked golden cases, library routines,
closed forms and adjoint identities).
"""
from __future__ import annotations

import contextlib
import ctypes
import dataclasses
import os
from typing import Optional

import numpy as np

from .build import build_oracle, oracle_library_path

STATUS_BAD_INDEX = 1
STATUS_OVERFLOW = 2

# Payload element types; 16-bit rows travel as uint16 bit patterns, fp32 rows
# as float32.
DTYPES = {"bf16": 0, "fp16": 1, "fp32": 2}
NP_ROW = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.float32}

_lib = None


def _configure(lib):
    i64, p = ctypes.c_int64, ctypes.c_void_p
    c_int = ctypes.c_int
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_prepare.argtypes = [p, i64, i64, i64, i64, i64, p, p, p, p, p, p]
    lib.oracle_prepare.restype = ctypes.c_int
    lib.oracle_dispatch.argtypes = [p, i64, i64, i64, c_int, p, p, p, p]
    lib.oracle_dispatch.restype = None
    lib.oracle_gather_sum.argtypes = [p, i64, i64, i64, c_int, p, p]
    lib.oracle_gather_sum.restype = None
    lib.oracle_combine_bwd.argtypes = [p, i64, i64, i64, c_int, p, p]
    lib.oracle_combine_bwd.restype = None
    lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f32.restype = ctypes.c_float
    lib.oracle_round_array_f16.argtypes = [p, p, i64]
    lib.oracle_round_array_f16.restype = None
    lib.oracle_weight_gather.argtypes = [p, i64, i64, p, p]
    lib.oracle_weight_gather.restype = None
    lib.oracle_round_array.argtypes = [p, p, i64]
    lib.oracle_round_array.restype = None
    lib.oracle_gather_weighted_sum.argtypes = [p, i64, i64, i64, c_int, p, p, p]
    lib.oracle_gather_weighted_sum.restype = None
    lib.oracle_combine_bwd_weighted.argtypes = [p, i64, i64, i64, c_int, p, p, p, p, p]
    lib.oracle_combine_bwd_weighted.restype = None
    lib.oracle_shard_prepare.argtypes = [p, p, i64, i64, i64, i64, i64, i64, p, p, p, p, p, p, p]
    lib.oracle_shard_prepare.restype = ctypes.c_int
    lib.oracle_shard_gather_sum.argtypes = [p, p, i64, i64, i64, c_int, p, p]
    lib.oracle_shard_gather_sum.restype = None
    lib.oracle_shard_weight_gather.argtypes = [p, p, i64, p, p]
    lib.oracle_shard_weight_gather.restype = None
    lib.oracle_rm_prepare.argtypes = [p, p, i64, i64, i64, i64, i64, p, p, p, p, p, p, p]
    lib.oracle_rm_prepare.restype = ctypes.c_int
    lib.oracle_rm_dispatch.argtypes = [p, i64, p, p, i64, i64, i64, i64, i64, c_int, p, p, p, p]
    lib.oracle_rm_dispatch.restype = None
    lib.oracle_rm_weight_gather.argtypes = [p, p, i64, i64, p, p]
    lib.oracle_rm_weight_gather.restype = None
    return lib


def _load():
    global _lib
    if _lib is not None:
        return _lib
    path = oracle_library_path()
    if not os.path.exists(path):
        build_oracle()
    _lib = _configure(ctypes.CDLL(path))
    return _lib


@contextlib.contextmanager
def use_library(path: str):
    """Run the oracle's Python functions against another build of ep_oracle.c
    (the mutation tests compile copies with planted mistakes)."""
    global _lib
    prev = _load()
    _lib = _configure(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = prev


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


@dataclasses.dataclass
class Routing:
    """Result of prepare: everything later steps need, plus status."""

    T: int
    K: int
    E: int
    A: int
    R: int
    token_counts: np.ndarray  # int32 [E]
    offsets: np.ndarray       # int32 [E+1]
    slot: np.ndarray          # int32 [T,K]
    inv: np.ndarray           # int32 [P]
    P: int
    status: int

    @property
    def overflow(self) -> bool:
        return bool(self.status & STATUS_OVERFLOW)


def bf16_to_f32(bits: int) -> float:
    return float(_load().oracle_bf16_to_f32(bits))


def f32_to_bf16(x: float) -> int:
    return int(_load().oracle_f32_to_bf16(x))


def f16_to_f32(bits: int) -> float:
    return float(_load().oracle_f16_to_f32(bits))


def round_to_f16(x: np.ndarray) -> np.ndarray:
    """Elementwise binary32 -> binary16 bits (round to nearest, ties to even)."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(a.shape, np.uint16)
    _load().oracle_round_array_f16(_ptr(a), _ptr(out), a.size)
    return out


def _rows(a, dtype):
    return np.ascontiguousarray(a, dtype=NP_ROW[dtype])


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Elementwise binary32 -> bf16 bits (round to nearest, ties to even)."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(a.shape, np.uint16)
    _load().oracle_round_array(_ptr(a), _ptr(out), a.size)
    return out


def prepare(topk_idx: np.ndarray, num_experts: int, alignment: int,
            recv_capacity: Optional[int] = None) -> Routing:
    """Steps a1-a3: counts, aligned offsets, (t,k)-stable slots."""
    lib = _load()
    idx = np.ascontiguousarray(topk_idx, dtype=np.int64)
    T, K = idx.shape
    E, A = int(num_experts), int(alignment)
    room = T * K + E * (A - 1)
    R = room if recv_capacity is None else int(recv_capacity)
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    slot = np.zeros((T, K), np.int32)
    inv = np.zeros(max(room, 1), np.int32)
    P = ctypes.c_int64(0)
    st = ctypes.c_uint32(0)
    rc = lib.oracle_prepare(_ptr(idx), T, K, E, A, R, _ptr(counts), _ptr(offsets),
                            _ptr(slot), _ptr(inv), ctypes.byref(P), ctypes.byref(st))
    if rc != 0:
        raise ValueError("oracle_prepare rejected its arguments")
    return Routing(T, K, E, A, R, counts, offsets, slot, inv[: P.value].copy(),
                   int(P.value), int(st.value))


def dispatch(rt: Routing, tokens: np.ndarray, topk_weights: np.ndarray, dtype: str = "bf16"):
    """Step a4: returns (recv_tokens [P,H] rows, recv_topk_weights f32 [P]);
    (None, None) on overflow (the row operations write nothing)."""
    if rt.overflow:
        return None, None
    tok = _rows(tokens, dtype)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32)
    H = tok.shape[1]
    out = np.empty((rt.P, H), NP_ROW[dtype])
    ow = np.empty(rt.P, np.float32)
    _load().oracle_dispatch(_ptr(rt.inv), rt.P, rt.K, H, DTYPES[dtype], _ptr(tok), _ptr(w),
                            _ptr(out), _ptr(ow))
    return out, ow


def combine(rt: Routing, expert_out: np.ndarray, dtype: str = "bf16"):
    """Step a5: result [T,H] = round(sum_k f32(expert_out[slot[t,k]]))."""
    if rt.overflow:
        return None
    rows = _rows(expert_out, dtype)
    H = rows.shape[1]
    assert rows.shape[0] >= rt.P
    out = np.empty((rt.T, H), NP_ROW[dtype])
    _load().oracle_gather_sum(_ptr(rt.slot), rt.T, rt.K, H, DTYPES[dtype], _ptr(rows), _ptr(out))
    return out


def combine_bwd(rt: Routing, grad: np.ndarray, dtype: str = "bf16"):
    """Step a6: grad_expert_out [P,H], padded rows zero."""
    if rt.overflow:
        return None
    g = _rows(grad, dtype)
    H = g.shape[1]
    out = np.empty((rt.P, H), NP_ROW[dtype])
    _load().oracle_combine_bwd(_ptr(rt.inv), rt.P, rt.K, H, DTYPES[dtype], _ptr(g), _ptr(out))
    return out


def dispatch_bwd(rt: Routing, grad: np.ndarray, g_recv_topk_weights: Optional[np.ndarray],
                 dtype: str = "bf16"):
    """Step a7: (grad_tokens [T,H], grad_topk_weights f32 [T,K])."""
    if rt.overflow:
        return None, None
    rows = _rows(grad, dtype)
    H = rows.shape[1]
    assert rows.shape[0] >= rt.P
    out = np.empty((rt.T, H), NP_ROW[dtype])
    lib = _load()
    lib.oracle_gather_sum(_ptr(rt.slot), rt.T, rt.K, H, DTYPES[dtype], _ptr(rows), _ptr(out))
    gw = None
    if g_recv_topk_weights is not None:
        gw = np.ascontiguousarray(g_recv_topk_weights, dtype=np.float32)
        assert gw.shape[0] >= rt.P
    ow = np.empty((rt.T, rt.K), np.float32)
    lib.oracle_weight_gather(_ptr(rt.slot), rt.T, rt.K, _ptr(gw), _ptr(ow))
    return out, ow


def combine_weighted(rt: Routing, expert_out: np.ndarray, recv_topk_weights: np.ndarray,
                     dtype: str = "bf16"):
    """Weighted combine: result [T,H] = round(sum_k f32(w[slot] * expert_out[slot]))."""
    if rt.overflow:
        return None
    rows = _rows(expert_out, dtype)
    w = np.ascontiguousarray(recv_topk_weights, dtype=np.float32)
    H = rows.shape[1]
    assert rows.shape[0] >= rt.P and w.shape[0] >= rt.P
    out = np.empty((rt.T, H), NP_ROW[dtype])
    _load().oracle_gather_weighted_sum(_ptr(rt.slot), rt.T, rt.K, H, DTYPES[dtype], _ptr(rows),
                                       _ptr(w), _ptr(out))
    return out


def combine_bwd_weighted(rt: Routing, grad: np.ndarray, recv_topk_weights: np.ndarray,
                         expert_out: np.ndarray, dtype: str = "bf16"):
    """Backward of the weighted combine: (grad_expert_out [P,H],
    g_recv_topk_weights float64 [P])."""
    if rt.overflow:
        return None, None
    g = _rows(grad, dtype)
    w = np.ascontiguousarray(recv_topk_weights, dtype=np.float32)
    rows = _rows(expert_out, dtype)
    H = g.shape[1]
    assert rows.shape[0] >= rt.P and w.shape[0] >= rt.P
    out = np.empty((rt.P, H), NP_ROW[dtype])
    gw = np.empty(rt.P, np.float64)
    _load().oracle_combine_bwd_weighted(_ptr(rt.inv), rt.P, rt.K, H, DTYPES[dtype], _ptr(g),
                                        _ptr(w), _ptr(rows), _ptr(out), _ptr(gw))
    return out, gw


# ----------------------------------------------------------------------------
# Sharded expert parallelism: N ranks, rank q owning experts [q*E/N, (q+1)*E/N)
# (TransformerEngine PR #3035, "Sequence Diagram": routing-table all-gather in
# prepare, push of token rows in dispatch, pull in combine, reverse scatter
# and reverse gather in the backward pass).
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class ShardRouting:
    """Result of the sharded prepare over all N ranks."""

    N: int
    K: int
    E: int
    A: int
    R: int
    tokens_per_rank: list
    counts: np.ndarray        # int32 [E], over all ranks
    offsets: np.ndarray       # int32 [E+1], first row of each expert's block on its owner
    P: np.ndarray             # int64 [N], rows in use per owner
    slot: list                # per source rank: int32 [T_r, K], row on the owner or -1
    dest: list                # per source rank: int32 [T_r, K], owner rank or -1
    inv: list                 # per owner: int32 [P_q], concatenated route index or -1
    status: np.ndarray        # uint32 [N], per rank

    @property
    def overflow(self) -> bool:
        return bool(self.status[0] & STATUS_OVERFLOW)

    def local_counts(self, q: int) -> np.ndarray:
        """Counts of owner q's own experts (summed over source ranks)."""
        el = self.E // self.N
        return self.counts[q * el:(q + 1) * el].copy()

    def local_offsets(self, q: int) -> np.ndarray:
        """Offsets of owner q's experts, [E/N + 1], ending with P[q]."""
        el = self.E // self.N
        return np.concatenate([self.offsets[q * el:(q + 1) * el], [self.P[q]]]).astype(np.int32)

    def _cat(self, arrs):
        return np.ascontiguousarray(np.concatenate([np.asarray(a).reshape(-1, self.K) for a in arrs]))


def shard_prepare(idx_per_rank, num_experts: int, alignment: int, num_ranks: int,
                  recv_capacity: Optional[int] = None) -> ShardRouting:
    """Sharded prepare over every rank's topk_idx (the all-gathered table)."""
    lib = _load()
    N, E, A = int(num_ranks), int(num_experts), int(alignment)
    assert len(idx_per_rank) == N
    arrs = [np.ascontiguousarray(a, dtype=np.int64) for a in idx_per_rank]
    K = arrs[0].shape[1]
    tpr = np.array([a.shape[0] for a in arrs], np.int64)
    idx = np.ascontiguousarray(np.concatenate([a.reshape(-1, K) for a in arrs]))
    n = int(idx.size)
    room = max(n + (E // N) * (A - 1), 1)
    R = room if recv_capacity is None else int(recv_capacity)
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    P = np.zeros(N, np.int64)
    slot = np.zeros(max(n, 1), np.int32)
    dest = np.zeros(max(n, 1), np.int32)
    inv = np.zeros(N * room, np.int32)
    st = np.zeros(N, np.uint32)
    rc = lib.oracle_shard_prepare(_ptr(idx), _ptr(tpr), N, K, E, A, R, room, _ptr(counts),
                                  _ptr(offsets), _ptr(P), _ptr(slot), _ptr(dest), _ptr(inv), _ptr(st))
    if rc != 0:
        raise ValueError("oracle_shard_prepare rejected its arguments")
    cuts = np.cumsum(np.concatenate([[0], tpr * K]))
    slots = [slot[cuts[r]:cuts[r + 1]].reshape(-1, K).copy() for r in range(N)]
    dests = [dest[cuts[r]:cuts[r + 1]].reshape(-1, K).copy() for r in range(N)]
    invs = [inv[q * room:q * room + (P[q] if P[q] <= room else 0)].copy() for q in range(N)]
    return ShardRouting(N, K, E, A, R, [int(x) for x in tpr], counts, offsets, P, slots, dests,
                        invs, st)


def shard_dispatch(sr: ShardRouting, tokens_per_rank, weights_per_rank, dtype: str = "bf16"):
    """Push: per owner q, (recv_tokens [P_q, H], recv_topk_weights f32 [P_q]),
    padding rows zero; None on overflow."""
    if sr.overflow:
        return None
    tok = np.ascontiguousarray(np.concatenate([_rows(t, dtype) for t in tokens_per_rank]))
    w = np.ascontiguousarray(np.concatenate([np.asarray(x, np.float32).reshape(-1, sr.K)
                                             for x in weights_per_rank]))
    H = tok.shape[1]
    out = []
    for q in range(sr.N):
        Pq = int(sr.P[q])
        rows = np.empty((Pq, H), NP_ROW[dtype])
        rw = np.empty(Pq, np.float32)
        _load().oracle_dispatch(_ptr(sr.inv[q]), Pq, sr.K, H, DTYPES[dtype], _ptr(tok), _ptr(w),
                                _ptr(rows), _ptr(rw))
        out.append((rows, rw))
    return out


def shard_combine_bwd(sr: ShardRouting, grad_per_rank, dtype: str = "bf16"):
    """Reverse scatter: per owner q, grad_expert_out [P_q, H], padding rows zero."""
    if sr.overflow:
        return None
    g = np.ascontiguousarray(np.concatenate([_rows(x, dtype) for x in grad_per_rank]))
    H = g.shape[1]
    out = []
    for q in range(sr.N):
        Pq = int(sr.P[q])
        rows = np.empty((Pq, H), NP_ROW[dtype])
        _load().oracle_combine_bwd(_ptr(sr.inv[q]), Pq, sr.K, H, DTYPES[dtype], _ptr(g), _ptr(rows))
        out.append(rows)
    return out


def _row_table(arrs, dtype):
    keep = [np.ascontiguousarray(a, dtype=NP_ROW[dtype]) for a in arrs]
    table = (ctypes.c_void_p * len(keep))(*[a.ctypes.data for a in keep])
    return keep, table


def shard_combine(sr: ShardRouting, rows_per_owner, dtype: str = "bf16"):
    """Pull: per source rank, result [T_r, H] = round(sum_k f32(rows of the
    route's owner at its slot)), k ascending from +0.0f."""
    if sr.overflow:
        return None
    keep, table = _row_table(rows_per_owner, dtype)
    H = keep[0].shape[1]
    slot, dest = sr._cat(sr.slot), sr._cat(sr.dest)
    T = slot.shape[0]
    out = np.empty((T, H), NP_ROW[dtype])
    _load().oracle_shard_gather_sum(_ptr(slot), _ptr(dest), T, sr.K, H, DTYPES[dtype], table,
                                    _ptr(out))
    cuts = np.cumsum([0] + sr.tokens_per_rank)
    return [out[cuts[r]:cuts[r + 1]].copy() for r in range(sr.N)]


def shard_dispatch_bwd(sr: ShardRouting, grad_per_owner, g_recv_w_per_owner, dtype: str = "bf16"):
    """Reverse gather: per source rank (grad_tokens [T_r, H], grad_topk_weights
    f32 [T_r, K]); weight gradients all zero when g_recv_w_per_owner is None."""
    if sr.overflow:
        return None
    toks = shard_combine(sr, grad_per_owner, dtype)
    slot, dest = sr._cat(sr.slot), sr._cat(sr.dest)
    n = slot.size
    gw = np.empty(n, np.float32)
    if g_recv_w_per_owner is None:
        _load().oracle_shard_weight_gather(_ptr(slot), _ptr(dest), n, None, _ptr(gw))
    else:
        keep = [np.ascontiguousarray(a, dtype=np.float32) for a in g_recv_w_per_owner]
        table = (ctypes.c_void_p * len(keep))(*[a.ctypes.data for a in keep])
        _load().oracle_shard_weight_gather(_ptr(slot), _ptr(dest), n, table, _ptr(gw))
    cuts = np.cumsum([0] + [t * sr.K for t in sr.tokens_per_rank])
    return [(toks[r], gw[cuts[r]:cuts[r + 1]].reshape(-1, sr.K).copy()) for r in range(sr.N)]


# ----------------------------------------------------------------------------
# Rank-major receive layout (TransformerEngine PR #3035, review thread on the
# receive buffers: at most max_tokens_per_rank x num_ranks rows per owner, the
# owner permuting locally into expert-major order).  Readings in the header
# of ep_oracle.c.
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class RankMajorRouting:
    """Result of the rank-major prepare over all N ranks."""

    N: int
    K: int
    E: int
    R: int
    tokens_per_rank: list
    counts: np.ndarray        # int32 [N, N]: tokens of rank r going to owner q
    M: np.ndarray             # int64 [N], rows each owner receives
    row: list                 # per source rank: int32 [T_r, K], row on the route's owner or -1
    dest: list                # per source rank: int32 [T_r, K], owner or -1
    first: list               # per source rank: bool [T_r, K], first route of its owner in the token
    src: list                 # per owner: int64 [M_q], concatenated token index of each row
    status: np.ndarray        # uint32 [N]

    @property
    def overflow(self) -> bool:
        return bool(self.status[0] & STATUS_OVERFLOW)

    def _cat(self, arrs):
        return np.ascontiguousarray(np.concatenate([np.asarray(a).reshape(-1, self.K) for a in arrs]))

    def first_rows(self):
        """Concatenated [T, K] map of the row kernels: the row at each owner's
        first route in the token, -1 elsewhere."""
        return np.ascontiguousarray(np.where(self._cat(self.first), self._cat(self.row), -1).astype(np.int32))


def rm_prepare(idx_per_rank, num_experts: int, num_ranks: int,
               recv_capacity: Optional[int] = None) -> RankMajorRouting:
    """Rank-major prepare over every rank's topk_idx."""
    lib = _load()
    N, E = int(num_ranks), int(num_experts)
    assert len(idx_per_rank) == N
    arrs = [np.ascontiguousarray(a, dtype=np.int64) for a in idx_per_rank]
    K = arrs[0].shape[1]
    tpr = np.array([a.shape[0] for a in arrs], np.int64)
    idx = np.ascontiguousarray(np.concatenate([a.reshape(-1, K) for a in arrs]))
    T = int(tpr.sum())
    room = max(T, 1)
    R = room if recv_capacity is None else int(recv_capacity)
    counts = np.zeros(N * N, np.int32)
    M = np.zeros(N, np.int64)
    n = max(T * K, 1)
    row, dest, first = np.zeros(n, np.int32), np.zeros(n, np.int32), np.zeros(n, np.int32)
    src = np.zeros(N * room, np.int64)
    st = np.zeros(N, np.uint32)
    rc = lib.oracle_rm_prepare(_ptr(idx), _ptr(tpr), N, K, E, R, room, _ptr(counts), _ptr(M),
                               _ptr(row), _ptr(dest), _ptr(first), _ptr(src), _ptr(st))
    if rc != 0:
        raise ValueError("oracle_rm_prepare rejected its arguments")
    cuts = np.cumsum(np.concatenate([[0], tpr * K]))
    split = lambda a: [a[cuts[r]:cuts[r + 1]].reshape(-1, K).copy() for r in range(N)]
    return RankMajorRouting(N, K, E, R, [int(x) for x in tpr], counts.reshape(N, N), M,
                            split(row), split(dest), [f.astype(bool) for f in split(first)],
                            [src[q * room:q * room + M[q]].copy() for q in range(N)], st)


def rm_dispatch(rr: RankMajorRouting, idx_per_rank, tokens_per_rank, weights_per_rank,
                dtype: str = "bf16"):
    """Push: per owner q, (recv_tokens [M_q, H], recv_topk_idx int64 [M_q, K]
    relative to q, recv_topk_weights f32 [M_q, K]); None on overflow."""
    if rr.overflow:
        return None
    K = rr.K
    idx = rr._cat([np.asarray(a, np.int64) for a in idx_per_rank]).astype(np.int64)
    tok = np.ascontiguousarray(np.concatenate([_rows(t, dtype) for t in tokens_per_rank]))
    w = np.ascontiguousarray(np.concatenate([np.asarray(x, np.float32).reshape(-1, K)
                                             for x in weights_per_rank]))
    H = tok.shape[1]
    out = []
    for q in range(rr.N):
        Mq = int(rr.M[q])
        rows = np.empty((Mq, H), NP_ROW[dtype])
        ids = np.empty((Mq, K), np.int64)
        rw = np.empty((Mq, K), np.float32)
        _load().oracle_rm_dispatch(_ptr(np.ascontiguousarray(rr.src[q])), Mq, _ptr(idx), _ptr(w), K, rr.E,
                                   rr.N, q, H, DTYPES[dtype], _ptr(tok), _ptr(rows), _ptr(ids), _ptr(rw))
        out.append((rows, ids, rw))
    return out


def rm_combine_bwd(rr: RankMajorRouting, grad_per_rank, dtype: str = "bf16"):
    """Reverse of rm_combine: per owner q, grad rows [M_q, H] (the token's
    gradient on every row that holds the token)."""
    if rr.overflow:
        return None
    g = np.ascontiguousarray(np.concatenate([_rows(x, dtype) for x in grad_per_rank]))
    return [g[rr.src[q]].copy() for q in range(rr.N)]


def rm_combine(rr: RankMajorRouting, partial_per_owner, dtype: str = "bf16"):
    """Pull: per source rank, result [T_r, H] = round(sum of f32(owner
    partial rows)), owners in the order of their first route, from +0.0f."""
    if rr.overflow:
        return None
    keep, table = _row_table(partial_per_owner, dtype)
    H = keep[0].shape[1]
    slot, dest = rr.first_rows(), rr._cat(rr.dest)
    T = slot.shape[0]
    out = np.empty((T, H), NP_ROW[dtype])
    _load().oracle_shard_gather_sum(_ptr(slot), _ptr(dest), T, rr.K, H, DTYPES[dtype], table, _ptr(out))
    cuts = np.cumsum([0] + rr.tokens_per_rank)
    return [out[cuts[r]:cuts[r + 1]].copy() for r in range(rr.N)]


def rm_dispatch_bwd(rr: RankMajorRouting, grad_per_owner, g_recv_w_per_owner, dtype: str = "bf16"):
    """Reverse of rm_dispatch: per source rank (grad_tokens [T_r, H],
    grad_topk_weights f32 [T_r, K]); the weight gradient of route (t, k) is
    entry k of the owner's [M_q, K] weight gradient at the token's row, all
    zero when g_recv_w_per_owner is None."""
    if rr.overflow:
        return None
    toks = rm_combine(rr, grad_per_owner, dtype)
    row, dest = rr._cat(rr.row), rr._cat(rr.dest)
    T = row.shape[0]
    gw = np.empty((T, rr.K), np.float32)
    if g_recv_w_per_owner is None:
        _load().oracle_rm_weight_gather(_ptr(row), _ptr(dest), T, rr.K, None, _ptr(gw))
    else:
        keep = [np.ascontiguousarray(a, dtype=np.float32) for a in g_recv_w_per_owner]
        table = (ctypes.c_void_p * len(keep))(*[a.ctypes.data for a in keep])
        _load().oracle_rm_weight_gather(_ptr(row), _ptr(dest), T, rr.K, table, _ptr(gw))
    cuts = np.cumsum([0] + rr.tokens_per_rank)
    return [(toks[r], gw[cuts[r]:cuts[r + 1]].copy()) for r in range(rr.N)]
