"""ctypes binding of libep (include/ep.h).

Argument marshalling only: tensors become device pointers and sizes, the
current torch stream becomes a cudaStream_t, status codes become
exceptions.  Every step of the path runs in libep's CUDA kernels; there is no
fallback, and importing this module fails loudly when libep.so is missing.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import library_path

EP_OK = 0
EP_ST_BAD_INDEX = 1
EP_ST_OVERFLOW = 2
EP_ST_TOKENS_MISMATCH = 4
EP_ST_NOT_PREPARED = 8
EP_ST_COUNTS_MISMATCH = 16
EP_ST_BAD_POINTER = 32
EP_ST_TIMEOUT = 64
ERROR_NAMES = {1: "EP_ERR_INVALID_ARG", 2: "EP_ERR_SHAPE", 3: "EP_ERR_UNSUPPORTED_ARCH",
               4: "EP_ERR_CUDA", 5: "EP_ERR_NOT_REGISTERED", 6: "EP_ERR_LIMIT"}


class EpError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__("%s: %s" % (ERROR_NAMES.get(code, str(code)), message))
        self.code = code


class LayerConfig(ctypes.Structure):
    _fields_ = [("num_experts", ctypes.c_int64), ("top_k", ctypes.c_int64),
                ("hidden", ctypes.c_int64), ("max_tokens", ctypes.c_int64),
                ("max_alignment", ctypes.c_int64), ("recv_capacity", ctypes.c_int64),
                ("dtype", ctypes.c_int64)]


# Payload element types (ep_dtype_t) and the torch dtype of each.
DTYPE_CODES = {"bf16": 0, "fp16": 1, "fp32": 2}
TORCH_DTYPES = {0: torch.bfloat16, 1: torch.float16, 2: torch.float32}
_layer_dtype = {}  # layer id -> torch dtype of its payload rows


class Handle(ctypes.Structure):
    _fields_ = [("id", ctypes.c_uint64), ("mem", ctypes.c_void_p)]


class Info(ctypes.Structure):
    _fields_ = [("status", ctypes.c_uint32), ("num_tokens", ctypes.c_int32),
                ("used_rows", ctypes.c_int32), ("padding_rows", ctypes.c_int32)]


def _load(path=None):
    path = path or library_path()
    if not os.path.exists(path):
        raise ImportError("libep.so is not built (%s); run __graft_entry__.build() "
                          "or python -m combine_ep_prepare_gb300.build" % path)
    lib = ctypes.CDLL(path)
    u64, i64, p, st = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    sig = {
        "ep_abi_version": ([], ctypes.c_uint32),
        "ep_last_error": ([], ctypes.c_char_p),
        "ep_launch_count": ([], ctypes.c_uint64),
        "ep_register_layer": ([LayerConfig, ctypes.POINTER(u64), ctypes.POINTER(ctypes.c_size_t)], st),
        "ep_recv_capacity": ([u64, ctypes.POINTER(i64)], st),
        "ep_prepare": ([Handle, p, i64, p, i64, p], st),
        "ep_prepare_static_scratch": ([Handle, p, i64, p, i64, p], st),
        "ep_dispatch": ([Handle, p, i64, p, p, p, p, p], st),
        "ep_combine": ([Handle, p, i64, p, p], st),
        "ep_dispatch_bwd": ([Handle, p, p, i64, p, p, p], st),
        "ep_combine_bwd": ([Handle, p, i64, p, p], st),
        "ep_combine_weighted": ([Handle, p, p, i64, p, p], st),
        "ep_combine_weighted_bwd": ([Handle, p, p, p, i64, p, p, p], st),
        "ep_expert_offsets": ([Handle, p, p], st),
        "ep_token_slots": ([Handle, p, i64, p], st),
        "ep_read_info": ([Handle, ctypes.POINTER(Info), p], st),
        "ep_register_layer_sharded": ([LayerConfig, i64, i64, ctypes.POINTER(u64),
                                       ctypes.POINTER(ctypes.c_size_t)], st),
        "ep_shard_count": ([Handle, p, i64, p, p], st),
        "ep_shard_prepare": ([Handle, p, i64, p, p, i64, p], st),
        "ep_shard_dispatch": ([Handle, i64, p, p, p, p, p], st),
        "ep_shard_combine": ([Handle, p, i64, p, p], st),
        "ep_shard_combine_bwd": ([Handle, p, i64, p, p], st),
        "ep_shard_dispatch_bwd": ([Handle, p, p, i64, p, p, p], st),
        "ep_shard_token_owners": ([Handle, p, i64, p], st),
        "ep_register_layer_rank_major": ([LayerConfig, i64, i64, ctypes.POINTER(u64),
                                          ctypes.POINTER(ctypes.c_size_t)], st),
        "ep_rank_major_count": ([Handle, p, i64, p, p], st),
        "ep_rank_major_prepare": ([Handle, p, i64, p, p, p], st),
        "ep_rank_major_dispatch": ([Handle, p, i64, p, p, p, p, p, p], st),
        "ep_rank_major_combine": ([Handle, p, i64, p, p], st),
        "ep_rank_major_combine_bwd": ([Handle, p, i64, p, p], st),
        "ep_rank_major_dispatch_bwd": ([Handle, p, p, i64, p, p, p], st),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()
SYMBOLS = ("ep_abi_version", "ep_last_error", "ep_launch_count", "ep_register_layer",
           "ep_recv_capacity", "ep_prepare", "ep_prepare_static_scratch", "ep_dispatch", "ep_combine", "ep_dispatch_bwd",
           "ep_combine_bwd", "ep_combine_weighted", "ep_combine_weighted_bwd", "ep_expert_offsets", "ep_token_slots", "ep_read_info",
           "ep_register_layer_sharded", "ep_shard_count", "ep_shard_prepare", "ep_shard_dispatch",
           "ep_shard_combine", "ep_shard_combine_bwd", "ep_shard_dispatch_bwd", "ep_shard_token_owners",
           "ep_register_layer_rank_major", "ep_rank_major_count", "ep_rank_major_prepare",
           "ep_rank_major_dispatch", "ep_rank_major_combine", "ep_rank_major_combine_bwd",
           "ep_rank_major_dispatch_bwd")


def lib():
    return _lib


def _check(code: int):
    if code != EP_OK:
        raise EpError(code, _lib.ep_last_error().decode())


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor") -> Optional[int]:
    if t is None:
        return None
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if t.device.type != "cuda":
        raise ValueError("%s must be a CUDA tensor" % name)
    return t.data_ptr() or None


class EpHandle:
    """A registered layer id plus the caller-owned handle memory of one
    in-flight step (TransformerEngine's NVTEEpHandle {id, mem})."""

    def __init__(self, layer_id: int, mem: torch.Tensor):
        self.id = int(layer_id)
        self.mem = mem

    @property
    def c(self) -> Handle:
        return Handle(self.id, self.mem.data_ptr())


def ep_abi_version() -> int:
    return int(_lib.ep_abi_version())


def ep_last_error() -> str:
    return _lib.ep_last_error().decode()


def ep_launch_count() -> int:
    return int(_lib.ep_launch_count())


def _dtype_code(dtype) -> int:
    if not isinstance(dtype, str):
        dtype = {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float32: "fp32"}.get(dtype, str(dtype))
    if dtype not in DTYPE_CODES:
        raise TypeError("payload dtype must be bf16, fp16 or fp32, got %s" % dtype)
    return DTYPE_CODES[dtype]


def ep_register_layer(num_experts: int, top_k: int, hidden: int, max_tokens: int,
                      max_alignment: int = 128, recv_capacity: int = 0, dtype="bf16"):
    """Returns (layer_id, handle_mem_size_bytes).  dtype: "bf16", "fp16",
    "fp32" or the matching torch dtype."""
    code = _dtype_code(dtype)
    cfg = LayerConfig(num_experts, top_k, hidden, max_tokens, max_alignment, recv_capacity, code)
    lid = ctypes.c_uint64(0)
    size = ctypes.c_size_t(0)
    _check(_lib.ep_register_layer(cfg, ctypes.byref(lid), ctypes.byref(size)))
    _layer_dtype[int(lid.value)] = TORCH_DTYPES[code]
    return int(lid.value), int(size.value)


def ep_register_layer_sharded(num_experts: int, top_k: int, hidden: int, max_tokens: int,
                              num_ranks: int, rank: int, max_alignment: int = 128,
                              recv_capacity: int = 0, dtype="bf16"):
    """A layer of rank `rank` of `num_ranks` (expert parallelism): rank q
    owns experts [q*E/N, (q+1)*E/N).  max_tokens is the largest batch of any
    rank.  Returns (layer_id, handle_mem_size_bytes)."""
    code = _dtype_code(dtype)
    cfg = LayerConfig(num_experts, top_k, hidden, max_tokens, max_alignment, recv_capacity, code)
    lid = ctypes.c_uint64(0)
    size = ctypes.c_size_t(0)
    _check(_lib.ep_register_layer_sharded(cfg, num_ranks, rank, ctypes.byref(lid), ctypes.byref(size)))
    _layer_dtype[int(lid.value)] = TORCH_DTYPES[code]
    return int(lid.value), int(size.value)


def _payload(h) -> "torch.dtype":
    return _layer_dtype.get(h.id, torch.bfloat16)


def ep_recv_capacity(layer_id: int) -> int:
    rows = ctypes.c_int64(0)
    _check(_lib.ep_recv_capacity(layer_id, ctypes.byref(rows)))
    return int(rows.value)


def alloc_handle(layer_id: int, size: int, device="cuda") -> EpHandle:
    """Convenience: allocate handle memory (once, outside the step) with torch,
    zero-filled, so that memory the caching allocator hands back from an
    earlier handle cannot pass for a prepared one."""
    return EpHandle(layer_id, torch.zeros(size, dtype=torch.uint8, device=device))


def ep_prepare(h: EpHandle, topk_idx: torch.Tensor, token_counts: torch.Tensor,
               alignment: int, stream=None):
    T = topk_idx.shape[0]
    _check(_lib.ep_prepare(h.c, _ptr(topk_idx, torch.int64, "topk_idx"), T,
                           _ptr(token_counts, torch.int32, "token_counts"), alignment,
                           _stream(stream)))


def ep_prepare_static_scratch(h: EpHandle, topk_idx: torch.Tensor, token_counts: torch.Tensor,
                              alignment: int, stream=None):
    """ep_prepare without any scratch from the caller: for code that cannot
    allocate device memory (see include/ep.h)."""
    T = topk_idx.shape[0]
    _check(_lib.ep_prepare_static_scratch(h.c, _ptr(topk_idx, torch.int64, "topk_idx"), T,
                                          _ptr(token_counts, torch.int32, "token_counts"),
                                          alignment, _stream(stream)))


def ep_dispatch(h: EpHandle, topk_idx: torch.Tensor, tokens: torch.Tensor,
                topk_weights: torch.Tensor, recv_tokens: torch.Tensor,
                recv_topk_weights: torch.Tensor, stream=None):
    T = tokens.shape[0]
    _check(_lib.ep_dispatch(h.c, _ptr(topk_idx, torch.int64, "topk_idx"), T,
                            _ptr(tokens, _payload(h), "tokens"),
                            _ptr(topk_weights, torch.float32, "topk_weights"),
                            _ptr(recv_tokens, _payload(h), "recv_tokens"),
                            _ptr(recv_topk_weights, torch.float32, "recv_topk_weights"),
                            _stream(stream)))


def ep_combine(h: EpHandle, expert_out: torch.Tensor, result: torch.Tensor, stream=None):
    T = result.shape[0]
    _check(_lib.ep_combine(h.c, _ptr(expert_out, _payload(h), "expert_out"), T,
                           _ptr(result, _payload(h), "result"), _stream(stream)))


def ep_dispatch_bwd(h: EpHandle, grad: torch.Tensor, g_recv_topk_weights: Optional[torch.Tensor],
                    grad_tokens: torch.Tensor, grad_topk_weights: torch.Tensor, stream=None):
    T = grad_tokens.shape[0]
    _check(_lib.ep_dispatch_bwd(h.c, _ptr(grad, _payload(h), "grad"),
                                _ptr(g_recv_topk_weights, torch.float32, "g_recv_topk_weights"), T,
                                _ptr(grad_tokens, _payload(h), "grad_tokens"),
                                _ptr(grad_topk_weights, torch.float32, "grad_topk_weights"),
                                _stream(stream)))


def ep_combine_bwd(h: EpHandle, grad: torch.Tensor, grad_expert_out: torch.Tensor, stream=None):
    T = grad.shape[0]
    _check(_lib.ep_combine_bwd(h.c, _ptr(grad, _payload(h), "grad"), T,
                               _ptr(grad_expert_out, _payload(h), "grad_expert_out"),
                               _stream(stream)))


def ep_combine_weighted(h: EpHandle, expert_out: torch.Tensor, recv_topk_weights: torch.Tensor,
                        result: torch.Tensor, stream=None):
    T = result.shape[0]
    _check(_lib.ep_combine_weighted(h.c, _ptr(expert_out, _payload(h), "expert_out"),
                                    _ptr(recv_topk_weights, torch.float32, "recv_topk_weights"), T,
                                    _ptr(result, _payload(h), "result"), _stream(stream)))


def ep_combine_weighted_bwd(h: EpHandle, grad: torch.Tensor, expert_out: torch.Tensor,
                            recv_topk_weights: torch.Tensor, grad_expert_out: torch.Tensor,
                            g_recv_topk_weights: torch.Tensor, stream=None):
    T = grad.shape[0]
    _check(_lib.ep_combine_weighted_bwd(h.c, _ptr(grad, _payload(h), "grad"),
                                        _ptr(expert_out, _payload(h), "expert_out"),
                                        _ptr(recv_topk_weights, torch.float32, "recv_topk_weights"), T,
                                        _ptr(grad_expert_out, _payload(h), "grad_expert_out"),
                                        _ptr(g_recv_topk_weights, torch.float32, "g_recv_topk_weights"),
                                        _stream(stream)))


def ep_expert_offsets(h: EpHandle, offsets: torch.Tensor, stream=None):
    _check(_lib.ep_expert_offsets(h.c, _ptr(offsets, torch.int32, "offsets"), _stream(stream)))


def ep_token_slots(h: EpHandle, slots: torch.Tensor, stream=None):
    _check(_lib.ep_token_slots(h.c, _ptr(slots, torch.int32, "slots"), slots.shape[0],
                               _stream(stream)))


def ep_read_info(h: EpHandle, stream=None) -> dict:
    info = Info()
    _check(_lib.ep_read_info(h.c, ctypes.byref(info), _stream(stream)))
    return {"status": int(info.status), "num_tokens": int(info.num_tokens),
            "used_rows": int(info.used_rows), "padding_rows": int(info.padding_rows)}


# ----------------------------------------------------------------------------
# Sharded layers (expert parallelism over N ranks)
# ----------------------------------------------------------------------------

def pointer_table(tensors, device=None) -> torch.Tensor:
    """Device array of the tensors' addresses (int64 [N]), for the row calls
    of a sharded layer: entry r = rank r's buffer as this rank's device
    addresses it.  Build it once, outside the step."""
    ptrs = [0 if t is None else t.data_ptr() for t in tensors]
    dev = device if device is not None else next(t.device for t in tensors if t is not None)
    return torch.tensor(ptrs, dtype=torch.int64, device=dev)


def _table(tab: Optional[torch.Tensor], name: str) -> Optional[int]:
    if tab is None:
        return None
    return _ptr(tab, torch.int64, name)


def ep_shard_count(h: EpHandle, topk_idx: torch.Tensor, local_counts: torch.Tensor, stream=None):
    T = topk_idx.shape[0]
    _check(_lib.ep_shard_count(h.c, _ptr(topk_idx, torch.int64, "topk_idx"), T,
                               _ptr(local_counts, torch.int32, "local_counts"), _stream(stream)))


def exchange_counts(local_counts: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather every rank's ep_shard_count output over a
    torch.distributed group: returns int32 [N, E], row r = rank r's counts
    (the routing-table all-gather of the pages' prepare)."""
    import torch.distributed as dist
    n = dist.get_world_size(group)
    flat = local_counts.contiguous().view(-1)
    out = torch.empty(n * flat.numel(), dtype=local_counts.dtype, device=local_counts.device)
    dist.all_gather_into_tensor(out, flat, group=group)
    return out.view((n,) + tuple(local_counts.shape))


def ep_shard_prepare(h: EpHandle, topk_idx: torch.Tensor, all_counts: torch.Tensor,
                     token_counts: torch.Tensor, alignment: int, stream=None):
    T = topk_idx.shape[0]
    _check(_lib.ep_shard_prepare(h.c, _ptr(topk_idx, torch.int64, "topk_idx"), T,
                                 _ptr(all_counts, torch.int32, "all_counts"),
                                 _ptr(token_counts, torch.int32, "token_counts"), alignment,
                                 _stream(stream)))


def ep_shard_dispatch(h: EpHandle, tokens: torch.Tensor, topk_weights: torch.Tensor,
                      recv_tokens: torch.Tensor, recv_topk_weights: torch.Tensor, stream=None):
    """recv_tokens, recv_topk_weights: pointer tables (pointer_table)."""
    T = tokens.shape[0]
    _check(_lib.ep_shard_dispatch(h.c, T, _ptr(tokens, _payload(h), "tokens"),
                                  _ptr(topk_weights, torch.float32, "topk_weights"),
                                  _table(recv_tokens, "recv_tokens"),
                                  _table(recv_topk_weights, "recv_topk_weights"), _stream(stream)))


def ep_shard_combine(h: EpHandle, expert_out: torch.Tensor, result: torch.Tensor, stream=None):
    """expert_out: pointer table."""
    T = result.shape[0]
    _check(_lib.ep_shard_combine(h.c, _table(expert_out, "expert_out"), T,
                                 _ptr(result, _payload(h), "result"), _stream(stream)))


def ep_shard_combine_bwd(h: EpHandle, grad: torch.Tensor, grad_expert_out: torch.Tensor,
                         stream=None):
    """grad_expert_out: pointer table."""
    T = grad.shape[0]
    _check(_lib.ep_shard_combine_bwd(h.c, _ptr(grad, _payload(h), "grad"), T,
                                     _table(grad_expert_out, "grad_expert_out"), _stream(stream)))


def ep_shard_dispatch_bwd(h: EpHandle, grad: torch.Tensor, g_recv_topk_weights: Optional[torch.Tensor],
                          grad_tokens: torch.Tensor, grad_topk_weights: torch.Tensor, stream=None):
    """grad, g_recv_topk_weights: pointer tables (the latter may be None)."""
    T = grad_tokens.shape[0]
    _check(_lib.ep_shard_dispatch_bwd(h.c, _table(grad, "grad"),
                                      _table(g_recv_topk_weights, "g_recv_topk_weights"), T,
                                      _ptr(grad_tokens, _payload(h), "grad_tokens"),
                                      _ptr(grad_topk_weights, torch.float32, "grad_topk_weights"),
                                      _stream(stream)))


def ep_shard_token_owners(h: EpHandle, owners: torch.Tensor, stream=None):
    _check(_lib.ep_shard_token_owners(h.c, _ptr(owners, torch.int32, "owners"), owners.shape[0],
                                      _stream(stream)))


# ----------------------------------------------------------------------------
# Rank-major layers (sharded, at most N * max_tokens received rows per owner;
# the owner permutes them with a single-buffer layer of E/N experts)
# ----------------------------------------------------------------------------

def ep_register_layer_rank_major(num_experts: int, top_k: int, hidden: int, max_tokens: int,
                                 num_ranks: int, rank: int, recv_capacity: int = 0, dtype="bf16"):
    """A rank-major layer of rank `rank` of `num_ranks`.  recv_capacity =
    rows per owner (0: num_ranks * max_tokens).  Returns (layer_id,
    handle_mem_size_bytes)."""
    code = _dtype_code(dtype)
    cfg = LayerConfig(num_experts, top_k, hidden, max_tokens, 1, recv_capacity, code)
    lid = ctypes.c_uint64(0)
    size = ctypes.c_size_t(0)
    _check(_lib.ep_register_layer_rank_major(cfg, num_ranks, rank, ctypes.byref(lid), ctypes.byref(size)))
    _layer_dtype[int(lid.value)] = TORCH_DTYPES[code]
    return int(lid.value), int(size.value)


def ep_rank_major_count(h: EpHandle, topk_idx: torch.Tensor, local_counts: torch.Tensor, stream=None):
    """local_counts: int32 [N], this rank's tokens per owner."""
    T = topk_idx.shape[0]
    _check(_lib.ep_rank_major_count(h.c, _ptr(topk_idx, torch.int64, "topk_idx"), T,
                                    _ptr(local_counts, torch.int32, "local_counts"), _stream(stream)))


def ep_rank_major_prepare(h: EpHandle, topk_idx: torch.Tensor, all_counts: torch.Tensor,
                          recv_rows: torch.Tensor, stream=None):
    """all_counts: int32 [N, N] (exchange_counts of the count call);
    recv_rows: int32 [1], the rows this rank receives."""
    T = topk_idx.shape[0]
    _check(_lib.ep_rank_major_prepare(h.c, _ptr(topk_idx, torch.int64, "topk_idx"), T,
                                      _ptr(all_counts, torch.int32, "all_counts"),
                                      _ptr(recv_rows, torch.int32, "recv_rows"), _stream(stream)))


def ep_rank_major_dispatch(h: EpHandle, topk_idx: torch.Tensor, tokens: torch.Tensor,
                           topk_weights: Optional[torch.Tensor], recv_tokens: torch.Tensor,
                           recv_topk_idx: torch.Tensor, recv_topk_weights: Optional[torch.Tensor],
                           stream=None):
    """recv_tokens, recv_topk_idx, recv_topk_weights: pointer tables (the
    last may be None: ids only)."""
    T = tokens.shape[0]
    _check(_lib.ep_rank_major_dispatch(
        h.c, _ptr(topk_idx, torch.int64, "topk_idx"), T, _ptr(tokens, _payload(h), "tokens"),
        None if topk_weights is None else _ptr(topk_weights, torch.float32, "topk_weights"),
        _table(recv_tokens, "recv_tokens"), _table(recv_topk_idx, "recv_topk_idx"),
        _table(recv_topk_weights, "recv_topk_weights"), _stream(stream)))


def ep_rank_major_combine(h: EpHandle, partial: torch.Tensor, result: torch.Tensor, stream=None):
    """partial: pointer table of the owners' [M_q, H] partial rows."""
    T = result.shape[0]
    _check(_lib.ep_rank_major_combine(h.c, _table(partial, "partial"), T,
                                      _ptr(result, _payload(h), "result"), _stream(stream)))


def ep_rank_major_combine_bwd(h: EpHandle, grad: torch.Tensor, grad_recv: torch.Tensor, stream=None):
    """grad_recv: pointer table."""
    T = grad.shape[0]
    _check(_lib.ep_rank_major_combine_bwd(h.c, _ptr(grad, _payload(h), "grad"), T,
                                          _table(grad_recv, "grad_recv"), _stream(stream)))


def ep_rank_major_dispatch_bwd(h: EpHandle, grad_recv: torch.Tensor,
                               g_recv_topk_weights: Optional[torch.Tensor], grad_tokens: torch.Tensor,
                               grad_topk_weights: torch.Tensor, stream=None):
    """grad_recv, g_recv_topk_weights: pointer tables (the latter may be None)."""
    T = grad_tokens.shape[0]
    _check(_lib.ep_rank_major_dispatch_bwd(h.c, _table(grad_recv, "grad_recv"),
                                           _table(g_recv_topk_weights, "g_recv_topk_weights"), T,
                                           _ptr(grad_tokens, _payload(h), "grad_tokens"),
                                           _ptr(grad_topk_weights, torch.float32, "grad_topk_weights"),
                                           _stream(stream)))
