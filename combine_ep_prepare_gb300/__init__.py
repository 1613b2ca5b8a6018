"""combine_ep_prepare_gb300 -- MoE expert-parallel dispatch / combine on one
GB300, as hand-written sm_103a CUDA kernels behind a C ABI (libep).

    import combine_ep_prepare_gb300 as ep
    lid, size = ep.ep_register_layer(num_experts=E, top_k=K, hidden=H, max_tokens=T)
    h = ep.alloc_handle(lid, size)
    ep.ep_prepare(h, topk_idx, token_counts, alignment)
    ep.ep_dispatch(h, topk_idx, tokens, topk_weights, recv_tokens, recv_topk_weights)
    ... grouped expert GEMMs on recv_tokens ...
    ep.ep_combine(h, expert_out, result)

The binding (``_libep``) is loaded on first use of an ``ep_*`` name, and
raises ImportError when libep.so has not been built: there is no CPU path.
``workloads`` (seeded synthetic inputs) imports without the library.
"""
from . import workloads  # noqa: F401

_BINDING_NAMES = {
    "EpError", "EpHandle", "alloc_handle", "lib", "SYMBOLS",
    "EP_ST_BAD_INDEX", "EP_ST_OVERFLOW", "EP_ST_TOKENS_MISMATCH", "EP_ST_NOT_PREPARED",
    "ep_abi_version", "ep_last_error", "ep_launch_count", "ep_register_layer",
    "ep_recv_capacity", "ep_prepare", "ep_prepare_static_scratch", "ep_dispatch", "ep_combine", "ep_dispatch_bwd",
    "ep_combine_bwd", "ep_combine_weighted", "ep_combine_weighted_bwd", "ep_expert_offsets", "ep_token_slots", "ep_read_info",
    "EP_ST_COUNTS_MISMATCH", "EP_ST_BAD_POINTER", "EP_ST_TIMEOUT", "ep_register_layer_sharded", "pointer_table",
    "ep_shard_count", "exchange_counts", "ep_shard_prepare", "ep_shard_dispatch", "ep_shard_combine",
    "ep_shard_combine_bwd", "ep_shard_dispatch_bwd", "ep_shard_token_owners",
    "ep_register_layer_rank_major", "ep_rank_major_count", "ep_rank_major_prepare",
    "ep_rank_major_dispatch", "ep_rank_major_combine", "ep_rank_major_combine_bwd",
    "ep_rank_major_dispatch_bwd",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import _libep
        return getattr(_libep, name)
    raise AttributeError(name)
