"""ep_prepare_static_scratch: the routing map built without any device
allocation and without scratch memory from the caller.

Some callers cannot call cudaMalloc: a custom call inside a framework that
plans and owns all device memory (it only receives the buffers the framework
gave it), or a plug-in held to a fixed memory budget.  For them libep keeps the
per-chunk counters of prepare in a fixed 1 MiB __device__ array.  This file
checks, through the C ABI, that the result equals ep_prepare's bit for bit
(integer work: counts, padded offsets, slot map, status) on two calls in a
row with different routings -- the array is shared by every call and keeps the
previous call's contents -- and that sizes beyond the array are refused.

Kept in a file of its own, collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from combine_ep_prepare_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_ep_prepare_gb300 as ep
    return ep


def _routing_map(ep, h, E, T, K):
    off = torch.full((E + 1,), -9, dtype=torch.int32, device="cuda")
    slots = torch.full((T, K), -9, dtype=torch.int32, device="cuda")
    ep.ep_expert_offsets(h, off)
    ep.ep_token_slots(h, slots)
    info = ep.ep_read_info(h)
    return off.cpu().numpy(), slots.cpu().numpy(), info


def _call_c_abi(ep, h, idx, counts, A):
    """ep_prepare_static_scratch straight through ctypes (raw pointers)."""
    lib = ep.lib()
    from combine_ep_prepare_gb300._libep import Handle
    rc = lib.ep_prepare_static_scratch(Handle(h.id, h.mem.data_ptr()), idx.data_ptr(),
                                       idx.shape[0], counts.data_ptr(), A,
                                       torch.cuda.current_stream().cuda_stream)
    return rc


@pytest.mark.parametrize("E,K,T,A", [(256, 8, 16384, 128), (37, 3, 5000, 7)])
def test_matches_ep_prepare_twice(ep, E, K, T, A):
    lid, size = ep.ep_register_layer(E, K, 64, T, A)
    h_ref = ep.alloc_handle(lid, size)
    h_new = ep.alloc_handle(lid, size)
    for call in range(2):
        if E == 256:
            w = wl.WORKLOADS["dsv3"]
            idx, _ = wl.routing(w, T=T) if call == 0 else wl.random_routing(T, K, E, seed=91, p_mask=0.2)
        else:
            idx, _ = wl.random_routing(T, K, E, seed=80 + call, p_mask=0.1 * call, p_bad=0.01 * call)
        idx = idx.cuda()
        c_ref = torch.full((E,), -1, dtype=torch.int32, device="cuda")
        c_new = torch.full((E,), -2, dtype=torch.int32, device="cuda")
        ep.ep_prepare(h_ref, idx, c_ref, A)
        rc = _call_c_abi(ep, h_new, idx, c_new, A)
        assert rc == 0, ep.ep_last_error()
        torch.cuda.synchronize()
        o_ref, s_ref, i_ref = _routing_map(ep, h_ref, E, T, K)
        o_new, s_new, i_new = _routing_map(ep, h_new, E, T, K)
        assert np.array_equal(c_ref.cpu().numpy(), c_new.cpu().numpy())
        assert np.array_equal(o_ref, o_new)
        assert np.array_equal(s_ref, s_new)
        assert i_ref == i_new
        # and the rest of the step runs from that map as from ep_prepare's
        H = 64
        tok = wl.bf16_normal(T, H, seed=5 + call).cuda()
        wts = torch.rand(T, K, device="cuda")
        R = ep.ep_recv_capacity(lid)
        outs = []
        for h in (h_ref, h_new):
            recv = torch.zeros(R, H, dtype=torch.bfloat16, device="cuda")
            rw = torch.zeros(R, dtype=torch.float32, device="cuda")
            res = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
            ep.ep_dispatch(h, idx, tok, wts, recv, rw)
            ep.ep_combine(h, recv, res)
            outs.append((recv.view(torch.int16).cpu(), res.view(torch.int16).cpu()))
        assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_refuses_sizes_beyond_the_array(ep):
    E, K = 1024, 32
    T = (1 << 24) // K  # 2^24 routes over 1024 experts cannot fit 1 MiB of counters
    lid, size = ep.ep_register_layer(E, K, 8, T, 1)
    h = ep.EpHandle(lid, torch.empty(256, dtype=torch.uint8, device="cuda"))
    idx = torch.empty(1, dtype=torch.int64, device="cuda")
    counts = torch.empty(1, dtype=torch.int32, device="cuda")
    lib = ep.lib()
    from combine_ep_prepare_gb300._libep import Handle
    before = ep.ep_launch_count()
    rc = lib.ep_prepare_static_scratch(Handle(lid, h.mem.data_ptr()), idx.data_ptr(), T,
                                       counts.data_ptr(), 1, None)
    assert rc == 6  # EP_ERR_LIMIT, before any launch
    assert "fixed scratch" in ep.ep_last_error()
    assert ep.ep_launch_count() == before
