"""ep_prepare_static_scratch: the routing map built without any device
allocation and without scratch memory from the caller.

Some callers cannot call cudaMalloc: a custom call inside a framework that
plans and owns all device memory (it only receives the buffers the framework
gave it), or a plug-in held to a fixed memory budget.  For them libep keeps the
per-chunk counters of prepare in a fixed 1 MiB __device__ array.  This file
checks, through the C ABI:
  - the map (counts, padded offsets, slot map, status, used and padding rows)
    equals the CPU oracle's bit for bit, and equals ep_prepare's, on two calls
    in a row with different routings (the array is shared by every call and
    keeps the previous call's contents), and the rest of the step runs from it
    as from ep_prepare's map;
  - large batches that fit the array are accepted, up to the largest chunk
    count the array holds, and the first batch past it is refused;
  - a call leaves the device's free memory and torch's pool unchanged.

Kept in a file of its own, collected last.
"""
import numpy as np
import pytest
import torch

from combine_ep_prepare_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

EP_ERR_LIMIT = 6
ARRAY_INTS = 1 << 18


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


def _call_c_abi(ep, h, idx, counts, A, T=None):
    """ep_prepare_static_scratch straight through ctypes (raw pointers)."""
    lib = ep.lib()
    from combine_ep_prepare_gb300._libep import Handle
    return lib.ep_prepare_static_scratch(Handle(h.id, h.mem.data_ptr()), idx.data_ptr(),
                                         idx.shape[0] if T is None else T, counts.data_ptr(), A,
                                         torch.cuda.current_stream().cuda_stream)


def _assert_map_is_oracle(oracle_mod, idx_cpu, E, A, R, counts, offsets, slots, info):
    rt = oracle_mod.prepare(idx_cpu.numpy(), E, A, R)
    assert np.array_equal(counts, rt.token_counts)
    assert np.array_equal(offsets, rt.offsets)
    assert np.array_equal(slots, rt.slot)
    assert info["status"] == rt.status
    assert info["used_rows"] == rt.P
    assert info["padding_rows"] == int((rt.inv < 0).sum())


@pytest.mark.parametrize("E,K,T,A", [(256, 8, 16384, 128), (37, 3, 5000, 7)])
def test_matches_oracle_and_ep_prepare_twice(ep, oracle_mod, E, K, T, A):
    lid, size = ep.ep_register_layer(E, K, 64, T, A)
    R = ep.ep_recv_capacity(lid)
    h_ref = ep.alloc_handle(lid, size)
    h_new = ep.alloc_handle(lid, size)
    for call in range(2):
        if E == 256:
            w = wl.WORKLOADS["dsv3"]
            idx_cpu, _ = wl.routing(w, T=T) if call == 0 else wl.random_routing(T, K, E, seed=91, p_mask=0.2)
        else:
            idx_cpu, _ = wl.random_routing(T, K, E, seed=80 + call, p_mask=0.1 * call, p_bad=0.01 * call)
        idx = idx_cpu.cuda()
        c_ref = torch.full((E,), -1, dtype=torch.int32, device="cuda")
        c_new = torch.full((E,), -2, dtype=torch.int32, device="cuda")
        ep.ep_prepare(h_ref, idx, c_ref, A)
        rc = _call_c_abi(ep, h_new, idx, c_new, A)
        assert rc == 0, ep.ep_last_error()
        torch.cuda.synchronize()
        o_ref, s_ref, i_ref = _routing_map(ep, h_ref, E, T, K)
        o_new, s_new, i_new = _routing_map(ep, h_new, E, T, K)
        _assert_map_is_oracle(oracle_mod, idx_cpu, E, A, R, c_new.cpu().numpy(), o_new, s_new, i_new)
        assert np.array_equal(c_ref.cpu().numpy(), c_new.cpu().numpy())
        assert np.array_equal(o_ref, o_new)
        assert np.array_equal(s_ref, s_new)
        assert i_ref == i_new
        # and the rest of the step runs from that map as from ep_prepare's
        H = 64
        tok = wl.bf16_normal(T, H, seed=5 + call).cuda()
        wts = torch.rand(T, K, device="cuda")
        outs = []
        for h in (h_ref, h_new):
            recv = torch.zeros(R, H, dtype=torch.bfloat16, device="cuda")
            rw = torch.zeros(R, dtype=torch.float32, device="cuda")
            res = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
            ep.ep_dispatch(h, idx, tok, wts, recv, rw)
            ep.ep_combine(h, recv, res)
            outs.append((recv.view(torch.int16).cpu(), res.view(torch.int16).cpu()))
        assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


# Batches past the ~2.5M routes where chunks of 512 routes per warp first
# outnumber two per SM; the array still holds their counters.  The last case
# is the largest batch the array holds at E = 1024: chunks of 8 warps x 512
# routes, 255 chunks, (1024 + 1) x 255 = 261,375 of the 262,144 counters.
@pytest.mark.parametrize("E,K,T,A", [(8, 2, 2_000_000, 128), (256, 8, 400_000, 16),
                                     (1024, 8, 130_560, 3)])
def test_large_batches_that_fit(ep, oracle_mod, E, K, T, A):
    lid, size = ep.ep_register_layer(E, K, 8, T, A)
    R = ep.ep_recv_capacity(lid)
    h = ep.alloc_handle(lid, size)
    idx_cpu, _ = wl.random_routing(T, K, E, seed=7 + E, p_mask=0.05, p_bad=0.001)
    idx = idx_cpu.cuda()
    counts = torch.full((E,), -2, dtype=torch.int32, device="cuda")
    rc = _call_c_abi(ep, h, idx, counts, A)
    assert rc == 0, ep.ep_last_error()
    torch.cuda.synchronize()
    off, slots, info = _routing_map(ep, h, E, T, K)
    _assert_map_is_oracle(oracle_mod, idx_cpu, E, A, R, counts.cpu().numpy(), off, slots, info)


def test_first_batch_past_the_array_is_refused(ep):
    E, K = 1024, 8
    T = 130_561  # one route more than 255 chunks of 4096 routes: 256 x 1025 counters
    assert 256 * (E + 1) > ARRAY_INTS >= 255 * (E + 1)
    lid, size = ep.ep_register_layer(E, K, 8, T, 1)
    h = ep.alloc_handle(lid, size)
    idx = torch.zeros(T, K, dtype=torch.int64, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    before = ep.ep_launch_count()
    rc = _call_c_abi(ep, h, idx, counts, 1)
    assert rc == EP_ERR_LIMIT
    assert "fixed scratch" in ep.ep_last_error()
    assert ep.ep_launch_count() == before


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
    assert rc == EP_ERR_LIMIT  # before any launch
    assert "fixed scratch" in ep.ep_last_error()
    assert ep.ep_launch_count() == before


def test_allocates_nothing(ep):
    """After a first call on the device (which looks up the array's address
    and loads the kernels), further calls change neither the device's free
    memory nor torch's caching pool."""
    E, K, T, A = 256, 8, 16384, 128
    lid, size = ep.ep_register_layer(E, K, 8, T, A)
    h = ep.alloc_handle(lid, size)
    idx = wl.routing(wl.WORKLOADS["dsv3"], T=T)[0].cuda()
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    assert _call_c_abi(ep, h, idx, counts, A) == 0, ep.ep_last_error()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    res0, alloc0 = torch.cuda.memory_reserved(), torch.cuda.memory_allocated()
    for _ in range(3):
        assert _call_c_abi(ep, h, idx, counts, A) == 0, ep.ep_last_error()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_reserved() == res0
    assert torch.cuda.memory_allocated() == alloc0
