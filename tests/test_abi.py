"""The C ABI without a GPU: the library loads, exports every call that
include/ep.h declares, and its host-side logic (registration, layout sizes,
argument validation, error codes) behaves as documented.  No call here
reaches a kernel launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ep():
    from combine_ep_prepare_gb300 import build
    build.build()
    import combine_ep_prepare_gb300 as ep
    return ep


def header_functions():
    src = open(os.path.join(ROOT, "include", "ep.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(ep_\w+)\s*\(", src, flags=re.M)))


def test_header_symbols_exported(ep):
    names = header_functions()
    assert len(names) >= 13, names
    lib = ctypes.CDLL(ep.lib()._name)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(ep.SYMBOLS)


def test_abi_version(ep):
    assert ep.ep_abi_version() == 4


def test_register_and_capacity(ep):
    lid, size = ep.ep_register_layer(num_experts=256, top_k=8, hidden=7168, max_tokens=16384,
                                     max_alignment=128)
    assert lid >= 1 and size % 256 == 0
    assert ep.ep_recv_capacity(lid) == 16384 * 8 + 256 * 127
    # handle memory holds at least the slot map and the per-chunk counters
    assert size >= 16384 * 8 * 4 + 256 * 4
    lid2, _ = ep.ep_register_layer(8, 2, 4096, 4096, 128, recv_capacity=1000)
    assert lid2 == lid + 1
    assert ep.ep_recv_capacity(lid2) == 1000
    # worst case when experts outnumber routes
    lid3, _ = ep.ep_register_layer(64, 2, 16, 3, 16)
    assert ep.ep_recv_capacity(lid3) == 6 + 6 * 15


@pytest.mark.parametrize("cfg", [
    dict(num_experts=0, top_k=2, hidden=64, max_tokens=10),
    dict(num_experts=1025, top_k=2, hidden=64, max_tokens=10),
    dict(num_experts=8, top_k=0, hidden=64, max_tokens=10),
    dict(num_experts=8, top_k=33, hidden=64, max_tokens=10),
    dict(num_experts=8, top_k=2, hidden=12, max_tokens=10),
    dict(num_experts=8, top_k=2, hidden=0, max_tokens=10),
    dict(num_experts=8, top_k=2, hidden=64, max_tokens=-1),
    dict(num_experts=8, top_k=8, hidden=64, max_tokens=(1 << 21) + 1),
    dict(num_experts=8, top_k=2, hidden=64, max_tokens=10, max_alignment=0),
    dict(num_experts=8, top_k=2, hidden=64, max_tokens=10, recv_capacity=-5),
])
def test_register_rejects(ep, cfg):
    with pytest.raises(ep.EpError) as ei:
        ep.ep_register_layer(**cfg)
    assert ei.value.code in (1, 6)
    assert ep.ep_last_error()


def _raw_handle(ep, lid, mem):
    from combine_ep_prepare_gb300._libep import Handle
    return Handle(lid, mem)


def test_unregistered_and_bad_handle(ep):
    lib = ep.lib()
    h = _raw_handle(ep, 10**9, 4096)
    assert lib.ep_combine(h, 4096, 0, None, None) == 5  # EP_ERR_NOT_REGISTERED
    lid, _ = ep.ep_register_layer(8, 2, 64, 16)
    assert lib.ep_combine(_raw_handle(ep, lid, None), 4096, 0, None, None) == 1
    assert lib.ep_combine(_raw_handle(ep, lid, 4096 + 8), 4096, 0, None, None) == 1  # misaligned
    assert "aligned" in ep.ep_last_error()


def test_shape_and_pointer_checks(ep):
    lib = ep.lib()
    lid, _ = ep.ep_register_layer(8, 2, 64, 16, max_alignment=8)
    h = _raw_handle(ep, lid, 1 << 20)
    # too many tokens
    assert lib.ep_prepare(h, 4096, 17, 4096, 4, None) == 2
    # alignment outside [1, max_alignment]
    assert lib.ep_prepare(h, 4096, 4, 4096, 9, None) == 2
    assert lib.ep_prepare(h, 4096, 4, 4096, 0, None) == 2
    # NULL topk_idx with tokens, NULL counts
    assert lib.ep_prepare(h, None, 4, 4096, 4, None) == 1
    assert lib.ep_prepare(h, 4096, 4, None, 4, None) == 1
    # misaligned payloads
    assert lib.ep_dispatch(h, 4096, 4, 4096 + 2, 4096, 4096, 4096, None) == 1
    assert lib.ep_combine(h, 4096, 4, 4096 + 8, None) == 1
    assert lib.ep_combine_bwd(h, None, 4, 4096, None) == 1
    assert lib.ep_dispatch_bwd(h, 4096, 4096 + 1, 4, 4096, 4096, None) == 1


def test_weighted_and_static_scratch_checks(ep):
    lib = ep.lib()
    lid, _ = ep.ep_register_layer(8, 2, 64, 16, max_alignment=8)
    h = _raw_handle(ep, lid, 1 << 20)
    launches = ep.ep_launch_count()
    # weighted combine: weights are required and float-aligned, payloads 16-byte aligned
    assert lib.ep_combine_weighted(h, 4096, None, 4, 4096, None) == 1
    assert lib.ep_combine_weighted(h, 4096, 4096 + 2, 4, 4096, None) == 1
    assert lib.ep_combine_weighted(h, 4096 + 8, 4096, 4, 4096, None) == 1
    assert lib.ep_combine_weighted(h, 4096, 4096, 17, 4096, None) == 2  # too many tokens
    # its backward: every buffer checked
    assert lib.ep_combine_weighted_bwd(h, 4096, 4096, 4096, 4, 4096, None, None) == 1
    assert lib.ep_combine_weighted_bwd(h, 4096, None, 4096, 4, 4096, 4096, None) == 1
    assert lib.ep_combine_weighted_bwd(h, 4096, 4096, 4096, 4, 4096 + 4, 4096, None) == 1
    # the fixed-scratch prepare validates like ep_prepare
    assert lib.ep_prepare_static_scratch(h, 4096, 17, 4096, 4, None) == 2
    assert lib.ep_prepare_static_scratch(h, 4096, 4, 4096, 9, None) == 2
    assert lib.ep_prepare_static_scratch(h, 4096, 4, None, 4, None) == 1
    assert ep.ep_launch_count() == launches  # rejected before any launch


def test_no_gpu_gives_error_not_crash(ep):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    lib = ep.lib()
    lid, _ = ep.ep_register_layer(8, 2, 64, 16, max_alignment=8)
    h = _raw_handle(ep, lid, 1 << 20)
    rc = lib.ep_prepare(h, 4096, 4, 4096, 4, None)
    assert rc in (3, 4)  # no device: the device check fails, nothing is launched
    assert ep.ep_launch_count() == 0


def test_register_dtypes(ep):
    for dt in ("bf16", "fp16", "fp32"):
        lid, size = ep.ep_register_layer(8, 2, 64, 16, 4, dtype=dt)
        assert lid >= 1 and size > 0
    with pytest.raises(TypeError):
        ep.ep_register_layer(8, 2, 64, 16, 4, dtype="int8")
    # the C ABI itself rejects an unknown payload type
    from combine_ep_prepare_gb300._libep import LayerConfig
    lid = ctypes.c_uint64(0)
    size = ctypes.c_size_t(0)
    rc = ep.lib().ep_register_layer(LayerConfig(8, 2, 64, 16, 4, 0, 7), ctypes.byref(lid), ctypes.byref(size))
    assert rc == 1 and "dtype" in ep.ep_last_error()


def test_binding_checks_payload_tensors(ep):
    """The Python binding rejects a payload of the wrong type, a
    non-contiguous tensor and a host tensor before calling libep."""
    import torch
    lid, size = ep.ep_register_layer(8, 2, 64, 16, 4, dtype="fp16")
    h = ep.EpHandle(lid, torch.empty(size, dtype=torch.uint8))
    f16 = torch.empty(4, 64, dtype=torch.float16)
    with pytest.raises(TypeError, match="float16"):
        ep.ep_combine(h, torch.empty(4, 64, dtype=torch.bfloat16), f16)
    with pytest.raises(ValueError, match="contiguous"):
        ep.ep_combine(h, torch.empty(64, 4, dtype=torch.float16).t(), f16)
    with pytest.raises(ValueError, match="CUDA"):
        ep.ep_combine(h, f16, f16)


def test_binding_constants_match_header(ep):
    """Status bits, error codes and payload-type codes of the binding are the
    ones include/ep.h declares."""
    from combine_ep_prepare_gb300 import _libep
    src = open(os.path.join(ROOT, "include", "ep.h")).read()
    st = {m[0]: int(m[1]) for m in re.findall(r"#define (EP_ST_\w+) (\d+)u", src)}
    assert st == {"EP_ST_BAD_INDEX": _libep.EP_ST_BAD_INDEX, "EP_ST_OVERFLOW": _libep.EP_ST_OVERFLOW,
                  "EP_ST_TOKENS_MISMATCH": _libep.EP_ST_TOKENS_MISMATCH,
                  "EP_ST_NOT_PREPARED": _libep.EP_ST_NOT_PREPARED,
                  "EP_ST_COUNTS_MISMATCH": _libep.EP_ST_COUNTS_MISMATCH,
                  "EP_ST_BAD_POINTER": _libep.EP_ST_BAD_POINTER,
                  "EP_ST_TIMEOUT": _libep.EP_ST_TIMEOUT}
    errs = {int(m[1]): m[0] for m in re.findall(r"(EP_ERR_\w+) = (\d+)", src)}
    assert errs == _libep.ERROR_NAMES
    dts = {m[0]: int(m[1]) for m in re.findall(r"EP_DTYPE_(\w+) = (\d+)", src)}
    assert {k.lower(): v for k, v in dts.items()} == _libep.DTYPE_CODES
    assert int(re.search(r"#define EP_ABI_VERSION (\d+)u", src).group(1)) == ep.ep_abi_version()


# ----------------------------------------------------------------------------
# Sharded layers: host-side checks (no GPU needed; nothing is launched)
# ----------------------------------------------------------------------------

def test_sharded_registration_limits(ep):
    lid, size = ep.ep_register_layer_sharded(8, 2, 64, 100, num_ranks=2, rank=1, max_alignment=128)
    # an owner may receive every rank's routes to its 4 experts: 2*100*2 + 4*127
    assert ep.ep_recv_capacity(lid) == 400 + 4 * 127
    bad = [dict(num_ranks=3, rank=0),        # 3 does not divide 8
           dict(num_ranks=2, rank=2),        # rank out of range
           dict(num_ranks=0, rank=0),
           dict(num_ranks=65, rank=0)]
    for kw in bad:
        with pytest.raises(ep.EpError):
            ep.ep_register_layer_sharded(8, 2, 64, 100, **kw)
    with pytest.raises(ep.EpError, match="routes"):
        ep.ep_register_layer_sharded(256, 8, 64, 16385, num_ranks=4, rank=0)  # 131,080 routes
    ep.ep_register_layer_sharded(256, 8, 64, 16384, num_ranks=4, rank=0)      # 131,072 routes


def test_sharded_and_single_calls_do_not_mix(ep):
    import torch
    lid_s, size_s = ep.ep_register_layer_sharded(8, 2, 64, 16, num_ranks=2, rank=0)
    lid_1, size_1 = ep.ep_register_layer(8, 2, 64, 16)
    from combine_ep_prepare_gb300._libep import Handle
    lib = ep.lib()
    mem = ctypes.create_string_buffer(max(size_s, size_1) + 256)
    base = (ctypes.addressof(mem) + 255) // 256 * 256
    counts = ctypes.create_string_buffer(64)
    before = ep.ep_launch_count()
    rc = lib.ep_prepare(Handle(lid_s, base), None, 0, ctypes.addressof(counts), 1, None)
    assert rc == 1 and "sharded" in ep.ep_last_error()
    rc = lib.ep_shard_count(Handle(lid_1, base), None, 0, ctypes.addressof(counts), None)
    assert rc == 1 and "not an expert-major sharded layer" in ep.ep_last_error()
    # null pointer tables are refused before any launch
    rc = lib.ep_shard_combine(Handle(lid_s, base), None, 0, None, None)
    assert rc == 1 and "table" in ep.ep_last_error()
    rc = lib.ep_shard_dispatch(Handle(lid_s, base), 0, None, None, None, None, None)
    assert rc == 1 and "table" in ep.ep_last_error()
    assert ep.ep_launch_count() == before


def test_header_is_plain_c_and_links(ep, tmp_path):
    """include/ep.h compiles as C99 with warnings as errors, every declared
    call links against libep.so, and a C program calls the host-only entry
    points (version, registration, capacity, error message) without a GPU."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    names = header_functions()
    lib = ep.lib()._name
    src = tmp_path / "use_ep.c"
    refs = "\n".join("  fns[%d] = (void (*)(void))%s;" % (i, n) for i, n in enumerate(names))
    src.write_text("""
#include <stdio.h>
#include <string.h>
#include "ep.h"
int main(void) {
  void (*fns[%d])(void);
%s
  for (int i = 0; i < %d; ++i) if (fns[i] == 0) return 2;
  if (ep_abi_version() != EP_ABI_VERSION) return 3;
  ep_layer_config_t c;
  memset(&c, 0, sizeof c);
  c.num_experts = 8; c.top_k = 2; c.hidden = 64; c.max_tokens = 16; c.max_alignment = 4;
  uint64_t id = 0; size_t size = 0; int64_t rows = 0;
  if (ep_register_layer(c, &id, &size) != EP_OK || id == 0 || size == 0) return 4;
  if (ep_recv_capacity(id, &rows) != EP_OK || rows != 16 * 2 + 8 * 3) return 5;
  c.num_experts = 0;
  if (ep_register_layer(c, &id, &size) != EP_ERR_LIMIT || strlen(ep_last_error()) == 0) return 6;
  c.num_experts = 8;
  if (ep_register_layer_sharded(c, 3, 0, &id, &size) != EP_ERR_INVALID_ARG) return 7;
  printf("ok\\n");
  return 0;
}
""" % (len(names), refs, len(names)))
    exe = tmp_path / "use_ep"
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe), lib, "-Wl,-rpath," + os.path.dirname(lib)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0 and out.stdout.strip() == "ok", (out.returncode, out.stdout, out.stderr)


def test_rank_major_registration_and_refusals(ep):
    """Host-only: registration limits and capacity of rank-major layers, and
    calls of the wrong layer kind or with null tables refused before any
    launch."""
    lid, size = ep.ep_register_layer_rank_major(8, 2, 64, 16, num_ranks=4, rank=3)
    assert ep.ep_recv_capacity(lid) == 4 * 16  # a token goes once to each owner
    lid_c, _ = ep.ep_register_layer_rank_major(8, 2, 64, 16, num_ranks=4, rank=0, recv_capacity=20)
    assert ep.ep_recv_capacity(lid_c) == 20
    for bad in (dict(num_ranks=3, rank=0), dict(num_ranks=4, rank=4), dict(num_ranks=0, rank=0),
                dict(num_ranks=65, rank=0)):
        with pytest.raises(ep.EpError):
            ep.ep_register_layer_rank_major(8, 2, 64, 16, **bad)
    with pytest.raises(ep.EpError):  # beyond the routing map's batch
        ep.ep_register_layer_rank_major(8, 2, 64, 1 << 20, num_ranks=4, rank=0)
    lid_s, size_s = ep.ep_register_layer_sharded(8, 2, 64, 16, num_ranks=4, rank=0)
    from combine_ep_prepare_gb300._libep import Handle
    lib = ep.lib()
    mem = ctypes.create_string_buffer(max(size, size_s) + 256)
    base = (ctypes.addressof(mem) + 255) // 256 * 256
    counts = ctypes.create_string_buffer(64)
    before = ep.ep_launch_count()
    rc = lib.ep_shard_count(Handle(lid, base), None, 0, ctypes.addressof(counts), None)
    assert rc == 1 and "not an expert-major sharded layer" in ep.ep_last_error()
    rc = lib.ep_rank_major_count(Handle(lid_s, base), None, 0, ctypes.addressof(counts), None)
    assert rc == 1 and "not a rank-major layer" in ep.ep_last_error()
    rc = lib.ep_prepare(Handle(lid, base), None, 0, ctypes.addressof(counts), 1, None)
    assert rc == 1 and "sharded" in ep.ep_last_error()
    rc = lib.ep_rank_major_combine(Handle(lid, base), None, 0, None, None)
    assert rc == 1 and "table" in ep.ep_last_error()
    rc = lib.ep_rank_major_dispatch(Handle(lid, base), None, 0, None, None, None, None, None, None)
    assert rc == 1 and "table" in ep.ep_last_error()
    rc = lib.ep_rank_major_prepare(Handle(lid, base), None, 0, None, ctypes.addressof(counts), None)
    assert rc == 1 and "all_counts" in ep.ep_last_error()
    rc = lib.ep_expert_offsets(Handle(lid, base), ctypes.addressof(counts), None)
    assert rc == 1 and "rank-major" in ep.ep_last_error()
    assert ep.ep_launch_count() == before
