"""The C ABI driven from plain C on the GPU: tests/c/ep_c_step.c runs a whole
step (prepare, dispatch, combine, combine_bwd, dispatch_bwd, read-back) on
cudaMalloc buffers through libep.so alone, with no Python or PyTorch in the
process; its outputs are compared bit for bit with the oracle, and the rows at
or beyond P with the sentinel they started with."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from combine_ep_prepare_gb300 import workloads as wl
from ep_harness import SENTINEL, bits, custom_inputs, oracle_step

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def c_step(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    libdir = os.path.join(ROOT, "combine_ep_prepare_gb300")
    if not os.path.exists(os.path.join(libdir, "libep.so")):
        pytest.fail("libep.so is not built")
    exe = str(tmp_path_factory.mktemp("c_api") / "ep_c_step")
    cmd = ["gcc", "-std=c99", "-O1", "-Wall", "-Wextra", "-Werror", "-o", exe,
           os.path.join(ROOT, "tests", "c", "ep_c_step.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", libdir, "-lep", "-Wl,-rpath," + libdir,
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(CUDA, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


CASES = [
    # T, K, E, H, A, p_mask, p_bad, seed
    (64, 2, 8, 128, 16, 0.0, 0.0, 1),        # the tiny workload's shape
    (300, 4, 37, 200, 5, 0.2, 0.02, 2),      # ragged rows, masked and invalid routes, A not a power of 2
    (0, 3, 5, 64, 4, 0.0, 0.0, 3),           # no tokens
]


@pytest.mark.parametrize("T,K,E,H,A,p_mask,p_bad,seed", CASES)
def test_c_step_matches_oracle(c_step, oracle_mod, tmp_path, T, K, E, H, A, p_mask, p_bad, seed):
    idx, wts = wl.random_routing(T, K, E, seed=600 + seed, p_mask=p_mask, p_bad=p_bad)
    inp = custom_inputs(idx, wts, E, H, A, oracle_mod, seed=6000 + 10 * seed)
    d = str(tmp_path)
    files = {"idx.bin": idx.numpy().astype(np.int64), "w.bin": wts.numpy().astype(np.float32),
             "tok.bin": bits(inp.tokens), "eo.bin": bits(inp.expert_out), "gres.bin": bits(inp.grad_result),
             "grecv.bin": bits(inp.grad_recv), "grecv_w.bin": inp.grad_recv_w.numpy().astype(np.float32)}
    for name, a in files.items():
        np.ascontiguousarray(a).tofile(os.path.join(d, name))
    r = subprocess.run([c_step, str(E), str(K), str(H), str(A), str(T), d], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    R, P, npad, status = (int(x) for x in r.stdout.split())
    o = oracle_step(inp, oracle_mod, R)
    rd = lambda name, dt: np.fromfile(os.path.join(d, name), dtype=dt)  # noqa: E731
    assert status == o["status"] and P == o["P"]
    assert npad == int((o["rt"].inv < 0).sum())
    assert np.array_equal(rd("out_counts.bin", np.int32), o["counts"])
    assert np.array_equal(rd("out_offsets.bin", np.int32), o["offsets"])
    assert np.array_equal(rd("out_slots.bin", np.int32).reshape(T, K), o["slot"])
    recv = rd("out_recv.bin", np.uint16).reshape(R, H)
    recv_w = rd("out_recv_w.bin", np.float32)
    gexp = rd("out_gexp.bin", np.uint16).reshape(R, H)
    assert np.array_equal(recv[:P], o["recv_tokens"]) and np.all(recv[P:] == SENTINEL)
    assert np.array_equal(recv_w[:P].view(np.uint32), o["recv_w"].view(np.uint32)) and np.all(recv_w[P:] == -3.0)
    assert np.array_equal(gexp[:P], o["grad_expert_out"]) and np.all(gexp[P:] == SENTINEL)
    assert np.array_equal(rd("out_result.bin", np.uint16).reshape(T, H), o["result"])
    assert np.array_equal(rd("out_gtok.bin", np.uint16).reshape(T, H), o["grad_tokens"])
    assert np.array_equal(rd("out_gtw.bin", np.float32).view(np.uint32),
                          o["grad_topk_weights"].reshape(-1).view(np.uint32))
