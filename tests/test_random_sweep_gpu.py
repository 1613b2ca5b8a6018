"""Randomised GPU parity sweep: many seeded configurations of the whole step
(prepare, dispatch, combine, combine_bwd, dispatch_bwd), each compared bit for
bit with the CPU oracle, rows beyond the used extent checked untouched.

The configurations are drawn from one seeded generator over the space the
layer registration allows: expert counts from 1 to 1024 (both prepare paths,
every cluster width), top-k from 1 to 32 with repeats or distinct experts,
ragged hidden sizes (16- and 32-byte row vectors), alignments from 1 to 200,
masked and invalid routes, zero tokens, and the three payload types.  Sizes
are kept small enough for the oracle to finish in well under a second each.
"""
import numpy as np
import pytest
import torch

from combine_ep_prepare_gb300 import workloads as wl
from ep_harness import GpuLayer, assert_step_equal, custom_inputs, gpu_step, oracle_step

pytestmark = pytest.mark.gpu


def _configs(n=160, seed=20261202):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.choice([1, 2, 3, 7, 8, 16, 37, 64, 128, 256, 1000, 1024]))
        K = int(rng.choice([1, 2, 3, 4, 6, 8, 16, 32]))
        T = int(rng.choice([0, 1, 2, 31, 100, 333, 777, 2049, 5000, 9001]))
        if T * K > 40000:
            T = 40000 // K
        H = 8 * int(rng.integers(1, 72))
        A = int(rng.choice([1, 2, 3, 16, 128, 200]))
        p_mask = float(rng.choice([0.0, 0.0, 0.1, 0.5, 1.0]))
        p_bad = float(rng.choice([0.0, 0.0, 0.0, 0.02]))
        distinct = K <= E and bool(rng.random() < 0.5)
        dtype = str(rng.choice(["bf16", "bf16", "fp16", "fp32"]))
        out.append((i, T, K, E, H, A, p_mask, p_bad, distinct, dtype))
    return out


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_ep_prepare_gb300 as ep
    return ep


@pytest.mark.parametrize("cfg", _configs(), ids=lambda c: "c%d_T%d_K%d_E%d_H%d_A%d_%s" % (c[0], c[1], c[2], c[3], c[4], c[5], c[9]))
def test_random_step_parity(ep, oracle_mod, cfg):
    i, T, K, E, H, A, p_mask, p_bad, distinct, dtype = cfg
    idx, wts = wl.random_routing(T, K, E, seed=7000 + i, p_mask=p_mask, p_bad=p_bad, distinct=distinct)
    inp = custom_inputs(idx, wts, E, H, A, oracle_mod, seed=70000 + 10 * i, dtype=dtype)
    layer = GpuLayer(ep, E, K, H, max(T, 1), A, dtype=dtype)
    g = gpu_step(ep, layer, inp)
    o = oracle_step(inp, oracle_mod, layer.R)
    assert_step_equal(g, o, layer.R)


def _weighted_configs(n=64, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        E = int(rng.choice([1, 3, 8, 16, 64, 128, 256, 1024]))
        K = int(rng.choice([1, 2, 3, 4, 8, 16, 32]))
        T = int(rng.choice([1, 2, 31, 333, 2049, 5000]))
        if T * K > 40000:
            T = 40000 // K
        H = 8 * int(rng.integers(1, 72))
        A = int(rng.choice([1, 2, 3, 16, 128]))
        p_mask = float(rng.choice([0.0, 0.1, 0.5, 1.0]))
        p_bad = float(rng.choice([0.0, 0.0, 0.02]))
        out.append((i, T, K, E, H, A, p_mask, p_bad))
    return out


@pytest.mark.parametrize("cfg", _weighted_configs(), ids=lambda c: "w%d_T%d_K%d_E%d_H%d_A%d" % c[:6])
def test_random_weighted_parity(ep, oracle_mod, cfg):
    """The weighted combine (bit for bit) and its backward (token gradient bit
    for bit, weight gradient within its float32 summation bound)."""
    from test_weighted_gpu import run_weighted
    i, T, K, E, H, A, p_mask, p_bad = cfg
    idx, _ = wl.random_routing(T, K, E, seed=9000 + i, p_mask=p_mask, p_bad=p_bad)
    run_weighted(ep, oracle_mod, idx, E, H, A, seed=90000 + 10 * i)
