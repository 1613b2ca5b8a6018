"""Randomised GPU parity sweep of the sharded layouts: seeded configurations
of N ranks emulated on one GPU (as in test_shard_gpu.py and
test_rank_major_gpu.py), each rank's whole step compared bit for bit with the
sharded and the rank-major oracle.

The configurations cover 1 to 16 ranks, experts per rank from 1 to 32, top-k
from 1 to 32 (repeats allowed), ragged hidden sizes, alignments from 1 to 128
(expert-major layers), ranks without tokens, masked and invalid routes, and
the three payload types.
"""
import numpy as np
import pytest
import torch

import test_rank_major_gpu as rm
import test_shard_gpu as sh

pytestmark = pytest.mark.gpu


def _configs(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        N = int(rng.choice([1, 2, 3, 4, 5, 8, 16]))
        E = N * int(rng.choice([1, 2, 3, 8, 32]))
        K = int(rng.choice([1, 2, 3, 4, 6, 8, 16, 32]))
        tpr = [int(rng.choice([0, 1, 7, 33, 100, 257])) for _ in range(N)]
        while max(tpr) * K > 16384:
            tpr = [t // 2 for t in tpr]
        H = 8 * int(rng.integers(1, 40))
        A = int(rng.choice([1, 2, 5, 16, 128]))
        p_mask = float(rng.choice([0.0, 0.1, 0.5]))
        p_bad = float(rng.choice([0.0, 0.0, 0.02]))
        dtype = str(rng.choice(["bf16", "bf16", "fp16", "fp32"]))
        out.append((i, N, E, K, H, tpr, A, p_mask, p_bad, dtype))
    return out


def _id(c):
    return "c%d_N%d_E%d_K%d_H%d_A%d_%s" % (c[0], c[1], c[2], c[3], c[4], c[6], c[9])


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import combine_ep_prepare_gb300 as ep
    return ep


@pytest.mark.parametrize("cfg", _configs(40, 20261204), ids=_id)
def test_random_expert_major_sharded_step(ep, oracle_mod, cfg):
    i, N, E, K, H, tpr, A, p_mask, p_bad, dtype = cfg
    routing = sh._routing(N, tpr, K, E, 300 + i, p_mask=p_mask, p_bad=p_bad)
    ranks = sh.Ranks(ep, N, E, K, H, max(max(tpr), 1), 128, dtype=dtype)
    sr = oracle_mod.shard_prepare([x.numpy() for x, _ in routing], E, A, N, ranks.R)
    pay = sh._payloads(sr, routing, H, dtype, 3000 + 10 * i, oracle_mod)
    g = ranks.step(routing, A, pay)
    sh._check(g, sr, routing, pay, oracle_mod, dtype, ranks.R)


@pytest.mark.parametrize("cfg", _configs(40, 20261205), ids=_id)
def test_random_rank_major_step(ep, oracle_mod, cfg):
    i, N, E, K, H, tpr, A, p_mask, p_bad, dtype = cfg
    routing = rm._routing(tpr, K, E, 500 + i, p_mask=p_mask, p_bad=p_bad)
    ranks = rm.Ranks(ep, N, E, K, H, max(max(tpr), 1), dtype=dtype)
    rr = oracle_mod.rm_prepare([x.numpy() for x, _ in routing], E, N, ranks.R)
    pay = rm._payloads(rr, routing, H, K, dtype, 5000 + 10 * i)
    g = ranks.step(routing, pay)
    rm._check(g, rr, routing, pay, oracle_mod, dtype)
