"""The seeded input recipes have the structure the workloads are described
with: K distinct experts per token (uniform, Zipf and group-limited
routing), group-limited routing inside the top groups, masking of the experts
another rank owns, weights that sum to one, and the same draws on every run."""
import numpy as np
import pytest
import torch

from combine_ep_prepare_gb300 import workloads as wl


def _routing(name, T=512):
    w = wl.WORKLOADS[name]
    idx, wts = wl.routing(w, T=min(T, w.T))
    return w, idx.numpy(), wts.numpy()


@pytest.mark.parametrize("name", ["tiny", "mixtral", "qwen3", "dsv3"])
def test_distinct_experts_and_normalised_weights(name):
    w, idx, wts = _routing(name)
    assert idx.shape[1] == w.K and idx.dtype == np.int64
    assert np.all((idx >= 0) & (idx < w.E))
    assert all(len(set(row)) == w.K for row in idx.tolist())
    assert np.allclose(wts.sum(1), 1.0, atol=1e-5) and np.all(wts > 0)


def test_group_limited_routing():
    w, idx, _ = _routing("dsv3")
    per_group = w.E // w.n_groups
    groups = idx // per_group
    assert all(len(set(row)) <= w.topk_groups for row in groups.tolist())


def test_zipf_popularity_is_skewed():
    w = wl.WORKLOADS["qwen3"]
    idx, _ = wl.routing(w)
    counts = np.bincount(idx.numpy().ravel(), minlength=w.E)
    top = np.sort(counts)[::-1]
    assert top[0] > 4 * np.median(counts)  # a few experts take most routes


def test_decode_masks_the_other_ranks_experts():
    w, idx, _ = _routing("decode")
    assert np.all((idx == -1) | ((idx >= 0) & (idx < w.local_experts)))
    assert 0.2 < (idx == -1).mean() < 0.8


def test_same_draws_every_run():
    w = wl.WORKLOADS["qwen3"]
    a, b = wl.routing(w, T=64), wl.routing(w, T=64)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(wl.tokens(w, T=8).view(torch.int16), wl.tokens(w, T=8).view(torch.int16))
    x = wl.payload_normal(4, 8, 2001, "fp16")
    assert x.dtype == torch.float16 and torch.equal(x, wl.payload_normal(4, 8, 2001, "fp16"))
