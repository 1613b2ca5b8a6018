"""Host-side pieces of bench.py that need no GPU: the kernel-source digest
that ties the committed ncu traffic to the code it was measured on, the
lookup of that traffic, and the algorithmic byte counts of the roofline."""
import os

import pytest

import bench


def _tree(tmp_path, text):
    d = tmp_path / "combine_ep_prepare_gb300" / "csrc"
    d.mkdir(parents=True, exist_ok=True)
    (d / "k.cu").write_text(text)
    return str(tmp_path)


def test_digest_ignores_comments_not_code(tmp_path, monkeypatch):
    code = "__global__ void k(int* a) {\n  a[0] = 1;  // one\n}\n"
    monkeypatch.setattr(bench, "ROOT", _tree(tmp_path / "a", code))
    d0 = bench.source_digest()
    monkeypatch.setattr(bench, "ROOT", _tree(tmp_path / "b", "/* header */\n" + code.replace("// one", "// first")))
    assert bench.source_digest() == d0
    monkeypatch.setattr(bench, "ROOT", _tree(tmp_path / "c", code.replace("a[0] = 1", "a[0] = 2")))
    assert bench.source_digest() != d0


def test_traffic_lookup_follows_the_digest(tmp_path, monkeypatch):
    root = _tree(tmp_path, "__global__ void k() {}\n")
    monkeypatch.setattr(bench, "ROOT", root)
    dg = bench.source_digest()
    os.makedirs(os.path.join(root, "profiles"))
    with open(os.path.join(root, "profiles", "ncu_traffic.txt"), "w") as f:
        f.write("# header\n")
        f.write("dispatch mixtral 1234 %s   # kernel 1234\n" % dg)
        f.write("combine mixtral 99 0000000000000000\n")
    assert bench.committed_traffic("dispatch", "mixtral") == 1234.0
    assert bench.committed_traffic("dispatch", "qwen3") is None
    assert bench.committed_traffic("combine", "mixtral") is None  # other code


def test_traffic_of_a_smaller_batch_scales_by_algorithmic_bytes(tmp_path, monkeypatch):
    root = _tree(tmp_path, "__global__ void k() {}\n")
    monkeypatch.setattr(bench, "ROOT", root)
    dg = bench.source_digest()
    os.makedirs(os.path.join(root, "profiles"))
    with open(os.path.join(root, "profiles", "ncu_traffic.txt"), "w") as f:
        f.write("dispatch dsv3@T4096 600 %s alg=500   # kernel 600\n" % dg)
        f.write("combine dsv3@T4096 400 %s   # no algorithmic bytes: not scalable\n" % dg)
        f.write("combine_bwd dsv3 777 %s\n" % dg)
    assert bench.committed_traffic("dispatch", "dsv3", 2000) == pytest.approx(2400.0)
    assert bench.committed_traffic("dispatch", "dsv3") is None
    assert bench.committed_traffic("combine", "dsv3", 2000) is None
    assert bench.committed_traffic("combine_bwd", "dsv3", 2000) == 777.0  # own row first
    assert bench.committed_traffic("dispatch", "dsv", 2000) is None


@pytest.mark.parametrize("T,H,E,K,V,P,npad", [(4096, 4096, 8, 2, 8192, 8832, 640), (3, 8, 2, 2, 5, 6, 1)])
def test_algorithmic_bytes(T, H, E, K, V, P, npad):
    b = bench.algorithmic_bytes(T, H, E, K, V, P, npad)
    # rows of 2H bytes: dispatch reads each token once and writes every used
    # receive row; combine reads the valid rows and writes the tokens
    assert b["dispatch"] == 2 * H * (T + P) + 8 * T * K + 4 * P + 4 * npad
    assert b["combine"] == 2 * H * (V + T) + 4 * T * K
    assert b["combine_bwd"] == 2 * H * (T + P) + 4 * T * K + 4 * npad
    assert b["dispatch_bwd"] == 2 * H * (V + T) + 8 * T * K + 4 * V
    assert b["prepare"] == 12 * T * K + 12 * E + 4 + 4 * npad
