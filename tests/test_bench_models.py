"""Host-side models behind bench.py's roofline and traffic figures, checked
against independent counts: the expected fraction of 32-byte sectors and
128-byte lines of a row that the kept dims touch (the fused mask ops' byte
model) against the oracle's own index sets, and the lookup that reports ncu
traffic only while the profiled kernel's sources are unchanged."""
import hashlib

import numpy as np
import pytest

import bench
import oracle


@pytest.mark.parametrize("H,K", [(256, 13), (2048, 102), (2048, 205), (4096, 205)])
@pytest.mark.parametrize("elems", [16, 64])
def test_coverage_model_matches_the_index_sets(H, K, elems):
    rows = 4096
    idx = oracle.mask_indices(rows, H, K, 3, 7)
    touched = np.zeros((rows, H // elems), dtype=bool)
    np.put_along_axis(touched, (idx // elems).astype(np.int64), True, axis=1)
    expected = bench.sector_coverage(H, K, elems)
    # the blocks a row touches are negatively correlated (K dims without
    # replacement), so the binomial standard error bounds that of the mean
    se = np.sqrt(expected * (1.0 - expected) / touched.size)
    assert abs(touched.mean() - expected) <= 6.0 * se


def test_coverage_model_limits():
    assert bench.sector_coverage(2048, 0) == 0.0
    assert bench.sector_coverage(2048, 2048) == 1.0
    assert bench.sector_coverage(2048, 102, elems=1) == pytest.approx(102 / 2048, rel=1e-15)
    # one block of H elements always holds a kept dim once K >= 1
    assert bench.sector_coverage(64, 1, elems=64) == pytest.approx(1.0, rel=1e-15)


def test_traffic_is_reported_only_for_unchanged_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "spectral_corrected_optimizer_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "a.cu").write_bytes(b"first kernel")
    (csrc / "b.cuh").write_bytes(b"shared header")
    sha = hashlib.sha256(b"first kernel" + b"shared header").hexdigest()[:16]
    (tmp_path / "profiles" / "p.md").write_text(
        "notes\nmachine-readable: k1 traffic_bytes_per_launch=12.5e6 code_sha256_16=%s\n"
        "machine-readable: k2 traffic_bytes_per_launch=3e6 code_sha256_16=%s\n" % (sha, sha))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sources = ("a.cu", "b.cuh")
    assert bench.profiled_traffic("p.md", sources, key="k1") == 12.5e6
    assert bench.profiled_traffic("p.md", sources, key="k2") == 3e6
    assert bench.profiled_traffic("p.md", sources, key="k3") is None
    assert bench.profiled_traffic("missing.md", sources, key="k1") is None
    # a comment or blank-space edit keeps the figure, a code edit drops it
    (csrc / "b.cuh").write_bytes(b"shared  // a note\n/* more */ header")
    assert bench.profiled_traffic("p.md", sources, key="k1") == 12.5e6
    (csrc / "b.cuh").write_bytes(b"shared header, edited")
    assert bench.profiled_traffic("p.md", sources, key="k1") is None


def test_strip_comments_keeps_literals():
    src = 'a = "x // y /* z */"; // line\nb = \'/\'; /* block\n */ c = "\\"//"; // end'
    assert bench.strip_comments(src) == 'a = "x // y /* z */"; \nb = \'/\';   c = "\\"//"; '


@pytest.mark.parametrize("W,K", [(3, 20), (5, 20), (3, 40), (25, 20)])
def test_refresh_schedule_of_the_timed_region(W, K):
    """Warm-up steps refresh in one call every REFRESH_EVERY steps; the timed
    steps begin a refresh with their first step and every REFRESH_EVERY steps
    after, and end each one REFRESH_USE_AFTER steps after its begin, so a timed
    region of K = multiple of REFRESH_EVERY steps holds whole refreshes only."""
    class L:
        use_after = bench.REFRESH_USE_AFTER
    what = [bench.Layer.schedule(L, i, W) for i in range(W + K)]
    L.use_after = 0
    serial = [bench.Layer.schedule(L, i, W) for i in range(W + K)]
    assert [i for i, x in enumerate(serial) if x] == [i for i in range(W) if i % bench.REFRESH_EVERY == 0] + \
        list(range(W, W + K, bench.REFRESH_EVERY))
    assert set(serial) <= {None, "refresh"}
    assert what[0] == "refresh"
    assert [i for i in range(W) if what[i]] == [i for i in range(W) if i % bench.REFRESH_EVERY == 0]
    begins = [i for i in range(W, W + K) if what[i] == "begin"]
    ends = [i for i in range(W, W + K) if what[i] == "end"]
    assert begins == list(range(W, W + K, bench.REFRESH_EVERY))
    assert ends == [b + bench.REFRESH_USE_AFTER for b in begins]
    assert "refresh" not in what[W:]
    # the anchors alternate, continuing after the warm-up's
    idx = [bench.Layer.anchor_index(i, W) for i in begins]
    assert idx == list(range(1, len(begins) + 1))
