"""Host-side logic of bench.py, without a GPU: the ncu traffic figure is reported only while
the kernel sources still match the capture, and the oracle check of sampled rows rejects
outputs past the parity bars."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_is_null_unless_the_sources_match(tmp_path, monkeypatch):
    md = "fake_summary.md"
    files = ["common.cuh", "kernels.h"]
    monkeypatch.setattr(bench, "TRAFFIC_SOURCES", {"k": (md, files)})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    os.makedirs(tmp_path / "profiles")
    # no summary
    assert bench.committed_traffic("k")[0] is None
    # a summary for the current sources
    good = bench.sources_sha256(files)
    (tmp_path / "profiles" / md).write_text(
        f"...\nbench-traffic: bytes_per_launch=12345 sources_sha256={good}\n")
    assert bench.committed_traffic("k")[0] == 12345
    # a summary taken on other sources is stale
    (tmp_path / "profiles" / md).write_text(
        f"bench-traffic: bytes_per_launch=12345 sources_sha256={'0' * 64}\n")
    n, why = bench.committed_traffic("k")
    assert n is None and "changed" in why


def test_row_check_accepts_within_bars_and_rejects_past_them():
    rng = np.random.default_rng(0)
    ref = rng.standard_normal((64, 128))
    lse = rng.standard_normal(64)
    rec = bench._check_rows("ok", ref + 1e-3, lse + 1e-4, ref, lse, "bf16")
    assert rec["ok"] and rec["rows"] == 64
    bad = ref.copy()
    bad[3, 7] += 0.05                       # one element past the 2e-2 max bar
    with pytest.raises(RuntimeError):
        bench._check_rows("bad", bad, lse, ref, lse, "bf16")
    with pytest.raises(RuntimeError):      # fp32 bar is 1e-4
        bench._check_rows("fp32", ref + 2e-4, lse, ref, lse, "fp32")
    with pytest.raises(RuntimeError):      # LSE bar is 1e-3
        bench._check_rows("lse", ref, lse + 2e-3, ref, lse, "bf16")
