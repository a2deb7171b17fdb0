"""bench.py's ncu record: the DRAM bytes and L1/shared throughput it reports
beside the roofline come from profiles/dram_traffic.txt only while the digest
recorded there matches the CUDA sources; otherwise they are null."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _write(tmp_path, digest):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        "# comment line\n"
        f"source_digest {digest}\n"
        "B@VCSR 28383488   # gather_kernel<...>, 44.3 us under ncu\n"
        "l1pct:B@VCSR 71.9\n")


def test_record_read_while_digest_matches(tmp_path, monkeypatch):
    _write(tmp_path, "abc123")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_digest", lambda: "abc123")
    assert bench.recorded_traffic("B@VCSR") == 28383488
    assert bench.recorded_profile("l1pct:B@VCSR") == 71.9
    assert bench.recorded_traffic("CSR@B") is None          # not recorded


def test_record_ignored_once_sources_change(tmp_path, monkeypatch):
    _write(tmp_path, "abc123")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_digest", lambda: "def456")
    assert bench.recorded_traffic("B@VCSR") is None
    assert bench.recorded_profile("l1pct:B@VCSR") is None

