"""The benchmark's roofline traffic comes from the ncu record under profiles/
only for the exact kernel sources the record was captured on: a record keyed
to another source hash (or no record) gives null, never a stale number."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _with_record(monkeypatch, tmp_path, lines):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "ncu_traffic.txt").write_text("".join(l + "\n" for l in lines))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))


def test_traffic_only_for_the_captured_sources(monkeypatch, tmp_path):
    h = bench.kernel_source_hash()  # hash of the real kernel sources (read before ROOT moves)
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: h)
    _with_record(monkeypatch, tmp_path, ["# comment", f"chain_f32_B64 {h} 353419520", "other_tag deadbeef 1"])
    assert bench.ncu_traffic("chain_f32_B64") == 353419520.0
    assert bench.ncu_traffic("other_tag") is None        # captured on other sources
    assert bench.ncu_traffic("missing_tag") is None


def test_traffic_null_without_a_matching_record(monkeypatch, tmp_path):
    _with_record(monkeypatch, tmp_path, ["chain_f32_B64 0000000000000000 353419520"])
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "1111111111111111")
    assert bench.ncu_traffic("chain_f32_B64") is None
    monkeypatch.setattr(bench, "ROOT", str(tmp_path / "nowhere"))
    assert bench.ncu_traffic("chain_f32_B64") is None


def test_source_hash_follows_the_kernel_sources(monkeypatch, tmp_path):
    csrc = tmp_path / "speculative_decoding_token_spv_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cu").write_text("x")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h1 = bench.kernel_source_hash()
    (csrc / "a.cu").write_text("y")
    assert bench.kernel_source_hash() != h1
