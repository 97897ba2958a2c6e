"""bench.py's link between the committed ncu summary and the current kernel
sources: the recorded DRAM traffic is reported only while the one-read
row-statistics kernel's sources (rows_topp.cu and the kernel headers it
includes) are those the capture was taken on."""

import os
import shutil

import bench


def _tree(tmp_path):
    root = tmp_path / "repo"
    src = os.path.join(bench.ROOT, "speculative_decoding_verification_60_gb300", "csrc")
    shutil.copytree(src, root / "speculative_decoding_verification_60_gb300" / "csrc")
    shutil.copytree(os.path.join(bench.ROOT, "profiles"), root / "profiles")
    return root


def test_hash_follows_the_row_statistics_sources_only(tmp_path, monkeypatch):
    root = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    csrc = root / "speculative_decoding_verification_60_gb300" / "csrc"
    h0 = bench.source_sha()
    # a unit the kernel does not include leaves the hash alone
    (csrc / "compact.cu").write_text((csrc / "compact.cu").read_text() + "\n// edit\n")
    (csrc / "linear.cu").write_text((csrc / "linear.cu").read_text() + "\n// edit\n")
    (csrc / "unrelated.cu").write_text("// another unit\n")
    assert bench.source_sha() == h0
    # a header the kernel includes (transitively) changes it
    (csrc / "common.cuh").write_text((csrc / "common.cuh").read_text() + "\n// edit\n")
    assert bench.source_sha() != h0


def test_recorded_traffic_needs_matching_sources(tmp_path, monkeypatch):
    root = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    prof = root / "profiles" / "summary.txt"
    prof.write_text(f"- source_sha: `{bench.source_sha()}` (a comment)\n"
                    "- traffic_bytes_per_launch: `123456789` (scaled)\n")
    monkeypatch.setattr(bench, "PROFILE", str(prof))
    assert bench.recorded_traffic() == 123456789.0
    rs = root / "speculative_decoding_verification_60_gb300" / "csrc" / "rowstats.cuh"
    rs.write_text(rs.read_text() + "\n// edit\n")
    assert bench.recorded_traffic() is None
