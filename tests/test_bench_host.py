"""Host-side logic of the benchmark (CPU only): the byte counts its roofline
uses, the source files behind each phase, and the lookup of DRAM traffic in
the committed ncu summary (a row counts only for the source it was taken on)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from combine_ep_layout_03_gb300 import synth  # noqa: E402


def test_algorithmic_bytes_of_the_default_workload():
    w = synth.WORKLOADS[5]
    rows, V = 3790528, 3774664          # from the layout of the seeded routing
    b = bench.algorithmic_bytes(w, 0, rows, V)
    N, H, K, S = w.N, w.H, w.K, w.num_shared
    assert b["dispatch"] == N * H * 2 + N * K * 4 + rows * H * 2
    assert b["combine"] == V * H * 2 + N * K * 8 + S * N * H * 2 + N * H * 2


def test_rms_norm_epilogue_counts_each_output_once():
    w = synth.WORKLOADS[2]
    rows = V = w.N * w.K
    plain = bench.algorithmic_bytes(w, 0, rows, V)["combine"]
    norm = bench.algorithmic_bytes(w, 0, rows, V, fmt="norm")["combine"]
    # residual in and x out (y is the combine's own output), gamma, rstd
    assert norm - plain == 2 * w.N * w.H * 2 + w.H * 2 + w.N * 4


def test_phase_files():
    assert bench.phase_files("dispatch", "5")[0] == "dispatch.cu"
    assert bench.phase_files("dispatch", "3e")[0] == "dispatch_scaled.cu"
    assert bench.phase_files("combine", "5")[0] == "combine.cu"
    assert "split.cu" in bench.phase_files("dispatch", "2a")
    for key in bench.WORKLOAD_KEYS:
        for phase in ("dispatch", "combine"):
            for f in bench.phase_files(phase, key):
                assert os.path.exists(os.path.join(ROOT, "combine_ep_layout_03_gb300", "csrc", f))


def test_traffic_rows_exist_for_every_key_and_follow_the_source(tmp_path, monkeypatch):
    table = open(os.path.join(ROOT, "profiles", "traffic.md")).read()
    for key in bench.WORKLOAD_KEYS:
        for phase in ("dispatch", "combine"):
            assert f"| {phase} | {key} |" in table, (phase, key)
    # a row whose digest is not the current source's does not count
    fake = tmp_path / "profiles"
    fake.mkdir()
    digest = bench.source_digest(bench.phase_files("combine", "5"))
    (fake / "traffic.md").write_text(f"| combine | 5 | 123 | {digest} |\n| dispatch | 5 | 456 | 0000000000000000 |\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_digest", lambda files: digest)
    assert bench.profiled_traffic("combine", "5") == 123
    monkeypatch.setattr(bench, "source_digest", lambda files: "ffffffffffffffff")
    assert bench.profiled_traffic("combine", "5") is None


def test_source_digest_ignores_comments():
    a = bench.code_text("int x = 1; // a comment\n/* block\ncomment */ int y;")
    b = bench.code_text("int x = 1;\n int y;")
    assert a == b
