"""Host-side pieces of bench.py that build the JSON line (no GPU): the
algorithmic byte counts the rates divide by, and the notes the line carries."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_algorithmic_bytes_of_the_cells():
    M, N = 131072, 8192
    mn = M * N
    cast = mn + mn // 32                      # E4M3 codes + one E8M0 byte per 32
    assert bench.cell_bytes("fwd", 1, M, N) == 4 * mn + cast       # gate, up in; one cast out
    assert bench.cell_bytes("fwd", 3, M, N) == 4 * mn + 2 * cast
    assert bench.cell_bytes("bwd", 2, M, N) == 6 * mn + 2 * cast   # dh, gate, up in; dgate, dup out
    assert bench.cell_bytes("bwd", 3, M, N) == 6 * mn + 4 * cast
    assert bench.step_bytes(M, N) == sum(bench.cell_bytes(k, m, M, N) for k, m in bench.CELLS)


def test_configs_note_formats():
    note = bench.configs_note(20)
    assert "median of 20" in note and "5 % of" in note


def test_traffic_is_none_for_other_kernel_sources():
    t = bench.TRAFFIC.get("bwd_both")
    assert t is not None
    assert bench.traffic_for("bwd_both") == (t[0] if t[1] == bench.kernel_source_hash() else None)
    assert bench.traffic_for("no such cell") is None
