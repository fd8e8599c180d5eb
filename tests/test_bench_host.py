"""Host-side arithmetic of bench.py (no GPU): algorithmic HBM bytes and the GB/s figures."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def test_hbm_bytes_of_the_headline_workload():
    import bench
    from attention_relative_position_gb300 import workloads as wl
    w = wl.WORKLOADS[1]  # 8 x 1024 tokens, 8 heads, d 64, table [32, 8]
    b = bench.hbm_bytes(w)
    elems = 8 * 1024 * 8 * 64
    assert b["fwd"] == 4 * elems * 2 + 8192 * 8 * 4 + 32 * 8 * 4  # Q K V in, O out, lse, table
    assert b["bwd_pre"] == 2 * elems * 2 + 8192 * 8 * 4 + elems * 4 + 32 * 8 * 4
    assert b["bwd_fin"] == elems * 4 + elems * 2


def test_hbm_bytes_without_table():
    import bench
    from attention_relative_position_gb300 import workloads as wl
    w = wl.WORKLOADS[3]  # ALiBi only: no table traffic
    elems = w.total_tokens * w.num_heads * w.head_dim
    assert bench.hbm_bytes(w)["bwd_fin"] == 6 * elems
    assert bench.hbm_bytes(w)["fwd"] == 8 * elems + 4 * w.total_tokens * w.num_heads


def test_hbm_figures_units():
    import bench
    from attention_relative_position_gb300 import workloads as wl
    w = wl.WORKLOADS[1]
    b = bench.hbm_bytes(w)
    per = {"fwd": [0.05, 0.05], "bwd_pre": [0.01], "bwd_fin": [0.02, 0.0200]}
    r = bench.hbm_figures(w, per, 5000.0)
    assert abs(r["bwd_pre_gbs"] - round(b["bwd_pre"] / 0.01 / 1e6, 1)) < 1e-9  # bytes/ms -> GB/s
    assert r["bwd_fin_us"] == 20.0
    assert abs(r["fwd_gbs_frac"] - r["fwd_gbs"] / 5000.0) < 1e-4
    assert r["peak_gbs"] == 5000.0


def test_guarded_side_figure_records_errors():
    import bench
    assert bench._guarded(lambda a: a + 1, 1) == 2
    r = bench._guarded(lambda: 1 / 0)
    assert r["error"].startswith("ZeroDivisionError")
