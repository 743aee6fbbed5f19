"""Host-side pieces of bench.py (no GPU): the nominal-rate fractions added
next to the measured ones, the row split of the all-cores oracle timing, and
the host CPU description."""
import os

import bench


def test_nominal_fractions_nested():
    d = {"a": {"M1": {"us": 1.0, "GBps": 4000.0, "frac_of_measured_hbm": 0.6}},
         "gemm": {"TFLOPS": 1125.0, "note": "x"}, "s": "text"}
    bench.add_nominal_fractions(d, bf16_sustained=1500.0)
    assert d["a"]["M1"]["frac_of_nominal_8000"] == 0.5
    assert d["gemm"]["frac_of_nominal_bf16"] == 0.5
    assert d["gemm"]["frac_of_measured_bf16_sustained"] == 0.75
    assert "frac_of_nominal_8000" not in d["gemm"] and d["s"] == "text"


def test_split_rows_partitions():
    for n, parts in ((32768, 16), (10, 3), (3, 8), (1, 1)):
        r = bench.split_rows(n, parts)
        assert all(nn > 0 for _, nn in r) and len(r) <= parts
        assert [n0 for n0, _ in r] == [0] + [n0 + nn for n0, nn in r[:-1]]
        assert r[-1][0] + r[-1][1] == n


def test_host_cpu_description():
    h = bench.host_cpu()
    assert h["nproc"] == os.cpu_count()
    assert h["model"] is None or isinstance(h["model"], str)
