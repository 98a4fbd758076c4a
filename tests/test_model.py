"""The byte/flop model the benchmark uses, pinned to figures the pages print."""
import json
import math
import os

import pytest

from exact_io_aware_32_gb300 import model

FIG = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))


def close(value, fig):
    tol = fig.get("rel_tol", 0.0)
    return abs(value - fig["value"]) <= tol * fig["value"]


def test_score_table_n1024():
    f = FIG["score_table_entries_n1024"]
    assert model.standard_score_bytes(f["N"], elem=1) == f["value"]
    assert close(model.standard_score_bytes(1024) / 1e6, FIG["score_table_mb_n1024_16bit"])


def test_ridge_h100():
    f = FIG["h100_ridge_flop_per_byte"]
    assert close(f["peak_tflops"] * 1e12 / (f["hbm_tbs"] * 1e12), f)


def test_standard_way_n4096_d128():
    s = FIG["standard_S_mb_n4096"]
    assert close(model.standard_score_bytes(s["N"]) / 1e6, s)
    r = FIG["standard_S_over_Q_n4096_d128"]
    assert model.standard_score_bytes(r["N"]) / (r["N"] * r["d"] * 2) == r["value"]
    rt = FIG["standard_round_trip_mb_n4096"]
    assert close(model.standard_round_trip_bytes(rt["N"]) / 1e6, rt)
    us = FIG["standard_round_trip_us_n4096_h100"]
    assert close(model.standard_round_trip_bytes(us["N"]) / (us["hbm_tbs"] * 1e12) * 1e6, us)
    mm = FIG["standard_matmul_us_n4096_d128_h100"]
    assert close(model.standard_matmul_flops(mm["N"], mm["d"]) / (mm["peak_tflops"] * 1e12) * 1e6, mm)
    ai = FIG["standard_intensity_d128"]
    assert close(model.standard_intensity(ai["N"], ai["d"]), ai)


def test_nonmatmul_ratio():
    f = FIG["a100_nonmatmul_cost_ratio"]
    assert f["tensor_tflops"] / f["fp32_tflops"] == f["value"]


def test_tiled_counts():
    # forward: 4 N^2 d per head (two products), halved when causal; bwd 2.5x.
    assert model.fwd_flops(1, 1, 1024, 64, False) == 4 * 1024 * 1024 * 64
    assert model.fwd_flops(2, 3, 128, 64, True) == 2 * 3 * 4 * 128 * 128 * 64 / 2
    assert model.bwd_flops(1, 1, 256, 64, False) == 2.5 * 4 * 256 * 256 * 64
    # compulsory bytes: q,k,v,o bf16 + lse fp32
    assert model.fwd_bytes(1, 1, 100, 64) == 4 * 100 * 64 * 2 + 4 * 100
    assert model.bwd_bytes(1, 1, 100, 64) == 8 * 100 * 64 * 2 + 12 * 100
    # Q-outer loop without L2 reuse: K and V are re-read once per block of Q.
    assert model.blocked_q_outer_bytes(1024, 64, 128) == 2 * 1024 * 64 * 2 * (1 + 8)
    # the tiled forward moves far less than the standard way once N >> d
    assert model.fwd_bytes(1, 1, 4096, 128) < model.standard_total_bytes(4096, 128) / 30


def test_roofline_time():
    assert model.roofline_time(2e12, 1e9, 1e15, 1e12) == pytest.approx(2e-3)
    assert model.roofline_time(1e9, 2e12, 1e15, 1e12) == pytest.approx(2.0)
