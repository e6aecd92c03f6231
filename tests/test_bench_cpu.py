"""Host logic of bench.py that needs no GPU: the oracle arm's JSON line (its
steps are bounded samples, extrapolated, and say so in keys; its config is
the GPU arm's), and the clock-normalised kernel figures."""
import argparse

import bench
from streaming_avatar_video_gb300 import inputs as I


def test_reference_arm_labels_extrapolation():
    w = I.WORKLOADS["tiny"]
    args = argparse.Namespace(steps=3, warmup=3)
    res = bench.run_reference(args, w, 1, 0)
    assert res["impl"] == "reference" and res["extrapolated"] is True
    assert res["samples"] == 3 and res["steps"] == 3 and res["warmup"] == 3
    assert res["ms_per_sample"] > 0 and res["ms_per_step"] > 0
    assert res["config"] == bench.config_of(w, 1)
    assert res["cpu_baseline"]["kind"] == "oracle" and res["cpu_baseline"]["extrapolated"] is True
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["e2e"]["value"] == res["value"]
    assert bench.run_reference(args, w, 2, 1) is None  # only rank 0 runs it


def test_clock_normalised_figures():
    # 1 ms of a kernel doing 152 SMs x 1000 MMAs of 128x128x16 at 2000 MHz: 2e6 clocks / 1000 MMAs
    mma = 2.0 * 128 * 128 * 16
    f = bench.clock_normalised(152 * 1000 * mma, 1.0, 152 * 500 * mma, 1.0, 2000.0, 152)
    assert f["chunk_attention"]["clocks_per_mma_128x128x16"] == 2000.0
    assert f["out_proj_euler"]["clocks_per_mma_128x128x16"] == 4000.0
    assert abs(f["chunk_attention"]["flop_per_clk_per_sm"] - mma / 2000.0) < 0.1
    assert bench.clock_normalised(1.0, 1.0, 1.0, 1.0, None, 152) is None
