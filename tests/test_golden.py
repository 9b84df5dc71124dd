"""The pages' printed arithmetic pins the measurement formulas of bench.py.

The pages print no attention input/output example, so these fixtures pin how the
benchmark counts work (FLOPs per (row, key), bytes per key) and the occupancy
arithmetic the split policy restates; see tests/golden/pages_arithmetic.json for
the citation of every number."""
import json
import os

import numpy as np
import pytest

import bench
import workloads as w

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_arithmetic.json")))


def test_flop_count_matches_the_pages_estimate():
    f = G["verify_flops"]
    wl = f["workload"]
    keys = wl["prefix"] + wl["q_len"]
    fmas = bench.flops_per_row_key() / 2 * wl["q_len"] * wl["heads"] * keys
    assert fmas == pytest.approx(f["fmas_about"], rel=0.05)            # "about 10^10 FMAs"
    t_ms = 2 * fmas / (f["fp32_tflops"] * 1e12) * 1e3
    assert t_ms == pytest.approx(f["theoretical_min_ms"], rel=0.05)    # "0.22 ms at 90 TFLOP/s"
    assert f["measured_ms"] / t_ms == pytest.approx(f["gap_about"], rel=0.1)


def test_visible_key_count_of_a_chain_workload():
    # the same workload with all drafts chained: every row sees the prefix plus t+1 drafts
    inp = w.make_verify("g", 1, 9, 2, [100], seed=3, mask_kind="chain")
    expect = sum((100 + t + 1) * 2 for t in range(9))
    assert bench.visible_keys(inp) == expect
    inp.mask = None
    assert bench.visible_keys(inp) == expect


def test_algorithmic_bytes_per_key():
    inp = w.make_verify("g", 2, 9, 8, [50, 70], seed=4)
    a = bench.algorithmic(inp)
    keys = 50 + 70 + 18
    rows = 2 * 9 * 8
    assert a["kv_bytes"] == keys * 576 * 2
    assert a["bytes"] == keys * (1152 + 4) + rows * 1152 + rows * 513 * 4


def test_grid_and_wave_arithmetic():
    g = G["grid_waves"]
    assert 1 * 9 * 64 * 16 == g["blocks_h64_nsplit16"]
    assert 1 * 9 * 8 * 16 == g["blocks_h8_nsplit16"]
    assert 1 * 9 * 8 * 64 == g["blocks_h8_nsplit64"]
    assert g["blocks_h8_nsplit16"] / g["sms"] == pytest.approx(g["waves_h8_nsplit16_about"], abs=0.5)
    assert g["blocks_h8_nsplit64"] / g["sms"] == pytest.approx(g["waves_h8_nsplit64_about"], abs=0.6)


def test_tile_arithmetic():
    k = G["warp_per_key"]
    assert k["dims"] // k["lanes"] == k["per_lane"] and k["dims"] % k["lanes"] == 0
    f = G["fp8_tile"]
    assert f["block_t"] * f["latent"] * 2 == f["tile_bytes"]
    assert 3 * f["tile_bytes"] == pytest.approx(f["stages3_bytes_about"], rel=0.01)
    assert f["acc_rows"] * f["latent"] // f["threads_num_warps8"] == f["acc_f32_per_thread"]


def test_pages_c2_number_used_for_vs_baseline():
    t = G["microbench_table"]
    i = t["prefix"].index(4096)
    assert bench.PAGES_C2_US == min(t["naive_us"][i], t["flash_us"][i])
