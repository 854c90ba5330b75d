"""The CPU oracle against brute force, library routines, invariants and the
values printed on the source pages (no GPU needed)."""
import json
import math
import os

import pytest

import oracle.moe_oracle as o
import workloads
from tests import _pins


@pytest.mark.parametrize("check", _pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(o)


def test_cost_model_counters_match_printed_values():
    """The benchmark's FLOP and byte counters reproduce the Ling-2.6-1T cost
    model worked example (section 1 of the Ling-2.6-1T TPU page)."""
    g = json.load(open(os.path.join(_pins.GOLDEN, "ling_cost_model.json")))
    w, p = g["workload"], g["printed"]
    rows = w["tokens"] * w["top_k"] // w["ep"]
    assert rows == p["routed_rows_per_device"]
    assert rows // w["local_experts"] == p["rows_per_local_expert"]
    D, I = w["D"], w["I"]
    ffn1 = workloads.ffn_gate_up_flops(rows, D, I) / 1e9
    ffn2 = workloads.ffn_down_flops(rows, D, I) / 1e9
    shared = workloads.ffn_flops(rows, D, I) / 1e9
    assert round(ffn1, 1) == p["ffn1_gflop"]
    assert round(ffn2, 1) == p["ffn2_gflop"]
    assert round(ffn1 + ffn2, 1) == p["routed_gflop"]
    assert round(shared, 1) == p["shared_gflop"]
    assert round(ffn1 + ffn2 + shared, 1) == p["total_gflop"]
    assert round((ffn1 + ffn2 + shared) / p["fp8_peak_tflops_per_device"], 2) == p["compute_bound_ms"]
    assert rows * D == p["scatter_elements"]
    assert round(rows * D * 2 / 1e6, 1) == p["scatter_bf16_mb"]
    assert math.floor(rows * D / 1e6 * 10) / 10 == p["scatter_fp8_mb"]
    per_expert = workloads.expert_weight_bytes(D, I, "fp8_e4m3", scales=False) / 1e6
    assert round(per_expert, 1) == p["expert_fp8_mb"]
    assert int(per_expert * w["local_experts"]) == p["local_experts_fp8_mb"]
    local = per_expert * w["local_experts"]
    assert round(local / 1e6 / p["hbm_tbps_per_device"] * 1e3, 2) == p["weight_read_bound_ms"]
    tiles = math.ceil(p["rows_per_local_expert"] / w["bts"])
    assert tiles == p["token_tiles"]
    assert round(tiles * local / 1e6 / p["hbm_tbps_per_device"] * 1e3, 2) == p["weight_read_bound_bts_ms"]
