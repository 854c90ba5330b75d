"""Heaviest-first tile order (MOE_OPT_TILE_ORDER = 1): the grouped GEMMs run
the experts by descending row count.  Every output tile is still computed by
one CTA with the same K order, so the layer's output is bit-identical to the
expert-order schedule's, on every tile kernel and for skewed routings."""
import dataclasses

import pytest
import torch

import mixture_experts_layer_gating_gb300 as moe
import workloads
from tests.test_gpu_parity import LAYER_CASES, check_layer, run_layer
from tests._lib import ensure_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return ensure_library()


@pytest.fixture(params=["default", "cta1", "pair", "decode16"])
def kernels(request):
    pair = moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, {"cta1": 0, "pair": 1}.get(request.param, 3))
    dec = moe.moe_set_option(moe.MOE_OPT_DECODE_KERNEL, {"decode16": 3}.get(request.param, 1))
    yield request.param
    moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, pair)
    moe.moe_set_option(moe.MOE_OPT_DECODE_KERNEL, dec)


SKEWED = {
    "qwen3_zipf_T384": LAYER_CASES["qwen3_zipf_T384"],
    "qwen35_zipf_T300": dataclasses.replace(workloads.CONFIGS["qwen35_prefill"].with_tokens(300),
                                            name="qwen35_zipf_T300"),
    "fp8_small_T300": LAYER_CASES["fp8_small_T300"],
    "gemma4_T256": LAYER_CASES["gemma4_T256"],
}


@pytest.mark.parametrize("case", sorted(SKEWED))
def test_heaviest_first_bit_identical(case, kernels):
    shape = SKEWED[case]
    layout = "nk" if shape.w_dtype == "fp8_e4m3" else "kn"
    inp = workloads.make_inputs(shape, seed=31, device="cuda")
    base = run_layer(shape, inp, layout)["out"].clone()
    old = moe.moe_set_option(moe.MOE_OPT_TILE_ORDER, 1)
    try:
        got = run_layer(shape, inp, layout)["out"]
    finally:
        moe.moe_set_option(moe.MOE_OPT_TILE_ORDER, old)
    assert torch.equal(got, base)


def test_heaviest_first_parity_qwen35_zipf():
    old = moe.moe_set_option(moe.MOE_OPT_TILE_ORDER, 1)
    try:
        check_layer(SKEWED["qwen35_zipf_T300"])
    finally:
        moe.moe_set_option(moe.MOE_OPT_TILE_ORDER, old)
