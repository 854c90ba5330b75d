"""The fused combine (MOE_OPT_FUSED_COMBINE): the routed down projection
multiplies each row by its routing weight and adds it into [T, D] fp32 sums
with atomics; the last kernel adds the shared row and rounds.  Same bars as
the default path against the fp64 oracle (2e-2 / 6e-2 * RMS(out), near ties
left out), on every tile kernel, and within a few bf16 ulps of the default
path's output (only the summation order of a token's k rows differs)."""
import numpy as np
import pytest
import torch

import mixture_experts_layer_gating_gb300 as moe
import workloads
from tests.test_gpu_parity import LAYER_CASES, check_layer, run_layer
from tests.test_gpu_w8a8 import A8_LAYERS, check_layer_a8
from tests._lib import ensure_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return ensure_library()


@pytest.fixture
def fused():
    old = moe.moe_set_option(moe.MOE_OPT_FUSED_COMBINE, 1)
    yield
    moe.moe_set_option(moe.MOE_OPT_FUSED_COMBINE, old)


@pytest.fixture(params=["default", "cta1", "pair", "decode16", "decode"])
def kernels(request):
    pair = moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, {"cta1": 0, "pair": 1}.get(request.param, 3))
    dec = moe.moe_set_option(moe.MOE_OPT_DECODE_KERNEL, {"decode": 2, "decode16": 3}.get(request.param, 1))
    yield request.param
    moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, pair)
    moe.moe_set_option(moe.MOE_OPT_DECODE_KERNEL, dec)


@pytest.mark.parametrize("case", ["qwen3_T512", "qwen3_T64_decode", "gemma4_T256", "qwen35_T64",
                                  "qwen3_zipf_T384", "fp8_small_T300"])
def test_layer_parity_fused_combine(case, fused, kernels):
    shape = LAYER_CASES[case]
    check_layer(shape, layout="nk" if shape.w_dtype == "fp8_e4m3" else "kn")


def test_layer_parity_fused_combine_full_qwen3_prefill(fused):
    check_layer(workloads.CONFIGS["qwen3_prefill"])


@pytest.mark.parametrize("case", ["fp8_small_T300", "prefill_like_T2048"])
def test_layer_w8a8_fused_combine(case, fused):
    check_layer_a8(A8_LAYERS[case])


@pytest.mark.parametrize("case", ["qwen3_T512", "gemma4_T256"])
def test_fused_combine_close_to_fixed_order(case):
    """Against the default path's output on the same inputs (bf16 layers,
    whose expert rows the default keeps in fp32): the two differ only in the
    fp32 summation order of a token's rows, so by at most a few bf16 ulps of
    the output (and are mostly identical).  fp8 layers are left out here: their
    default path rounds each expert row to bf16 before the combine, the fused
    one does not, so the two differ by that rounding (both are checked against
    the oracle above)."""
    shape = LAYER_CASES[case]
    layout = "nk" if shape.w_dtype == "fp8_e4m3" else "kn"
    inp = workloads.make_inputs(shape, seed=21, device="cuda")
    base = run_layer(shape, inp, layout)["out"].double()
    old = moe.moe_set_option(moe.MOE_OPT_FUSED_COMBINE, 1)
    try:
        got = run_layer(shape, inp, layout)["out"].double()
    finally:
        moe.moe_set_option(moe.MOE_OPT_FUSED_COMBINE, old)
    d = (got - base).abs()
    ulp = base.abs().clamp_min(2.0 ** -20) * 2.0 ** -7
    assert bool((d <= 2 * ulp).all()), f"max diff {float(d.max()):.3e}"
    assert float((d == 0).double().mean()) > 0.5
