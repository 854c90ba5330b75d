"""The shared expert as the last group of the routed grouped GEMMs
(MOE_OPT_SHARED_IN_GEMM): its token rows follow the routed rows in the
permuted buffer and its tiles follow the routed tiles in the same launches.
Same bars against the fp64 oracle as the default path, on layers whose shared
expert has the experts' width (bf16, two-term e4m3 and W8A8 weights, with and
without the fused combine, decode and prefill sizes); close to the side-stream
path's output; layers whose shared expert is wider (Gemma-4's dense MLP) keep
their own launches."""
import dataclasses

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
def in_gemm():
    old = moe.moe_set_option(moe.MOE_OPT_SHARED_IN_GEMM, 1)
    yield
    moe.moe_set_option(moe.MOE_OPT_SHARED_IN_GEMM, old)


C = workloads.CONFIGS
CASES = {
    "qwen35_T64": LAYER_CASES["qwen35_T64"],
    "qwen35_T600": dataclasses.replace(C["qwen35_prefill"].with_tokens(600), name="qwen35_T600"),
    "fp8_small_T300": LAYER_CASES["fp8_small_T300"],
    "ling_T64": LAYER_CASES["ling_T64"],
    "fp8_prefill_like": workloads.MoEShape("fp8_prefill_like", 2048, 1024, 16, 4, 512, I_shared=512,
                                           w_dtype="fp8_e4m3"),
    "bf16_prefill_like": workloads.MoEShape("bf16_prefill_like", 2048, 1024, 16, 4, 512, I_shared=512),
    "gemma4_T256_wider_shared": LAYER_CASES["gemma4_T256"],
}


@pytest.mark.parametrize("fused", [0, 1])
@pytest.mark.parametrize("case", sorted(CASES))
def test_layer_parity_shared_in_gemm(case, fused, in_gemm):
    shape = CASES[case]
    old = moe.moe_set_option(moe.MOE_OPT_FUSED_COMBINE, fused)
    try:
        check_layer(shape, layout="nk" if shape.w_dtype == "fp8_e4m3" else "kn")
    finally:
        moe.moe_set_option(moe.MOE_OPT_FUSED_COMBINE, old)


@pytest.mark.parametrize("case", ["fp8_small_T300", "prefill_like_T2048"])
def test_layer_w8a8_shared_in_gemm(case, in_gemm):
    check_layer_a8(A8_LAYERS[case])


@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("case", ["bf16_prefill_like", "qwen35_T600", "fp8_prefill_like"])
def test_shared_in_gemm_bit_identical_to_separate_launches(case, pair):
    """Against the layer with the shared expert in its own launches, on the
    same tile kernel (1-CTA or 2-CTA tiles for every pass): the same tiles
    compute the same sums, so the outputs are bit-identical.  (Under the
    default policy a separate shared expert of a few hundred tokens takes
    2-CTA tiles while the routed launch it joins may take 1-CTA tiles; the
    outputs then differ only by that kernel's accumulation order.)"""
    shape = CASES[case]
    layout = "nk" if shape.w_dtype == "fp8_e4m3" else "kn"
    inp = workloads.make_inputs(shape, seed=23, device="cuda")
    old_pair = moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, pair)
    try:
        base = run_layer(shape, inp, layout)["out"].double()
        old = moe.moe_set_option(moe.MOE_OPT_SHARED_IN_GEMM, 1)
        try:
            got = run_layer(shape, inp, layout)["out"].double()
        finally:
            moe.moe_set_option(moe.MOE_OPT_SHARED_IN_GEMM, old)
    finally:
        moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, old_pair)
    assert torch.equal(got, base)


def test_shared_in_gemm_launch_count():
    """A layer that takes the path makes no launches of its own for the shared
    expert (two GEMMs fewer; fp8 layers one row conversion fewer).  A bf16
    prefill layer then also takes the permuted copy of x (one gather launch
    more) instead of the routed GEMM's own row gather, since the shared
    expert's rows are appended to the permuted rows."""
    for name, layout, fewer in [("qwen35_prefill", "kn", 1), ("ling_prefill", "nk", 3),
                                ("gemma4_prefill", "kn", 0)]:
        cfg = moe.config_from_shape(C[name], layout)
        old = moe.moe_set_option(moe.MOE_OPT_SHARED_IN_GEMM, 0)
        n0 = moe.moe_layer_launch_count(cfg)
        moe.moe_set_option(moe.MOE_OPT_SHARED_IN_GEMM, 1)
        n1 = moe.moe_layer_launch_count(cfg)
        moe.moe_set_option(moe.MOE_OPT_SHARED_IN_GEMM, old)
        assert n0 - n1 == fewer, name


@pytest.mark.parametrize("name,layout", [("qwen35_prefill", "kn"), ("ling_prefill", "nk")])
def test_full_size_shared_in_gemm(name, layout, in_gemm):
    from tests.test_gpu_full_size import test_full_size_workload
    test_full_size_workload(name, layout)
