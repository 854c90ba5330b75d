"""The C-ABI library loads, exports every symbol include/moe.h declares, and
its host-side logic (workspace sizing, argument validation, status text)
behaves as documented.  No GPU needed: nothing here reaches a CUDA call."""
import ctypes

import pytest

import mixture_experts_layer_gating_gb300 as moe
import workloads
from tests._lib import ensure_library


@pytest.fixture(scope="module")
def lib():
    return ensure_library()


def test_exports_every_header_symbol(lib):
    names = moe.header_symbols()
    assert {"moe_route", "moe_permute", "moe_grouped_ffn", "moe_finalize", "moe_layer",
            "moe_workspace_size"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/moe.h but not exported"


@pytest.mark.parametrize("name", sorted(workloads.CONFIGS))
def test_workspace_size_covers_intermediates(lib, name):
    shape = workloads.CONFIGS[name]
    cfg = moe.config_from_shape(shape)
    n = moe.moe_workspace_size(cfg)
    ab = 4 if shape.act_dtype == "f32" else 2
    R = shape.R
    need = R * shape.D * ab * 2 + R * shape.I * ab + shape.T * shape.E * 4
    assert n >= need
    nslots = len(moe.WS_SLOTS) if shape.w_dtype == "fp8_e4m3" else 12
    offs = [moe.moe_workspace_offset(cfg, i) for i in range(nslots)]
    if shape.w_dtype != "fp8_e4m3":
        assert moe.moe_workspace_offset(cfg, 12) == 2 ** 64 - 1
    assert all(o % 256 == 0 for o in offs)
    assert offs == sorted(offs) and offs[-1] < n
    fp8_extra = (1 + (2 if shape.I_shared else 1)) if shape.w_dtype == "fp8_e4m3" else 0
    if shape.T * shape.k <= 8192:
        routing = 1  # small batches: init_routing and the gather in one kernel
    else:
        # one cluster launch (histogram, scan, scatter), and the gather kernel
        # unless the routed GEMM gathers its rows itself (bf16 layers with at
        # least 32 rows per expert, MOE_OPT_GATHER_A's default)
        gemm_gathers = shape.act_dtype == "bf16" and shape.w_dtype == "bf16" and \
            shape.T * shape.k >= 32 * shape.E
    # router projection and top-k as one kernel: bf16 activations, 64 <= E, and
    # more than the CUDA-core projection takes (64 tokens, 2^25 multiply-adds)
    # (and a grid of at least 64 CTAs: prefill batches; see bench.fused_router)
    fused = shape.act_dtype == "bf16" and shape.E >= 64 and not (
        shape.T <= 64 and shape.T * shape.D * shape.E <= 2 ** 25) and shape.T >= 2048
    if shape.T * shape.k > 8192:
        # the sort from the fused router's histograms, or the cluster sort up
        # to 65536 expanded rows: one launch; two kernels otherwise
        one = fused or shape.T * shape.k <= 65536
        routing = (1 if one else 2) + (0 if gemm_gathers else 1)
    # router (+ top-k), 2 (+2 shared) GEMMs, finalize
    base = (6 if fused else 7) if shape.I_shared else (4 if fused else 5)
    assert moe.moe_layer_launch_count(cfg) == base + fp8_extra + routing


@pytest.mark.parametrize("bad", [
    dict(k=0), dict(k=9, E=8), dict(E=513, k=8), dict(D=12), dict(I=100), dict(T=-1),
    dict(act=7), dict(k=17, E=64), dict(D=8, w_dtype="fp8_e4m3"),
])
def test_invalid_configs_rejected(lib, bad):
    base = dict(T=64, D=256, E=8, k=2, I=128)
    acts = {"act": bad.pop("act")} if "act" in bad else {}
    base.update(bad)
    cfg = moe.make_config(**{k: v for k, v in base.items()})
    if acts:
        cfg.act = acts["act"]
    assert moe.moe_workspace_size(cfg) == 0
    assert moe.moe_layer_launch_count(cfg) == 0


def _call_layer(lib, cfg, ptrs, ws, ws_bytes):
    return lib.moe_layer(ctypes.byref(cfg), *ptrs, ws, ws_bytes, None)


def test_host_validation_codes(lib):
    cfg = moe.make_config(64, 256, 8, 2, 128)
    n = moe.moe_workspace_size(cfg)
    good = 1 << 20  # a fake, aligned device address: validation fails before any use
    ptrs = [good, good, None, good, None, good, None, None, None, None, None, good]
    # workspace problems
    assert _call_layer(lib, cfg, ptrs, None, n) == -5
    assert _call_layer(lib, cfg, ptrs, good + 16, n) == -5
    assert _call_layer(lib, cfg, ptrs, good, n - 1) == -5
    # null / misaligned tensors
    bad = list(ptrs); bad[0] = None
    assert _call_layer(lib, cfg, bad, good, n) == -1
    bad = list(ptrs); bad[3] = good + 8
    assert _call_layer(lib, cfg, bad, good, n) == -1
    # fp8 weights need scales; bf16 weights must not get them
    cfg8 = moe.make_config(64, 256, 8, 2, 128, w_dtype="fp8_e4m3")
    assert _call_layer(lib, cfg8, ptrs, good, moe.moe_workspace_size(cfg8)) == -1
    bad = list(ptrs); bad[4] = good
    assert _call_layer(lib, cfg, bad, good, n) == -1
    # unsupported dtype pair
    cfg_mix = moe.make_config(64, 256, 8, 2, 128, act_dtype="f32", w_dtype="bf16")
    assert _call_layer(lib, cfg_mix, ptrs, good, moe.moe_workspace_size(cfg_mix)) == -2
    # shared expert weights required when I_shared > 0
    cfg_s = moe.make_config(64, 256, 8, 2, 128, I_shared=64)
    assert _call_layer(lib, cfg_s, ptrs, good, moe.moe_workspace_size(cfg_s)) == -1
    # T == 0 is a no-op that touches nothing
    cfg0 = moe.make_config(0, 256, 8, 2, 128)
    assert _call_layer(lib, cfg0, ptrs, good, moe.moe_workspace_size(cfg0)) == 0


def test_status_strings(lib):
    for st in (0, -1, -2, -3, -4, -5):
        assert moe.moe_status_string(st)
    assert "unknown" in moe.moe_status_string(12345)


def test_stage_validation(lib):
    cfg = moe.make_config(64, 256, 8, 2, 128)
    n = moe.moe_workspace_size(cfg)
    g = 1 << 20
    # moe_route: bias without x is rejected; missing outputs rejected
    assert lib.moe_route(ctypes.byref(cfg), None, None, g, g, g, g, g, n, None) == -1
    assert lib.moe_route(ctypes.byref(cfg), g, g, None, None, g, g, g, n, None) == -1
    # moe_permute: gather requested without destination
    assert lib.moe_permute(ctypes.byref(cfg), g, g, g, g, g, g, None, g, n, None) == -1
    # moe_finalize: missing weights
    assert lib.moe_finalize(ctypes.byref(cfg), g, g, None, None, g, g, n, None) == -1
    # moe_grouped_ffn: misaligned h
    assert lib.moe_grouped_ffn(ctypes.byref(cfg), g, g, g, None, g, None, g + 4, g, None, None,
                               None, None, None, None, None, g, n, None) == -1


def test_set_option_values():
    """moe_set_option returns the previous value, clamps ranges, rejects unknown options."""
    ensure_library()
    with pytest.raises(moe.MoEError):
        moe.moe_set_option(99, 1)
    cases = [
        (moe.MOE_OPT_PAIR_TILES, 5, 3),
        (moe.MOE_OPT_PAIR_TILES, 1, 1),
        (moe.MOE_OPT_GATHER_A, 1, 1),
        (moe.MOE_OPT_GATHER_A, 2, 2),
        (moe.MOE_OPT_GATHER_A, 9, 3),
        (moe.MOE_OPT_GATHER_A, 3, 3),
        (moe.MOE_OPT_GATHER_A, -1, 0),
        (moe.MOE_OPT_DECODE_KERNEL, 7, 3),
        (moe.MOE_OPT_DECODE_KERNEL, -3, 0),
        (moe.MOE_OPT_PDL, 0, 0),
        (moe.MOE_OPT_PDL, 3, 1),
        (moe.MOE_OPT_SHARED_STREAM, 0, 0),
        (moe.MOE_OPT_SHARED_STREAM, 2, 2),
        (moe.MOE_OPT_SHARED_STREAM, 5, 2),
        (moe.MOE_OPT_SHARED_STREAM, 1, 1),
        (moe.MOE_OPT_FUSED_COMBINE, 5, 1),
        (moe.MOE_OPT_FUSED_COMBINE, 0, 0),
        (moe.MOE_OPT_TILE_ORDER, 3, 1),
        (moe.MOE_OPT_TILE_ORDER, 0, 0),
        (moe.MOE_OPT_SHARED_IN_GEMM, 4, 1),
        (moe.MOE_OPT_SHARED_IN_GEMM, 0, 0),
        (moe.MOE_OPT_B_PREFETCH, 4, 4),
        (moe.MOE_OPT_B_PREFETCH, 99, 16),
        (moe.MOE_OPT_B_PREFETCH, -2, 0),
        (moe.MOE_OPT_DYNAMIC_TILES, 3, 2),
        (moe.MOE_OPT_DYNAMIC_TILES, 1, 1),
        (moe.MOE_OPT_DYNAMIC_TILES, 0, 0),
        (moe.MOE_OPT_SHARED_CTAS, 48, 48),
        (moe.MOE_OPT_SHARED_CTAS, -5, 0),
        (moe.MOE_OPT_FUSED_ROUTING, 0, 0),
        (moe.MOE_OPT_FUSED_ROUTING, 2, 2),
        (moe.MOE_OPT_FUSED_ROUTING, 3, 3),
        (moe.MOE_OPT_FUSED_ROUTING, 7, 3),
        (moe.MOE_OPT_FUSED_ROUTING, 1, 1),
    ]
    for opt, value, stored in cases:
        old = moe.moe_set_option(opt, value)
        assert moe.moe_set_option(opt, old) == stored


@pytest.mark.parametrize("T,E,D,k,fused", [
    (4096, 128, 2048, 8, True),    # Qwen3-MoE prefill
    (16384, 256, 8192, 8, True),   # Ling-style prefill
    (8192, 512, 4096, 10, True),   # two expert halves
    (512, 256, 8192, 8, False),    # decode batch: 16 CTAs, the split-K projection
    (64, 128, 2048, 8, False),     # decode: the CUDA-core projection
    (4096, 32, 2048, 4, False),    # fewer than 64 experts
    (4096, 128, 2050, 8, False),   # D not a multiple of 8 (row pitch)
])
def test_fused_router_launch_count(T, E, D, k, fused):
    """moe_layer makes one launch fewer where the router projection and the
    top-k run as one kernel (MOE_OPT_FUSED_ROUTING), none fewer for them where
    that kernel does not apply, and one more fewer where init_routing's
    histogram and scatter run as one launch (more than 8192 expanded rows:
    from the fused router's histograms, or as one cluster up to 65536 rows)."""
    ensure_library()
    cfg = moe.make_config(T, D, E, k, 768)
    old = moe.moe_set_option(moe.MOE_OPT_FUSED_ROUTING, 1)
    try:
        n_on = moe.moe_layer_launch_count(cfg)
        moe.moe_set_option(moe.MOE_OPT_FUSED_ROUTING, 0)
        n_off = moe.moe_layer_launch_count(cfg)
    finally:
        moe.moe_set_option(moe.MOE_OPT_FUSED_ROUTING, old)
    if D % 8:
        assert n_on == n_off == 0  # invalid configuration
    else:
        R = T * k
        one_sort = R > 8192 and (fused or R <= 65536)
        assert n_on == n_off - (1 if fused else 0) - (1 if one_sort else 0)


def test_fp8_nk_layout_host_logic(lib):
    """MOE_FP8_E4M3_NK: accepted with bf16 activations, the same launch count
    as the [.., K, N] fp8 layout, and the same workspace but for the T extra
    rows its shared expert may take as the last group of the routed GEMMs
    (two-term e4m3 rows take the fp16 rows' bytes); rejected with fp32
    activations or widths not a multiple of 16; moe_pack_weights_nk
    validates before enqueueing anything."""
    for name in ("ling_prefill", "ling_decode"):
        shape = workloads.CONFIGS[name]
        kn, nk = moe.config_from_shape(shape), moe.config_from_shape(shape, "nk")
        assert nk.w_dtype == moe.MOE_FP8_E4M3_NK
        T, D, I = shape.T, shape.D, shape.I
        extra = T * D * 2 + T * I * 4 + T * D * 4 + T * 4 + T * I * 2 + T * 4  # x_perm, h, y, scales, h rows
        assert 0 < moe.moe_workspace_size(nk) - moe.moe_workspace_size(kn) <= extra + 8 * 256
        assert moe.moe_layer_launch_count(nk) == moe.moe_layer_launch_count(kn)
        for i in range(8):  # the regions before the permuted rows sit at the same offsets
            assert moe.moe_workspace_offset(nk, i) == moe.moe_workspace_offset(kn, i)
    assert moe.moe_workspace_size(moe.make_config(64, 264, 8, 2, 128, w_dtype="fp8_e4m3_nk")) == 0
    good = 1 << 20
    cfg32 = moe.make_config(64, 256, 8, 2, 128, act_dtype="f32", w_dtype="fp8_e4m3_nk")
    ptrs = [good] * 12
    assert _call_layer(lib, cfg32, ptrs, good, moe.moe_workspace_size(cfg32)) == -2
    with pytest.raises(ValueError):
        moe.config_from_shape(workloads.CONFIGS["ling_decode"], "mn")
    P = lib.moe_pack_weights_nk
    assert P(good, 1, 40, 64, good * 8, None) == -1          # K not a multiple of 16
    assert P(good, 1, 64, 24, good * 8, None) == -1          # N not a multiple of 16
    assert P(good, 0, 64, 64, good * 8, None) == -1          # no matrices
    assert P(good + 8, 1, 64, 64, good * 8, None) == -1      # misaligned source
    assert P(None, 1, 64, 64, good * 8, None) == -1          # null source
    assert P(good, 2, 64, 64, good + 4096, None) == -1       # overlapping buffers
