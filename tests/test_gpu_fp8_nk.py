"""GPU parity of the fp8 layers whose weights are stored K-contiguous
(MOE_FP8_E4M3_NK): the one-time weight transpose, the two-term e4m3 rows,
the grouped FFN on every tile kernel, and whole layers against the fp64
oracle (same bars as the other fp8 layers: routing bit-exact, outputs within
6e-2 * RMS(out)).
"""
import dataclasses

import numpy as np
import pytest
import torch

import mixture_experts_layer_gating_gb300 as moe
import oracle
import workloads
from tests._lib import ensure_library, rms
from tests.test_gpu_parity import LAYER_CASES, _grouped_case, check_close, check_layer, tile_mode  # noqa: F401

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return ensure_library()


@pytest.mark.parametrize("G,K,N", [(3, 48, 80), (1, 8192, 64), (2, 128, 4096), (5, 16, 16), (1, 2064, 208)])
def test_pack_weights_nk_bit_exact(G, K, N):
    gen = torch.Generator(device="cuda").manual_seed(G * K + N)
    W = torch.randint(0, 256, (G, K, N), generator=gen, dtype=torch.uint8, device="cuda")
    assert torch.equal(moe.pack_weights_nk(W), W.transpose(1, 2).contiguous())
    assert torch.equal(moe.pack_weights_nk(W[0]), W[0].t().contiguous())


def test_pack_weights_nk_rejects_bad_shapes():
    W = torch.zeros((2, 32, 40), dtype=torch.uint8, device="cuda")  # N not a multiple of 16
    with pytest.raises(moe.MoEError):
        moe.pack_weights_nk(W)


def two_term_rows(h):
    """Emulates the library's bf16 / fp32 rows -> two-term e4m3 rows: a power
    of two 2^e with the row's largest |h| * 2^e in [128, 256), hi = e4m3(v),
    lo = e4m3(v - hi), round to nearest even; returns (hi + lo) / 2^e in fp64."""
    h = h.float()
    m = h.abs().amax(dim=1, keepdim=True)
    e = torch.where(m > 0, 8 - torch.frexp(m).exponent, torch.zeros_like(m, dtype=torch.int32))
    sc = torch.pow(2.0, e.double()).float()
    v = h * sc
    hi = v.to(torch.float8_e4m3fn).float()
    lo = (v - hi).to(torch.float8_e4m3fn).float()
    return (hi.double() + lo.double()) / sc.double()


GROUPED_CASES = [
    (4, [300, 0, 129, 1], 256, 128, "swiglu"),     # empty expert, ragged tails
    (2, [200, 57], 512, 384, "geglu_tanh"),        # column tile past I: zero-filled weight rows
    (3, [5, 140, 0], 192, 64, "swiglu"),           # K = 192: half of the second k-block past K
    (2, [700, 300], 256, 128, "swiglu"),           # >= 150 rows per group: 2-CTA tiles by default
    (3, [1000, 0, 560], 1024, 768, "geglu_tanh"),  # several 256-row tiles per group
    (1, [77], 16, 32, "swiglu"),                   # K and N at their minimum
]


@pytest.mark.parametrize("E,counts,D,I,act", GROUPED_CASES)
def test_grouped_ffn_nk_parity(E, counts, D, I, act, tile_mode):
    """h (bf16: one rounding) against the oracle from x carried exactly by its
    two-term rows; y (bf16) against the GPU's own h, rounded as the library
    rounds it to two-term rows, times the dequantised W2 (one bf16 rounding)."""
    xp, offsets, W13, W2, s13, s2 = _grouped_case(E, counts, D, I, act, seed=E + D + I + 5, fp8=True)
    R = xp.shape[0]
    cfg = moe.make_config(R, D, E, 1, I, act=act, w_dtype="fp8_e4m3_nk")
    ws = moe.alloc_workspace(cfg)
    h = torch.empty((R, I), dtype=torch.bfloat16, device="cuda")  # K-contiguous fp8: bf16 h
    y = torch.empty((R, D), dtype=torch.bfloat16, device="cuda")  # fp8 layers: bf16 expert rows
    moe.moe_grouped_ffn(cfg, xp, torch.from_numpy(offsets).cuda(), moe.pack_weights_nk(W13), s13,
                        moe.pack_weights_nk(W2), s2, h, y, ws=ws)
    assert moe.moe_read_device_status(ws) == 0
    h_o, y_o = oracle.grouped_ffn(oracle.to_f64(xp.cpu()), offsets, W13.cpu(), W2.cpu(), act,
                                  s13.cpu(), s2.cpu())
    check_close("h", h.cpu().double().numpy(), h_o, 2.0 ** -8, 1e-4)
    hq = two_term_rows(h.cpu()).numpy()
    y_ref = np.zeros((R, D))
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        y_ref[a:b] = oracle.scaled_projection(hq[a:b], oracle.to_f64(W2[e].cpu()), oracle.to_f64(s2[e].cpu()))
    check_close("y", y.cpu().double().numpy(), y_ref, 2.0 ** -8, 1e-5)
    # and against the exact layer: h carried to 8 significant bits
    check_close("y vs oracle", y.cpu().double().numpy(), y_o, 2.0 ** -7, 2e-2)


@pytest.mark.parametrize("act", ["swiglu", "geglu_tanh"])
@pytest.mark.parametrize("pair_mode", [0, 1])
def test_grouped_ffn_nk_tail_sizes(act, pair_mode):
    """Every kind of last tile of a group on 128-row tiles (mode 0) and on
    2-CTA 256-row tiles (mode 1): 1 row, multiples of 16 and their
    neighbours, exact multiples of the tile height.  The down pass has 320
    output columns: a full 256-row weight tile and one with 64 rows of
    weights (the rest of the box zero-filled)."""
    counts = [1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 80, 95, 96, 97, 112, 127, 128, 129, 200, 224,
              225, 256, 300, 385, 449, 511]
    E, D, I = len(counts), 320, 256
    old = moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, pair_mode)
    try:
        xp, offsets, W13, W2, s13, s2 = _grouped_case(E, counts, D, I, act, seed=pair_mode + 3 * len(act), fp8=True)
        R = xp.shape[0]
        cfg = moe.make_config(R, D, E, 1, I, act=act, w_dtype="fp8_e4m3_nk")
        ws = moe.alloc_workspace(cfg)
        h = torch.empty((R, I), dtype=torch.bfloat16, device="cuda")  # K-contiguous fp8: bf16 h
        y = torch.empty((R, D), dtype=torch.bfloat16, device="cuda")  # fp8 layers: bf16 expert rows
        moe.moe_grouped_ffn(cfg, xp, torch.from_numpy(offsets).cuda(), moe.pack_weights_nk(W13), s13,
                            moe.pack_weights_nk(W2), s2, h, y, ws=ws)
        assert moe.moe_read_device_status(ws) == 0
        h_o, _ = oracle.grouped_ffn(oracle.to_f64(xp.cpu()), offsets, W13.cpu(), W2.cpu(), act,
                                    s13.cpu(), s2.cpu())
        check_close("h", h.cpu().double().numpy(), h_o, 2.0 ** -8, 1e-4)
        hq = two_term_rows(h.cpu()).numpy()
        y_ref = np.zeros((R, D))
        for e in range(E):
            a, b = offsets[e], offsets[e + 1]
            y_ref[a:b] = oracle.scaled_projection(hq[a:b], oracle.to_f64(W2[e].cpu()),
                                                  oracle.to_f64(s2[e].cpu()))
        check_close("y", y.cpu().double().numpy(), y_ref, 2.0 ** -8, 1e-5)
    finally:
        moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, old)


def test_nk_weights_with_subnormal_codes(tile_mode):
    """Weight codes mostly from the e4m3 subnormal range go to the tensor core
    unchanged: y against the GPU's h (two-term rounding emulated) times the
    dequantised weights."""
    E, D, I = 2, 256, 128
    counts = [150, 90]
    R = sum(counts)
    gen = torch.Generator(device="cuda").manual_seed(13)
    codes = torch.tensor([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=torch.uint8)
    sub = torch.tensor([c for c in range(256) if (c & 0x78) == 0 and (c & 7) != 0], dtype=torch.uint8)

    def draw(shape):
        pick_sub = torch.rand(shape, generator=gen, device="cuda") < 0.8
        a = sub.cuda()[torch.randint(0, len(sub), shape, generator=gen, device="cuda")]
        b = codes.cuda()[torch.randint(0, len(codes), shape, generator=gen, device="cuda")]
        return torch.where(pick_sub, a, b).view(torch.float8_e4m3fn)

    W13, W2 = draw((E, D, 2 * I)), draw((E, I, D))
    s13 = torch.rand((E, 2 * I), generator=gen, device="cuda") * 0.01 + 0.001
    s2 = torch.rand((E, D), generator=gen, device="cuda") * 0.01 + 0.001
    xp = torch.randn((R, D), generator=gen, device="cuda").to(torch.bfloat16)
    offsets = np.array([0, counts[0], R], dtype=np.int32)
    cfg = moe.make_config(R, D, E, 1, I, w_dtype="fp8_e4m3_nk")
    ws = moe.alloc_workspace(cfg)
    h = torch.empty((R, I), dtype=torch.bfloat16, device="cuda")  # K-contiguous fp8: bf16 h
    y = torch.empty((R, D), dtype=torch.bfloat16, device="cuda")  # fp8 layers: bf16 expert rows
    moe.moe_grouped_ffn(cfg, xp, torch.from_numpy(offsets).cuda(), moe.pack_weights_nk(W13), s13,
                        moe.pack_weights_nk(W2), s2, h, y, ws=ws)
    assert moe.moe_read_device_status(ws) == 0
    h_o, _ = oracle.grouped_ffn(oracle.to_f64(xp.cpu()), offsets, W13.cpu(), W2.cpu(), "swiglu",
                                s13.cpu(), s2.cpu())
    check_close("h", h.cpu().double().numpy(), h_o, 2.0 ** -8, 1e-4)
    hq = two_term_rows(h.cpu()).numpy()
    y_ref = np.zeros((R, D))
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        y_ref[a:b] = oracle.scaled_projection(hq[a:b], oracle.to_f64(W2[e].cpu()), oracle.to_f64(s2[e].cpu()))
    check_close("y", y.cpu().double().numpy(), y_ref, 2.0 ** -8, 1e-5)
    assert rms(y_ref) > 0


NK_LAYERS = {
    "fp8_small_T300": LAYER_CASES["fp8_small_T300"],
    "fp8_small_geglu_T77": LAYER_CASES["fp8_small_geglu_T77"],
    "ling_T64": LAYER_CASES["ling_T64"],
    # 512 rows per group: 2-CTA tiles by default
    "fp8_T2048": workloads.MoEShape("fp8_T2048", 2048, 512, 16, 4, 256, I_shared=256, w_dtype="fp8_e4m3"),
    "ling_T1": LAYER_CASES["ling_T64"].with_tokens(1),
    # rows of 1040 and 1296 elements: thread groups of 64 whose last vectors
    # run past the row (the register-resident row conversion), ragged N tiles
    "fp8_rows_1040_1296": workloads.MoEShape("fp8_rows", 300, 1040, 8, 2, 1296, I_shared=1040,
                                             w_dtype="fp8_e4m3"),
}


@pytest.mark.parametrize("case", sorted(NK_LAYERS))
def test_layer_parity_nk(case):
    check_layer(NK_LAYERS[case], layout="nk")


@pytest.mark.parametrize("pair,decode", [(0, 0), (1, 0), (0, 2), (0, 3)])
@pytest.mark.parametrize("case", ["fp8_T2048", "ling_T64"])
def test_layer_parity_nk_tile_kernels(case, pair, decode):
    """The same layers on 1-CTA and 2-CTA tiles and on the decode kernel
    with 64- and 16-row tiles."""
    old_p = moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, pair)
    old_d = moe.moe_set_option(moe.MOE_OPT_DECODE_KERNEL, decode)
    try:
        check_layer(NK_LAYERS[case], layout="nk")
    finally:
        moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, old_p)
        moe.moe_set_option(moe.MOE_OPT_DECODE_KERNEL, old_d)


def test_nk_layer_matches_kn_layer_routing():
    """Both fp8 layouts see the same x and logits: identical routing, outputs
    within the fp8 bar of each other."""
    shape = NK_LAYERS["fp8_small_T300"]
    from tests.test_gpu_parity import run_layer

    inp = workloads.make_inputs(shape, seed=21, device="cuda")
    a, b = run_layer(shape, inp, "kn"), run_layer(shape, inp, "nk")
    for key in ("logits", "ids", "w", "counts", "offsets", "sorted_rows", "dest"):
        assert torch.equal(a[key], b[key]), key
    ref = a["out"].double().numpy()
    assert np.abs(b["out"].double().numpy() - ref).max() <= 6e-2 * rms(ref)


@pytest.mark.parametrize("case", ["fp8_small_T300", "fp8_T2048", "ling_T64"])
def test_layer_parity_nk_gemm_gathers_rows(case):
    """MOE_OPT_GATHER_A with e4m3 rows: the routed gate/up GEMM gathers the
    hi and lo terms of its rows from x's two-term rows with TMA gather4."""
    old = moe.moe_set_option(moe.MOE_OPT_GATHER_A, 1)
    try:
        check_layer(NK_LAYERS[case], layout="nk")
    finally:
        moe.moe_set_option(moe.MOE_OPT_GATHER_A, old)
