"""GPU parity of the W8A8 layers (MOE_FP8_E4M3_NK_A8): K-contiguous e4m3
weights, activations quantised per row to one e4m3 term with a dynamic
scale, one 8-bit tensor-core product per multiply-add.

The oracle emulates the same quantisation (oracle.quantize_rows_e4m3,
moe_layer(act_quant="e4m3_row")).  A quantised code is an integer decided by
floating point, so each decision is compared where both sides take it on the
same input: the codes and scales of x bit-exact (x is the layer's bf16
input); h (bf16) against the oracle's h within one bf16 rounding; y against
the oracle's down projection of the GPU's own h, quantised by the oracle
(same input, same decisions), within the bf16 rounding of y.  The whole layer
is compared with the oracle's emulation at the fp8 bar (6e-2 * RMS(out)),
leaving out near-tie tokens and tokens one of whose h rows has a different
largest |h| in bf16 on the two sides (that flips the row's scale, and with
it many of its codes); both counts are printed and bounded.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_gating_gb300 as moe
import oracle
import workloads
from tests._lib import ensure_library, max_near_ties, rms
from tests.test_gpu_parity import _grouped_case, check_close, tile_mode  # noqa: F401

pytestmark = pytest.mark.gpu
A8 = oracle.ACT_QUANT_E4M3_ROW


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return ensure_library()


def quant_deq(a):
    """The oracle's per-row e4m3 quantisation of bf16 rows, dequantised (fp64)."""
    return oracle.dequantize_rows(*oracle.quantize_rows_e4m3(oracle.to_f64(a)))


def y_from_gpu_h(h_gpu, offsets, W2, s2):
    """The oracle's down projection of the GPU's own bf16 h, quantised per row
    by the oracle: the same decisions as the kernel's, on the same input."""
    hq = quant_deq(h_gpu)
    y = np.zeros((hq.shape[0], W2.shape[-1]))
    for e in range(len(offsets) - 1):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a < b:
            y[a:b] = oracle.scaled_projection(hq[a:b], oracle.to_f64(W2[e]), oracle.to_f64(s2[e]))
    return y


GROUPED_CASES = [
    (4, [300, 0, 129, 1], 256, 128, "swiglu"),     # empty expert, ragged tails
    (2, [200, 57], 512, 384, "geglu_tanh"),        # column tile past I: zero-filled weight rows
    (3, [5, 140, 0], 192, 64, "swiglu"),           # K = 192: half of the second k-block past K
    (2, [700, 300], 256, 128, "swiglu"),           # >= 150 rows per group: 2-CTA tiles by default
    (3, [1000, 0, 560], 1024, 768, "geglu_tanh"),  # several 256-row tiles per group
    (1, [77], 16, 32, "swiglu"),                   # K and N at their minimum
]


@pytest.mark.parametrize("E,counts,D,I,act", GROUPED_CASES)
def test_grouped_ffn_w8a8_parity(E, counts, D, I, act, tile_mode):
    xp, offsets, W13, W2, s13, s2 = _grouped_case(E, counts, D, I, act, seed=E + D + I + 9, fp8=True)
    R = xp.shape[0]
    cfg = moe.make_config(R, D, E, 1, I, act=act, w_dtype="fp8_e4m3_nk_a8")
    ws = moe.alloc_workspace(cfg)
    h = torch.empty((R, I), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((R, D), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_ffn(cfg, xp, torch.from_numpy(offsets).cuda(), moe.pack_weights_nk(W13), s13,
                        moe.pack_weights_nk(W2), s2, h, y, ws=ws)
    assert moe.moe_read_device_status(ws) == 0
    # the permuted rows the GEMM read: the oracle's codes and scales, bit-exact
    q_o, s_o = oracle.quantize_rows_e4m3(oracle.to_f64(xp.cpu()))
    xq = moe.workspace_view(ws, cfg, "x_perm", (R, D), torch.uint8).cpu().view(torch.float8_e4m3fn)
    sc = moe.workspace_view(ws, cfg, "row_inv", (R,), torch.float32).cpu()
    assert np.array_equal(xq.double().numpy(), q_o), "x codes differ from the oracle's"
    assert np.array_equal(sc.double().numpy(), s_o), "x scales differ from the oracle's"
    # h before its bf16 rounding (the oracle's W8A8 h is rounded; comparing two
    # roundings would allow a one-ulp difference): one bf16 rounding of the GPU
    h_o, _ = oracle.grouped_ffn(oracle.dequantize_rows(q_o, s_o), offsets, W13.cpu(), W2.cpu(), act,
                                s13.cpu(), s2.cpu())
    check_close("h", h.cpu().double().numpy(), h_o, 2.0 ** -8, 1e-4)
    y_ref = y_from_gpu_h(h.cpu(), offsets, W2.cpu(), s2.cpu())
    check_close("y", y.cpu().double().numpy(), y_ref, 2.0 ** -8, 1e-5)


@pytest.mark.parametrize("act", ["swiglu", "geglu_tanh"])
@pytest.mark.parametrize("pair_mode", [0, 1])
def test_grouped_ffn_w8a8_tail_sizes(act, pair_mode):
    """Every kind of last tile of a group on 128-row tiles (mode 0) and on
    2-CTA 256-row tiles with swapped tails (mode 1, each CTA loading half of
    a tail's rows)."""
    counts = [1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 80, 95, 96, 97, 112, 127, 128, 129, 200, 224,
              225, 256, 300, 385, 449, 511]
    E, D, I = len(counts), 320, 256
    old = moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, pair_mode)
    try:
        xp, offsets, W13, W2, s13, s2 = _grouped_case(E, counts, D, I, act, seed=pair_mode + 7 * len(act),
                                                      fp8=True)
        R = xp.shape[0]
        cfg = moe.make_config(R, D, E, 1, I, act=act, w_dtype="fp8_e4m3_nk_a8")
        ws = moe.alloc_workspace(cfg)
        h = torch.empty((R, I), dtype=torch.bfloat16, device="cuda")
        y = torch.empty((R, D), dtype=torch.bfloat16, device="cuda")
        moe.moe_grouped_ffn(cfg, xp, torch.from_numpy(offsets).cuda(), moe.pack_weights_nk(W13), s13,
                            moe.pack_weights_nk(W2), s2, h, y, ws=ws)
        assert moe.moe_read_device_status(ws) == 0
        h_o, _ = oracle.grouped_ffn(quant_deq(xp.cpu()), offsets, W13.cpu(), W2.cpu(), act,
                                    s13.cpu(), s2.cpu())  # h before its bf16 rounding
        check_close("h", h.cpu().double().numpy(), h_o, 2.0 ** -8, 1e-4)
        check_close("y", y.cpu().double().numpy(), y_from_gpu_h(h.cpu(), offsets, W2.cpu(), s2.cpu()),
                    2.0 ** -8, 1e-5)
    finally:
        moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, old)


def run_layer_a8(shape, inp):
    cfg = moe.config_from_shape(shape, "nk_a8")
    ws = moe.alloc_workspace(cfg)
    out = torch.empty((shape.T, shape.D), dtype=torch.bfloat16, device="cuda")
    W = {n: (None if inp[n] is None else moe.pack_weights_nk(inp[n])) for n in ("W13", "W2", "W13s", "W2s")}
    moe.moe_layer(cfg, inp["x"], inp["Wg"], inp["logit_bias"], W["W13"], inp["s13"], W["W2"],
                  inp["s2"], W["W13s"], inp["s13s"], W["W2s"], inp["s2s"], out, ws)
    assert moe.moe_read_device_status(ws) == 0
    return cfg, ws, out


def amax_flips(h_gpu, h_oracle):
    """Rows whose largest |h| differs between the GPU's bf16 h and the
    oracle's h rounded to bf16 (their quantisation scales differ)."""
    a = np.abs(oracle.to_f64(h_gpu)).max(axis=1)
    b = np.abs(oracle.bf16_round(h_oracle)).max(axis=1)
    return a != b


def check_layer_a8(shape, seed=0):
    T, E, k, D, R = shape.T, shape.E, shape.k, shape.D, shape.R
    inp = workloads.make_inputs(shape, seed=seed, device="cuda")
    cfg, ws, out = run_layer_a8(shape, inp)
    view = lambda slot, shp, dt: moe.workspace_view(ws, cfg, slot, shp, dt).cpu()  # noqa: E731
    cinp = {kk: (v.cpu() if isinstance(v, torch.Tensor) else v) for kk, v in inp.items()}
    # routing, given the GPU's logits: bit-exact
    L_gpu = view("logits", (T, E), torch.float32).double().numpy()
    ids = view("topk_ids", (T, k), torch.int32).numpy()
    ids_o, _ = oracle.topk_softmax(L_gpu, k, shape.renormalize)
    assert np.array_equal(ids, ids_o)
    r = oracle.init_routing(ids, E)
    sorted_rows = view("sorted_rows", (R,), torch.int32).numpy()
    assert np.array_equal(sorted_rows, r["sorted_rows"])
    # x: codes and scales bit-exact; the permuted rows are copies of them
    q_o, s_o = oracle.quantize_rows_e4m3(oracle.to_f64(cinp["x"]))
    xq = view("x16", (T, D), torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(xq, q_o), "x codes differ from the oracle's"
    assert np.array_equal(view("tok_inv", (T,), torch.float32).double().numpy(), s_o)
    xpq = view("x_perm", (R, D), torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(xpq, q_o[sorted_rows // k]), "permuted rows must be copies of the codes"
    assert np.array_equal(view("row_inv", (R,), torch.float32).double().numpy(), s_o[sorted_rows // k])
    # the layer against the oracle's emulation
    ref = oracle.moe_layer(cinp, k, shape.act, shape.renormalize, act_quant=A8)
    ties = oracle.near_tie_tokens(ref["logits"], k)
    # routed h rows: GPU position p holds expanded row sorted_rows[p], which the
    # oracle holds at its own position dest_o[sorted_rows[p]] (a different
    # expert's row only for a near-tie token, which is left out anyway)
    h_gpu = view("h", (R, shape.I), torch.bfloat16)
    flip_rows = amax_flips(h_gpu, ref["h"][ref["dest"][sorted_rows]])
    flips = np.zeros(T, dtype=bool)
    flips[sorted_rows[flip_rows] // k] = True
    if shape.I_shared:
        # the shared expert's h: its own region, or rows R .. R+T-1 of h when it
        # ran as the last group of the routed GEMMs
        in_gemm = moe.moe_set_option(moe.MOE_OPT_SHARED_IN_GEMM, 0)
        moe.moe_set_option(moe.MOE_OPT_SHARED_IN_GEMM, in_gemm)
        if in_gemm and shape.I_shared == shape.I:
            hs_gpu = view("h", (R + T, shape.I), torch.bfloat16)[R:]
        else:
            hs_gpu = view("h_shared", (T, shape.I_shared), torch.bfloat16)
        xs = oracle.dequantize_rows(q_o, s_o)
        gu = oracle.scaled_projection(xs, oracle.to_f64(cinp["W13s"]), oracle.to_f64(cinp["s13s"]))
        Is = shape.I_shared
        hs_o = oracle.activation(gu[:, :Is], shape.act) * gu[:, Is:]
        flips |= amax_flips(hs_gpu, hs_o)
    print(f"{shape.name} W8A8: {int(ties.sum())} near-tie and {int(flips.sum())} h-scale-flip tokens "
          f"of {T} left out")
    assert ties.sum() <= max_near_ties(T)
    assert flips.sum() <= max_near_ties(T)
    keep = ~(ties | flips)
    got = out.cpu().double().numpy()
    err = np.abs(got - ref["out"])[keep]
    scale = rms(ref["out"])
    assert err.max() <= 6e-2 * scale, f"max|err| {err.max():.3e} > 6e-2 * RMS {scale:.3e}"
    # and how far W8A8 lies from the exact (bf16-activation) layer, for the record
    exact = oracle.moe_layer(cinp, k, shape.act, shape.renormalize)["out"]
    print(f"  vs emulation {err.max() / scale:.3e} RMS; vs exact layer "
          f"{np.abs(got - exact)[keep].max() / rms(exact):.3e} RMS")
    return err.max() / scale


C = workloads.CONFIGS
A8_LAYERS = {
    "fp8_small_T300": workloads.MoEShape("fp8_small", 300, 512, 16, 4, 256, I_shared=256, w_dtype="fp8_e4m3"),
    "fp8_small_geglu_T77": workloads.MoEShape("fp8_small_geglu", 77, 384, 24, 3, 320, I_shared=128,
                                              act=workloads.ACT_GEGLU_TANH, w_dtype="fp8_e4m3"),
    "ling_T64": C["ling_decode"].with_tokens(64),
    # ~512 rows per expert: 2-CTA tiles with swapped tails, as at full Ling size
    "prefill_like_T2048": workloads.MoEShape("fp8_prefill_like", 2048, 1024, 16, 4, 512, I_shared=512,
                                             w_dtype="fp8_e4m3"),
}


@pytest.mark.parametrize("case", sorted(A8_LAYERS))
def test_layer_w8a8_parity(case):
    check_layer_a8(A8_LAYERS[case])


@pytest.mark.parametrize("case", ["ling_T64", "prefill_like_T2048"])
@pytest.mark.parametrize("mode", ["cta1", "decode", "decode16"])
def test_layer_w8a8_other_tile_kernels(case, mode):
    pair = moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, 0)
    dec = moe.moe_set_option(moe.MOE_OPT_DECODE_KERNEL, {"cta1": 0, "decode": 2, "decode16": 3}[mode])
    try:
        check_layer_a8(A8_LAYERS[case])
    finally:
        moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, pair)
        moe.moe_set_option(moe.MOE_OPT_DECODE_KERNEL, dec)


def test_layer_w8a8_zero_rows():
    """Tokens whose x is all zero get scale 1 and zero codes; their routed and
    shared rows are zero, so their output is exactly zero."""
    shape = A8_LAYERS["fp8_small_T300"]
    inp = workloads.make_inputs(shape, seed=4, device="cuda")
    inp["x"][[0, 7, 299]] = 0
    cfg, ws, out = run_layer_a8(shape, inp)
    sc = moe.workspace_view(ws, cfg, "tok_inv", (shape.T,), torch.float32).cpu()
    assert torch.equal(sc[[0, 7, 299]], torch.ones(3))
    assert not out[[0, 7, 299]].any()


@pytest.mark.parametrize("name", ["ling_prefill", "ling_decode"])
def test_full_size_w8a8(name):
    """The Ling-style layers at full size in W8A8: routing of every token and
    the codes of every x row bit-exact; a seeded sample of tokens (first and
    last included) against the oracle's emulation run on those tokens alone."""
    shape = C[name]
    T, E, k, D, R = shape.T, shape.E, shape.k, shape.D, shape.R
    inp = workloads.make_inputs(shape, seed=11, device="cuda")
    cfg, ws, out = run_layer_a8(shape, inp)
    view = lambda slot, shp, dt: moe.workspace_view(ws, cfg, slot, shp, dt).cpu()  # noqa: E731
    logits = view("logits", (T, E), torch.float32).double().numpy()
    ids = view("topk_ids", (T, k), torch.int32).numpy()
    assert np.array_equal(ids, oracle.topk_softmax(logits, k, shape.renormalize)[0])
    r = oracle.init_routing(ids, E)
    dest = view("dest", (R,), torch.int32).numpy()
    assert np.array_equal(dest, r["dest"])
    q_o, s_o = oracle.quantize_rows_e4m3(oracle.to_f64(inp["x"].cpu()))
    assert np.array_equal(view("x16", (T, D), torch.uint8).view(torch.float8_e4m3fn).double().numpy(), q_o)
    assert np.array_equal(view("tok_inv", (T,), torch.float32).double().numpy(), s_o)

    gen = np.random.default_rng(T + E + 1)
    n = min(T, 256 if T > 4096 else 64)
    tokens = np.unique(np.concatenate([[0, T - 1], gen.choice(T, n, replace=False)]))
    sub = {kk: (v.cpu() if isinstance(v, torch.Tensor) else v) for kk, v in inp.items()}
    sub["x"] = sub["x"][torch.from_numpy(tokens)]
    ref = oracle.moe_layer(sub, k, shape.act, shape.renormalize, act_quant=A8)
    ties = oracle.near_tie_tokens(ref["logits"], k)
    # h-scale flips of the sampled tokens' routed and shared rows
    h_gpu = view("h", (R, shape.I), torch.bfloat16)
    rows_gpu = dest[(tokens[:, None] * k + np.arange(k)[None, :]).ravel()]
    rows_ref = ref["dest"][np.arange(len(tokens) * k)]
    flips = amax_flips(h_gpu[torch.from_numpy(rows_gpu)], ref["h"][rows_ref]).reshape(-1, k).any(axis=1)
    in_gemm = moe.moe_set_option(moe.MOE_OPT_SHARED_IN_GEMM, 0)
    moe.moe_set_option(moe.MOE_OPT_SHARED_IN_GEMM, in_gemm)
    hs_all = (view("h", (R + T, shape.I), torch.bfloat16)[R:] if in_gemm and shape.I_shared == shape.I
              else view("h_shared", (T, shape.I_shared), torch.bfloat16))
    hs_gpu = hs_all[torch.from_numpy(tokens)]
    xs = oracle.dequantize_rows(*oracle.quantize_rows_e4m3(oracle.to_f64(sub["x"])))
    gu = oracle.scaled_projection(xs, oracle.to_f64(sub["W13s"]), oracle.to_f64(sub["s13s"]))
    Is = shape.I_shared
    flips |= amax_flips(hs_gpu, oracle.activation(gu[:, :Is], shape.act) * gu[:, Is:])
    print(f"{name} W8A8: {int(ties.sum())} near-tie and {int(flips.sum())} h-scale-flip tokens of "
          f"{len(tokens)} sampled left out")
    assert ties.sum() <= max_near_ties(len(tokens)) and flips.sum() <= max_near_ties(len(tokens))
    keep = ~(ties | flips)
    got = out[torch.from_numpy(tokens).cuda()].double().cpu().numpy()
    err = np.abs(got - ref["out"])[keep]
    scale = rms(ref["out"][keep])
    assert err.max() <= 6e-2 * scale, f"{name}: max|err| {err.max():.3e} > 6e-2 * RMS {scale:.3e}"
