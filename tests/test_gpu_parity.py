"""GPU parity: every stage and the whole layer, through the C ABI, against the
CPU fp64 oracle on the same seeded inputs.

Bars: routing ids / counts / offsets / permutation bit-exact given the same
fp32 router logits; gate weights within 1e-6; layer outputs within
2e-2 * RMS(out) (bf16, fp32) or 6e-2 * RMS(out) (fp8), with tokens whose k-th
and (k+1)-th oracle logits lie within 1e-4 left out of the output and id
comparisons.
"""
import dataclasses

import numpy as np
import pytest
import torch

import mixture_experts_layer_gating_gb300 as moe
import oracle
import workloads
from tests._lib import ensure_library, max_near_ties, rms, tol_factor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return ensure_library()


def _cpu(d):
    return {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def packed_weights(inp, layout):
    """The layer's weight tensors in the layout the configuration names: as
    drawn ("kn"), or fp8 weights transposed once by moe_pack_weights_nk ("nk")."""
    names = ("W13", "W2", "W13s", "W2s")
    if layout == "kn":
        return {n: inp[n] for n in names}
    return {n: (None if inp[n] is None else moe.pack_weights_nk(inp[n])) for n in names}


def run_layer(shape, inp, layout="kn"):
    cfg = moe.config_from_shape(shape, layout)
    ws = moe.alloc_workspace(cfg)
    out = torch.empty((shape.T, shape.D), dtype=workloads.torch_dtype(shape.act_dtype), device="cuda")
    W = packed_weights(inp, layout)
    moe.moe_layer(cfg, inp["x"], inp["Wg"], inp["logit_bias"], W["W13"], inp["s13"], W["W2"],
                  inp["s2"], W["W13s"], inp["s13s"], W["W2s"], inp["s2s"], out, ws)
    flags = moe.moe_read_device_status(ws)
    assert flags == 0, f"device error flags {flags:#x}"
    R = shape.R
    view = lambda slot, shp, dt: moe.workspace_view(ws, cfg, slot, shp, dt).cpu()  # noqa: E731
    adt = workloads.torch_dtype(shape.act_dtype)
    res = {
        "out": out.cpu(),
        "logits": view("logits", (shape.T, shape.E), torch.float32),
        "ids": view("topk_ids", (shape.T, shape.k), torch.int32),
        "w": view("topk_w", (shape.T, shape.k), torch.float32),
        "counts": view("counts", (shape.E,), torch.int32),
        "offsets": view("offsets", (shape.E + 1,), torch.int32),
        "sorted_rows": view("sorted_rows", (R,), torch.int32),
        "dest": view("dest", (R,), torch.int32),
        "x_perm": view("x_perm", (R, shape.D), adt),
    }
    if shape.w_dtype == "fp8_e4m3":
        # fp16 rows, or two-term e4m3 rows (hi bytes, then lo bytes)
        res["x16"] = (view("x16", (shape.T, shape.D), torch.float16) if layout == "kn"
                      else view("x16", (shape.T, 2 * shape.D), torch.uint8))
        res["tok_inv"] = view("tok_inv", (shape.T,), torch.float32)
    return res


def check_two_term_rows(q, inv, x):
    """Two-term e4m3 rows [n, 2D] (hi bytes, then lo) with inverse power-of-two
    scales reproduce x exactly where |x| >= 2^-9 of the row's largest |x|, and
    within 2^-17 of it elsewhere; the scaled largest lies in [128, 256)."""
    D = x.shape[1]
    hi = q[:, :D].contiguous().view(torch.float8_e4m3fn).double()
    lo = q[:, D:].contiguous().view(torch.float8_e4m3fn).double()
    inv = inv.double()[:, None]
    xd = x.double()
    amax = xd.abs().amax(dim=1, keepdim=True)
    live = amax[:, 0] > 0
    assert torch.all((amax / inv)[live] >= 128) and torch.all((amax / inv)[live] < 256)
    rec = (hi + lo) * inv
    big = xd.abs() >= amax * 2.0 ** -9
    assert torch.equal(rec[big], xd[big]), "two-term e4m3 rows must carry x exactly"
    assert torch.all((rec - xd).abs() <= amax * 2.0 ** -17)


def check_layer(shape, seed=0, layout="kn"):
    inp = workloads.make_inputs(shape, seed=seed, device="cuda")
    g = run_layer(shape, inp, layout)
    cinp = _cpu(inp)
    k, E = shape.k, shape.E

    # 1. routing, given the GPU's own fp32 logits: bit-exact ids, weights to 1e-6
    L_gpu = g["logits"].double().numpy()
    ids_o, w_o = oracle.topk_softmax(L_gpu, k, shape.renormalize)
    assert np.array_equal(g["ids"].numpy(), ids_o), "top-k ids differ (same logits)"
    assert np.max(np.abs(g["w"].double().numpy() - w_o)) <= 1e-6
    r = oracle.init_routing(g["ids"].numpy(), E)
    assert np.array_equal(g["counts"].numpy(), r["counts"])
    assert np.array_equal(g["offsets"].numpy(), r["offsets"])
    assert np.array_equal(g["sorted_rows"].numpy(), r["sorted_rows"])
    assert np.array_equal(g["dest"].numpy(), r["dest"])
    gathered = moe.moe_set_option(moe.MOE_OPT_GATHER_A, 0)
    moe.moe_set_option(moe.MOE_OPT_GATHER_A, gathered)
    if not gathered or shape.act_dtype == "f32":
        # materialised permuted rows: a bit-exact copy of x (fp8: of its fp16 rows)
        xs = cinp["x"][torch.from_numpy(r["sorted_rows"] // k)]
        if shape.w_dtype == "fp8_e4m3":
            xs = g["x16"][torch.from_numpy(r["sorted_rows"] // k)]
            assert torch.equal(g["x_perm"].view(xs.dtype).reshape(xs.shape), xs)
        else:
            assert torch.equal(g["x_perm"], xs), "permutation gather must copy rows bit-exactly"
    if shape.w_dtype == "fp8_e4m3" and layout == "nk":
        check_two_term_rows(g["x16"], g["tok_inv"], cinp["x"])
    elif shape.w_dtype == "fp8_e4m3":
        # fp16 rows times exact powers of two: scaling back gives x bit-exactly
        x16 = g["x16"].float()
        inv = g["tok_inv"].float()[:, None]
        assert torch.equal((x16 * inv).to(torch.bfloat16), cinp["x"]), "fp16 row scaling must be exact"

    # 2. router projection against the fp64 definition
    L_ref = oracle.router_logits(cinp["x"], cinp["Wg"], cinp["logit_bias"])
    assert np.max(np.abs(L_gpu - L_ref)) <= 1e-3 * max(1.0, rms(L_ref))

    # 3. the layer output against the fp64 oracle (its own logits)
    ref = oracle.moe_layer(cinp, k, shape.act, shape.renormalize)
    ties = oracle.near_tie_tokens(ref["logits"], k)
    print(f"{shape.name}: {int(ties.sum())} of {shape.T} tokens with a near tie left out")
    assert ties.sum() <= max_near_ties(shape.T), f"{int(ties.sum())} near-tie tokens of {shape.T}"
    same = (ref["ids"] == g["ids"].numpy()).all(axis=1)
    assert (same | ties).all(), "ids differ on a token without a near tie"
    keep = ~ties
    out_g = g["out"].double().numpy()
    err = np.abs(out_g - ref["out"])[keep]
    scale = rms(ref["out"])
    assert np.isfinite(out_g).all()
    assert err.max() <= tol_factor(shape) * scale, \
        f"max|err| {err.max():.3e} > {tol_factor(shape)} * RMS {scale:.3e} ({int(ties.sum())} near-tie tokens left out)"
    return {"max_err_over_rms": float(err.max() / scale), "near_ties": int(ties.sum())}


C = workloads.CONFIGS
LAYER_CASES = {
    "toy": C["toy"],
    "qwen3_T512": C["qwen3_prefill"].with_tokens(512),
    "qwen3_T1": C["qwen3_decode"].with_tokens(1),
    "qwen3_T64_decode": C["qwen3_decode"],
    "qwen3_zipf_T384": dataclasses.replace(C["qwen3_prefill"].with_tokens(384), zipf=1.1, name="qwen3_zipf"),
    "gemma4_T256": C["gemma4_prefill"].with_tokens(256),
    "gemma4_T8_decode": C["gemma4_decode"],
    "qwen35_T64": C["qwen35_decode64"],
    "fp8_small_T300": workloads.MoEShape("fp8_small", 300, 512, 16, 4, 256, I_shared=256,
                                         w_dtype="fp8_e4m3"),
    "fp8_small_geglu_T77": workloads.MoEShape("fp8_small_geglu", 77, 384, 24, 3, 320, I_shared=128,
                                              act=workloads.ACT_GEGLU_TANH, w_dtype="fp8_e4m3"),
    "ling_T64": C["ling_decode"].with_tokens(64),
}


@pytest.mark.parametrize("case", sorted(LAYER_CASES))
def test_layer_parity(case):
    check_layer(LAYER_CASES[case])


@pytest.mark.parametrize("case", ["qwen3_T64_decode", "gemma4_T8_decode", "ling_T64", "qwen35_T64"])
def test_layer_parity_decode_sizes_on_tile_kernel(case):
    """Decode-size layers with the swap-AB kernel switched off (128-row tiles)."""
    old = moe.moe_set_option(moe.MOE_OPT_DECODE_KERNEL, 0)
    try:
        check_layer(LAYER_CASES[case])
    finally:
        moe.moe_set_option(moe.MOE_OPT_DECODE_KERNEL, old)


def test_layer_parity_full_qwen3_prefill(tile_mode):
    """The benchmarked workload at full size (T=4096), every token checked."""
    check_layer(C["qwen3_prefill"])


@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("case", ["qwen3_T512", "qwen3_T64_decode", "fp8_small_T300", "gemma4_T256",
                                  "toy"])
def test_layer_same_result_without_pdl(case, pair):
    """Programmatic dependent launch changes only when kernels are scheduled:
    the layer output is bit-identical with MOE_OPT_PDL on and off."""
    shape = LAYER_CASES[case]
    inp = workloads.make_inputs(shape, seed=3, device="cuda")
    old_pair = moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, pair)
    old = moe.moe_set_option(moe.MOE_OPT_PDL, 1)
    try:
        with_pdl = run_layer(shape, inp)["out"].clone()
        moe.moe_set_option(moe.MOE_OPT_PDL, 0)
        assert torch.equal(run_layer(shape, inp)["out"], with_pdl)
    finally:
        moe.moe_set_option(moe.MOE_OPT_PDL, old)
        moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, old_pair)


SIDE_CASES = {
    **{c: (LAYER_CASES[c], "kn") for c in ["gemma4_T256", "gemma4_T8_decode", "fp8_small_T300",
                                            "fp8_small_geglu_T77", "qwen35_T64"]},
    # more than 8192 expanded rows and the permutation kernel: the late fork
    # comes between init_routing and the permutation
    "qwen35_T1024": (C["qwen35_prefill"].with_tokens(1024), "kn"),
    "ling_T1100_nk": (C["ling_prefill"].with_tokens(1100), "nk"),
}


@pytest.mark.parametrize("fork", [1, 2])
@pytest.mark.parametrize("case", sorted(SIDE_CASES))
def test_layer_same_result_with_shared_expert_stream(case, fork):
    """The shared expert on the library's side stream, forked once x is ready
    (1, default) or after init_routing (2), and on the caller's stream give
    bit-identical outputs, over repeated calls."""
    shape, layout = SIDE_CASES[case]
    inp = workloads.make_inputs(shape, seed=7, device="cuda")
    old = moe.moe_set_option(moe.MOE_OPT_SHARED_STREAM, 0)
    try:
        serial = run_layer(shape, inp, layout)["out"].clone()
        moe.moe_set_option(moe.MOE_OPT_SHARED_STREAM, fork)
        for _ in range(3):
            assert torch.equal(run_layer(shape, inp, layout)["out"], serial)
    finally:
        moe.moe_set_option(moe.MOE_OPT_SHARED_STREAM, old)


@pytest.mark.parametrize("case", ["gemma4_T256", "qwen35_T1024", "ling_T1100_nk"])
def test_layer_same_result_with_capped_shared_grid(case):
    """MOE_OPT_SHARED_CTAS: the shared expert's side-stream GEMMs on at most 24
    CTAs (2-CTA tiles: 12 clusters) give the layer bit for bit, forked either
    way."""
    shape, layout = SIDE_CASES[case]
    inp = workloads.make_inputs(shape, seed=9, device="cuda")
    old = moe.moe_set_option(moe.MOE_OPT_SHARED_STREAM, 0)
    old_ctas = moe.moe_set_option(moe.MOE_OPT_SHARED_CTAS, 24)
    try:
        serial = run_layer(shape, inp, layout)["out"].clone()
        for fork in (1, 2):
            moe.moe_set_option(moe.MOE_OPT_SHARED_STREAM, fork)
            assert torch.equal(run_layer(shape, inp, layout)["out"], serial)
    finally:
        moe.moe_set_option(moe.MOE_OPT_SHARED_STREAM, old)
        moe.moe_set_option(moe.MOE_OPT_SHARED_CTAS, old_ctas)


DYN_CASES = [
    # case, layout, pair-tile policy, gather policy
    ("qwen3_T512", "kn", 3, 3),         # bf16: cp.async row gather (one-CTA tiles), 2-CTA down pass
    ("qwen3_T512", "kn", 0, 0),         # bf16 one-CTA tiles, permuted copy
    ("qwen3_T512", "kn", 1, 0),         # bf16 2-CTA tiles with swapped tails, both passes
    ("gemma4_T256", "kn", 1, 0),        # GEGLU + dense MLP on 2-CTA tiles
    ("qwen35_T64", "kn", 0, 0),         # shared expert, 128-row tiles
    ("fp8_small_T300", "kn", 0, 0),     # fp8 weights expanded on chip (converter warps)
    ("fp8_small_T300", "nk", 1, 0),     # K-contiguous e4m3 weights, 2-CTA tiles
    ("fp8_small_T300", "nk", 0, 0),
    ("fp8_small_geglu_T77", "nk", 1, 0),
]


@pytest.mark.parametrize("case,layout,pair,gather", DYN_CASES)
def test_layer_dynamic_tiles_same_result(case, layout, pair, gather):
    """MOE_OPT_DYNAMIC_TILES: tiles handed out by an atomic counter through
    the shared-memory tile queue give the layer bit for bit (every tile is
    computed the same way whichever CTA takes it), on every tile kernel, and
    the result passes the oracle bar."""
    shape = LAYER_CASES[case]
    inp = workloads.make_inputs(shape, seed=3, device="cuda")
    old_pair = moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, pair)
    old_gather = moe.moe_set_option(moe.MOE_OPT_GATHER_A, gather)
    old_dec = moe.moe_set_option(moe.MOE_OPT_DECODE_KERNEL, 0)  # the tile kernels, not swap-AB
    old = moe.moe_set_option(moe.MOE_OPT_DYNAMIC_TILES, 0)
    try:
        base = run_layer(shape, inp, layout)["out"].clone()
        moe.moe_set_option(moe.MOE_OPT_DYNAMIC_TILES, 1)
        for _ in range(3):
            assert torch.equal(run_layer(shape, inp, layout)["out"], base)
        check_layer(shape, layout=layout)
    finally:
        moe.moe_set_option(moe.MOE_OPT_DYNAMIC_TILES, old)
        moe.moe_set_option(moe.MOE_OPT_DECODE_KERNEL, old_dec)
        moe.moe_set_option(moe.MOE_OPT_GATHER_A, old_gather)
        moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, old_pair)


@pytest.mark.parametrize("dist", [2, 7])
@pytest.mark.parametrize("case,layout,pair", [
    ("qwen3_T512", "kn", 3),       # bf16: the routed gate/up pass gathers its rows; 2-CTA down pass
    ("qwen3_T512", "kn", 0),       # bf16 on one-CTA tiles
    ("gemma4_T256", "kn", 1),      # bf16 2-CTA tiles with swapped tails
    ("fp8_small_T300", "nk", 1),   # K-contiguous e4m3 weights, 2-CTA tiles
    ("fp8_small_T300", "nk", 0),
])
def test_layer_parity_weight_prefetch(case, layout, pair, dist):
    """MOE_OPT_B_PREFETCH: the producer's L2 prefetch of weight boxes ahead
    (into the next tile near a tile's end) leaves the results unchanged."""
    old = moe.moe_set_option(moe.MOE_OPT_B_PREFETCH, dist)
    old_pair = moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, pair)
    try:
        check_layer(LAYER_CASES[case], layout=layout)
    finally:
        moe.moe_set_option(moe.MOE_OPT_B_PREFETCH, old)
        moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, old_pair)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("case", ["qwen3_T512", "fp8_small_T300", "gemma4_T256"])
def test_layer_parity_gemm_gathers_rows(case, mode):
    """MOE_OPT_GATHER_A: the routed gate/up GEMM reads x rows itself, with TMA
    gather4 (1) or, for bf16 layers, with cp.async gather warps (2; fp8 layers
    keep gather4)."""
    old = moe.moe_set_option(moe.MOE_OPT_GATHER_A, mode)
    try:
        check_layer(LAYER_CASES[case])
    finally:
        moe.moe_set_option(moe.MOE_OPT_GATHER_A, old)


# ------------------------------------------------------------------ stages
def _ws_for(cfg):
    return moe.alloc_workspace(cfg)


@pytest.mark.parametrize("E,k,renorm", [(128, 8, True), (512, 10, True), (8, 2, True), (64, 5, False), (16, 16, True)])
def test_route_from_logits_bit_exact(E, k, renorm):
    T = 777
    gen = torch.Generator(device="cuda").manual_seed(E * 31 + k)
    L = torch.randn((T, E), generator=gen, device="cuda")
    L[: T // 3] = torch.round(L[: T // 3] * 2) / 2  # many exact ties
    L[5] = 0.0  # a token whose logits are all equal
    cfg = moe.make_config(T, 64, E, k, 64, renormalize=renorm)
    ws = _ws_for(cfg)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, None, None, None, L, ids, w, ws)
    assert moe.moe_read_device_status(ws) == 0
    ids_o, w_o = oracle.topk_softmax(L.cpu().double().numpy(), k, renorm)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.max(np.abs(w.cpu().double().numpy() - w_o)) <= 1e-6
    assert np.array_equal(ids[5].cpu().numpy(), np.arange(k))


@pytest.mark.parametrize("T,E,k,renorm,bias,D", [
    (2048, 64, 4, 1, False, 256), (2048, 256, 16, 0, True, 256), (3000, 128, 8, 1, True, 256),
    (2047, 64, 4, 1, False, 256), (512, 256, 8, 0, True, 256), (512, 128, 8, 1, True, 2048),
    # up to 64 tokens: the CUDA-core projection (one plane at D = 256, else 4-8
    # planes over slices of D, the last slices shorter or empty)
    (64, 128, 8, 1, False, 2048), (8, 128, 8, 1, True, 2816), (1, 128, 8, 1, False, 2048),
    (3, 512, 10, 0, True, 4096), (33, 64, 4, 1, True, 256), (64, 512, 16, 1, False, 1024),
    (65, 128, 8, 1, False, 2048),  # one token past it: the tensor-core projection
])
def test_route_projection_then_topk_bit_exact(T, E, k, renorm, bias, D):
    """moe_route from x and W_g: routing bit-exact against the oracle's top-k of
    the GPU's own logits, logits against the fp64 projection.  Duplicate
    columns of W_g make exact ties that the lowest expert index must win."""
    gen = torch.Generator(device="cuda").manual_seed(T + E + k + D)
    x = torch.randn((T, D), generator=gen, device="cuda").to(torch.bfloat16)
    Wg = (0.05 * torch.randn((D, E), generator=gen, device="cuda")).to(torch.bfloat16)
    Wg[:, 5] = Wg[:, 3]
    Wg[:, 11] = Wg[:, 10]
    Wg[:, 12] = Wg[:, 10]
    tz = min(7, T - 1)
    x[tz] = 0  # a token whose logits are all equal (zero, plus the bias)
    b = (0.01 * torch.randn((E,), generator=gen, device="cuda")) if bias else None
    if bias:
        b[5] = b[3]
        b[11] = b[10]
        b[12] = b[10]
    cfg = moe.make_config(T, D, E, k, 64, renormalize=renorm)
    ws = _ws_for(cfg)
    L = torch.empty((T, E), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, x, Wg, b, L, ids, w, ws)
    assert moe.moe_read_device_status(ws) == 0
    L_gpu = L.cpu().double().numpy()
    ids_o, w_o = oracle.topk_softmax(L_gpu, k, renorm)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.max(np.abs(w.cpu().double().numpy() - w_o)) <= 1e-6
    L_ref = oracle.router_logits(x.cpu(), Wg.cpu(), b.cpu() if bias else None)
    assert np.max(np.abs(L_gpu - L_ref)) <= 1e-3 * max(1.0, rms(L_ref))
    if not bias:
        assert np.array_equal(ids[tz].cpu().numpy(), np.arange(k))


@pytest.mark.parametrize("T,E,k,pattern,D", [
    (1000, 128, 8, "uniform", 136), (3000, 512, 10, "uniform", 136), (129, 8, 2, "one_hot", 136),
    (4096, 256, 8, "skew", 136), (1, 4, 1, "uniform", 136), (2500, 64, 6, "empty_half", 136),
    # either side of the one-launch small-batch path (at most 8192 expanded rows)
    (1024, 512, 8, "uniform", 136), (8193, 16, 1, "skew", 136), (64, 128, 8, "skew", 136),
    # x above 32 MB: each token row read once and written to its k positions
    (4200, 64, 4, "skew", 4096), (5000, 32, 16, "uniform", 4104),
])
def test_permute_bit_exact(T, E, k, pattern, D):
    gen = np.random.default_rng(T + E + k)
    if pattern == "one_hot":  # expert 3 and 5 take every token
        ids = np.tile(np.array([3, 5]), (T, 1))
    elif pattern == "skew":
        p = 1.0 / np.arange(1, E + 1) ** 1.2
        ids = np.stack([gen.choice(E, k, replace=False, p=p / p.sum()) for _ in range(T)])
    elif pattern == "empty_half":
        ids = np.stack([gen.permutation(E // 2)[:k] * 2 for _ in range(T)])
    else:
        ids = np.stack([gen.permutation(E)[:k] for _ in range(T)])
    cfg = moe.make_config(T, D, E, k, 64)
    ws = _ws_for(cfg)
    tids = torch.from_numpy(ids.astype(np.int32)).cuda()
    x = torch.randn((T, D), device="cuda").to(torch.bfloat16)
    R = T * k
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    sr = torch.empty(R, dtype=torch.int32, device="cuda")
    dest = torch.empty(R, dtype=torch.int32, device="cuda")
    xp = torch.empty((R, D), dtype=torch.bfloat16, device="cuda")
    moe.moe_permute(cfg, tids, x, counts, offsets, sr, dest, xp, ws)
    assert moe.moe_read_device_status(ws) == 0
    r = oracle.init_routing(ids, E)
    assert np.array_equal(counts.cpu().numpy(), r["counts"])
    assert np.array_equal(offsets.cpu().numpy(), r["offsets"])
    assert np.array_equal(sr.cpu().numpy(), r["sorted_rows"])
    assert np.array_equal(dest.cpu().numpy(), r["dest"])
    assert torch.equal(xp.cpu(), x.cpu()[torch.from_numpy(r["sorted_rows"] // k)])
    # un-permute(permute(x)) is the identity
    assert torch.equal(xp[dest.long()].view(T, k, D)[:, 0], x)


@pytest.mark.parametrize("T,D", [(300, 64), (5000, 64), (5000, 4096)])  # small-batch, segmented, x > 32 MB
def test_permute_flags_bad_ids_without_fault(T, D):
    E, k = 16, 2
    ids = torch.randint(0, E, (T, k), dtype=torch.int32, device="cuda")
    ids[7, 1] = E
    ids[100, 0] = -3
    cfg = moe.make_config(T, D, E, k, 64)
    ws = _ws_for(cfg)
    R = T * k
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    sr = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    dest = torch.empty(R, dtype=torch.int32, device="cuda")
    x = torch.randn((T, D), device="cuda").to(torch.bfloat16)
    xp = torch.empty((R, D), dtype=torch.bfloat16, device="cuda")
    moe.moe_permute(cfg, ids, x, counts, offsets, sr, dest, xp, ws)
    flags = moe.moe_read_device_status(ws)
    assert flags & moe.MOE_DEV_BAD_EXPERT_ID
    assert int(offsets[E]) == R - 2
    d = dest.cpu().numpy()
    assert d[7 * k + 1] == -1 and d[100 * k] == -1
    # valid rows copied, the positions past them zero-filled
    nvalid = int(offsets[E])
    xc, xpc = x.cpu(), xp.cpu()
    assert torch.equal(xpc[:nvalid], xc[torch.from_numpy(sr.cpu().numpy()[:nvalid] // k)])
    assert int(torch.count_nonzero(xpc[nvalid:])) == 0
    assert moe.moe_read_device_status(ws) == 0  # reading clears the word


def check_close(name, got, ref, rel, rms_slack):
    """|got - ref| <= rel * |ref| + rms_slack * RMS(ref), element by element."""
    bound = np.abs(ref) * rel + rms_slack * rms(ref)
    bad = np.abs(got - ref) > bound
    assert not bad.any(), (f"{name}: {int(bad.sum())} elements off; worst "
                           f"{np.abs(got - ref).max():.3e} (RMS {rms(ref):.3e})")


def _grouped_case(E, counts, D, I, act, seed, fp8=False):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    R = int(sum(counts))
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    xp = torch.randn((R, D), generator=gen, device="cuda").to(torch.bfloat16)
    W13 = torch.randn((E, D, 2 * I), generator=gen, device="cuda") * 0.02
    W2 = torch.randn((E, I, D), generator=gen, device="cuda") * 0.02
    if fp8:
        (W13, s13), (W2, s2) = workloads.quantize_fp8_per_column(W13), workloads.quantize_fp8_per_column(W2)
        return xp, offsets, W13, W2, s13, s2
    return xp, offsets, W13.to(torch.bfloat16), W2.to(torch.bfloat16)


@pytest.fixture(params=["cta1", "pair", "pair_noswap", "decode", "decode16"])
def tile_mode(request):
    """Run a grouped-GEMM test on 128-row 1-CTA tiles, on 2-CTA (256-row)
    tiles with and without swapped tails, and on the swap-AB decode kernel
    with 64- and 16-row tiles."""
    pair = moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, {"pair": 1, "pair_noswap": 2}.get(request.param, 0))
    dec_mode = {"decode": 2, "decode16": 3}.get(request.param, 0)
    dec = moe.moe_set_option(moe.MOE_OPT_DECODE_KERNEL, dec_mode)
    yield request.param
    moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, pair)
    moe.moe_set_option(moe.MOE_OPT_DECODE_KERNEL, dec)


@pytest.mark.parametrize("E,counts,D,I,act", [
    (4, [300, 0, 129, 1], 256, 128, "swiglu"),            # empty expert, ragged tails
    (3, [1, 2, 3], 192, 64, "geglu_tanh"),                # tiny segments, K not a multiple of 64*4
    (2, [1000, 24], 2816, 704, "geglu_tanh"),             # Gemma widths: ragged column tile
    (8, [0, 0, 0, 513, 0, 0, 0, 0], 2048, 768, "swiglu"),  # one expert takes everything
    (1, [77], 72, 40, "swiglu"),                          # K < 64, N < 64
    # >= 192 rows per group: 2-CTA (M = 256) tiles, with a peer CTA that has
    # a partial or no row range in the last tile of a group
    (2, [700, 300], 256, 128, "swiglu"),
    (3, [1000, 0, 560], 2048, 768, "geglu_tanh"),
])
def test_grouped_ffn_parity(E, counts, D, I, act, tile_mode):
    xp, offsets, W13, W2 = _grouped_case(E, counts, D, I, act, seed=E * 7 + D)
    R = xp.shape[0]
    T = R  # k = 1 view
    cfg = moe.make_config(T, D, E, 1, I, act=act)
    ws = _ws_for(cfg)
    h = torch.empty((2, R, I), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((R, D), dtype=torch.float32, device="cuda")
    toff = torch.from_numpy(offsets).cuda()
    moe.moe_grouped_ffn(cfg, xp, toff, W13, None, W2, None, h, y, ws=ws)
    assert moe.moe_read_device_status(ws) == 0
    h_o, y_o = oracle.grouped_ffn(oracle.to_f64(xp.cpu()), offsets, W13.cpu(), W2.cpu(), act)
    hc = h.cpu().double()
    # the hi plane is h rounded to bf16; hi + lo carries h to ~2^-16 relative
    check_close("h_hi", hc[0].numpy(), h_o, 2.0 ** -8, 1e-4)
    check_close("h_hi+h_lo", (hc[0] + hc[1]).numpy(), h_o, 2.0 ** -15, 1e-4)
    # y is fp32: only fp32 accumulation differs from the exact value
    check_close("y", y.cpu().double().numpy(), y_o, 1e-4, 1e-4)


@pytest.mark.parametrize("act", ["swiglu", "geglu_tanh"])
@pytest.mark.parametrize("pair_mode", [1, 2])
def test_grouped_ffn_pair_tail_sizes(act, pair_mode):
    """2-CTA tiles, every kind of last tile: swapped tails of 1..64 (gate/up)
    and 1..128 (down) rows, full-height tails above that, exact multiples of
    256; mode 2 runs the same groups without swapped tails."""
    counts = [1, 16, 17, 31, 32, 33, 63, 64, 65, 100, 127, 128, 129, 130, 200, 240, 255, 256, 257,
              300, 320, 383, 384, 385, 449, 511, 512]
    E, D, I = len(counts), 256, 128
    old = moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, pair_mode)
    try:
        xp, offsets, W13, W2 = _grouped_case(E, counts, D, I, act, seed=pair_mode + len(act))
        R = xp.shape[0]
        cfg = moe.make_config(R, D, E, 1, I, act=act)
        ws = _ws_for(cfg)
        h = torch.empty((2, R, I), dtype=torch.bfloat16, device="cuda")
        y = torch.empty((R, D), dtype=torch.float32, device="cuda")
        moe.moe_grouped_ffn(cfg, xp, torch.from_numpy(offsets).cuda(), W13, None, W2, None, h, y, ws=ws)
        assert moe.moe_read_device_status(ws) == 0
        h_o, y_o = oracle.grouped_ffn(oracle.to_f64(xp.cpu()), offsets, W13.cpu(), W2.cpu(), act)
        hc = h.cpu().double()
        check_close("h_hi", hc[0].numpy(), h_o, 2.0 ** -8, 1e-4)
        check_close("h_hi+h_lo", (hc[0] + hc[1]).numpy(), h_o, 2.0 ** -15, 1e-4)
        check_close("y", y.cpu().double().numpy(), y_o, 1e-4, 1e-4)
    finally:
        moe.moe_set_option(moe.MOE_OPT_PAIR_TILES, old)


@pytest.mark.parametrize("E,counts,D,I,act", [
    (4, [300, 0, 129, 1], 256, 128, "swiglu"),
    (2, [200, 57], 512, 384, "geglu_tanh"),   # column tile past I: zero-filled raw boxes
    (3, [5, 140, 0], 128, 64, "swiglu"),      # N < 128: one partly filled raw box
    (2, [600, 129], 512, 256, "swiglu"),      # 2-CTA tiles with fp8 weights
])
def test_grouped_ffn_fp8_parity(E, counts, D, I, act, tile_mode):
    """W8A16: e4m3 weights expanded exactly on chip, per-column scales after
    the K reduction; h is a single bf16 plane for fp8 layers."""
    xp, offsets, W13, W2, s13, s2 = _grouped_case(E, counts, D, I, act, seed=E + D + I, fp8=True)
    R = xp.shape[0]
    cfg = moe.make_config(R, D, E, 1, I, act=act, w_dtype="fp8_e4m3")
    ws = _ws_for(cfg)
    h = torch.empty((R, I), dtype=torch.float32, device="cuda")
    y = torch.empty((R, D), dtype=torch.bfloat16, device="cuda")  # fp8 layers: bf16 expert rows
    moe.moe_grouped_ffn(cfg, xp, torch.from_numpy(offsets).cuda(), W13, s13, W2, s2, h, y, ws=ws)
    assert moe.moe_read_device_status(ws) == 0
    h_o, y_o = oracle.grouped_ffn(oracle.to_f64(xp.cpu()), offsets, W13.cpu(), W2.cpu(), act,
                                  s13.cpu(), s2.cpu())
    # h is fp32 (exact fp16 x rows, fp32 accumulation)
    check_close("h", h.cpu().double().numpy(), h_o, 1e-4, 1e-4)
    # y from h rounded once to fp16 (11 bits) relative to its row maximum, then to bf16
    check_close("y", y.cpu().double().numpy(), y_o, 2.0 ** -8, 2e-3)


def test_fp8_weight_expansion_is_exact_including_subnormals(tile_mode):
    """Weight codes drawn mostly from the e4m3 subnormal range (|q| < 2^-6):
    a conversion that flushed them would zero whole outputs.  y is checked
    against the GPU's own h times the dequantised W2 in fp64 (fp32-accumulation
    tolerance), h against act(x W13) from the dequantised W13."""
    E, D, I = 2, 256, 128
    counts = [150, 90]
    R = sum(counts)
    gen = torch.Generator(device="cuda").manual_seed(11)
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
    cfg = moe.make_config(R, D, E, 1, I, w_dtype="fp8_e4m3")
    ws = _ws_for(cfg)
    h = torch.empty((R, I), dtype=torch.float32, device="cuda")
    y = torch.empty((R, D), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_ffn(cfg, xp, torch.from_numpy(offsets).cuda(), W13, s13, W2, s2, h, y, ws=ws)
    assert moe.moe_read_device_status(ws) == 0
    h_o, _ = oracle.grouped_ffn(oracle.to_f64(xp.cpu()), offsets, W13.cpu(), W2.cpu(), "swiglu",
                                s13.cpu(), s2.cpu())
    check_close("h", h.cpu().double().numpy(), h_o, 1e-4, 1e-4)
    # the down projection sees h as fp16 rows times powers of two: emulate that
    # rounding, then compare with the dequantised W2 at fp32-accumulation accuracy
    h32 = h.cpu()
    rmax = h32.abs().amax(dim=1, keepdim=True)
    e = torch.where(rmax > 0, 14 - torch.frexp(rmax).exponent, torch.zeros_like(rmax, dtype=torch.int32))
    sc = torch.pow(2.0, e.double()).float()
    hg = ((h32 * sc).half().float() / sc).double().numpy()
    y_ref = np.zeros((R, D))
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        y_ref[a:b] = oracle.scaled_projection(hg[a:b], oracle.to_f64(W2[e].cpu()), oracle.to_f64(s2[e].cpu()))
    # fp32 accumulation, then one bf16 rounding
    check_close("y", y.cpu().double().numpy(), y_ref, 2.0 ** -8, 1e-5)
    assert rms(y_ref) > 0


def test_grouped_ffn_flags_bad_offsets_without_fault():
    E, D, I = 3, 128, 64
    xp, offsets, W13, W2 = _grouped_case(E, [10, 10, 10], D, I, "swiglu", seed=3)
    bad = torch.tensor([0, 20, 10, 30], dtype=torch.int32, device="cuda")  # not monotone
    cfg = moe.make_config(30, D, E, 1, I)
    ws = _ws_for(cfg)
    h = torch.zeros((2, 30, I), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((30, D), dtype=torch.float32, device="cuda")
    moe.moe_grouped_ffn(cfg, xp, bad, W13, None, W2, None, h, y, ws=ws)
    assert moe.moe_read_device_status(ws) & moe.MOE_DEV_BAD_OFFSETS


@pytest.mark.parametrize("T,k,D,shared", [(513, 8, 2048, False), (64, 10, 4096, True), (3, 1, 264, True)])
def test_finalize_parity(T, k, D, shared):
    gen = torch.Generator(device="cuda").manual_seed(T + k)
    R = T * k
    y = torch.randn((R, D), generator=gen, device="cuda")
    perm = torch.randperm(R, generator=gen, device="cuda").to(torch.int32)
    w = torch.rand((T, k), generator=gen, device="cuda")
    w = w / w.sum(1, keepdim=True)
    s = torch.randn((T, D), generator=gen, device="cuda") if shared else None
    out = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    cfg = moe.make_config(T, D, 16, k, 64)
    ws = _ws_for(cfg)
    moe.moe_finalize(cfg, y, perm, w, s, out, ws)
    assert moe.moe_read_device_status(ws) == 0
    ref = oracle.finalize(oracle.to_f64(y.cpu()), perm.cpu().numpy(), w.cpu().double().numpy(),
                          None if s is None else oracle.to_f64(s.cpu()))
    got = out.cpu().double().numpy()
    # fp32 accumulation then one bf16 rounding: within one bf16 ulp of the exact sum
    assert (np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-5).all()


@pytest.mark.parametrize("case,layout", [("gemma4_T256", "kn"), ("qwen35_T64", "kn"), ("fp8_small_T300", "kn"),
                                         ("fp8_small_T300", "nk"), ("fp8_small_geglu_T77", "nk")])
def test_stage_calls_match_moe_layer(case, layout):
    """The four stage calls in a row -- moe_route, moe_permute, moe_grouped_ffn
    with the shared expert, moe_finalize -- give the same output as moe_layer,
    bit for bit, and meet the layer bar against the oracle."""
    shape = LAYER_CASES[case]
    inp = workloads.make_inputs(shape, seed=5, device="cuda")
    layer = run_layer(shape, inp, layout)["out"]
    cfg = moe.config_from_shape(shape, layout)
    ws = moe.alloc_workspace(cfg)
    T, E, k, D, I, Is, R = shape.T, shape.E, shape.k, shape.D, shape.I, shape.I_shared, shape.R
    adt = workloads.torch_dtype(shape.act_dtype)
    dev = "cuda"
    logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    moe.moe_route(cfg, inp["x"], inp["Wg"], inp["logit_bias"], logits, ids, w, ws)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sorted_rows = torch.empty(R, dtype=torch.int32, device=dev)
    dest = torch.empty(R, dtype=torch.int32, device=dev)
    x_perm = torch.empty((R, D), dtype=adt, device=dev)
    moe.moe_permute(cfg, ids, inp["x"], counts, offsets, sorted_rows, dest, x_perm, ws)
    fp8 = shape.w_dtype == "fp8_e4m3"
    hdt = torch.bfloat16 if layout == "nk" else torch.float32  # fp8 layers' h
    h = (torch.empty((R, I), dtype=hdt, device=dev) if fp8
         else torch.empty((2, R, I), dtype=torch.bfloat16, device=dev))
    h_s = (torch.empty((T, Is), dtype=hdt, device=dev) if fp8
           else torch.empty((2, T, Is), dtype=torch.bfloat16, device=dev))
    ydt = torch.bfloat16 if fp8 else torch.float32  # fp8 layers: bf16 expert and shared rows
    y = torch.empty((R, D), dtype=ydt, device=dev)
    s_out = torch.empty((T, D), dtype=ydt, device=dev)
    W = packed_weights(inp, layout)
    moe.moe_grouped_ffn(cfg, x_perm, offsets, W["W13"], inp["s13"], W["W2"], inp["s2"], h, y,
                        inp["x"], W["W13s"], inp["s13s"], W["W2s"], inp["s2s"], h_s, s_out, ws)
    out = torch.empty((T, D), dtype=adt, device=dev)
    moe.moe_finalize(cfg, y, dest, w, s_out, out, ws)
    assert moe.moe_read_device_status(ws) == 0
    assert torch.equal(out.cpu(), layer), "stage calls and moe_layer differ"
    ref = oracle.moe_layer(_cpu(inp), k, shape.act, shape.renormalize)
    ties = oracle.near_tie_tokens(ref["logits"], k)
    assert ties.sum() <= max_near_ties(T)
    keep = ~ties
    err = np.abs(out.cpu().double().numpy() - ref["out"])[keep]
    assert err.max() <= tol_factor(shape) * rms(ref["out"])


def test_layer_parity_max_k():
    """k = 16 (the largest top-k the interface takes) on 32 experts."""
    check_layer(workloads.MoEShape("maxk", 100, 256, 32, 16, 128, I_shared=64))


def test_layer_parity_one_hot_expert():
    """A logit bias that sends every token to expert 0 (its group holds all T
    rows, several full tiles) while the other choices stay spread."""
    shape = workloads.MoEShape("hot", 700, 512, 64, 4, 256)
    inp = workloads.make_inputs(shape, seed=9, device="cuda")
    bias = torch.zeros(shape.E, dtype=torch.float32, device="cuda")
    bias[0] = 50.0
    inp["logit_bias"] = bias
    g = run_layer(shape, inp)
    assert int(g["counts"][0]) == shape.T
    cinp = _cpu(inp)
    ref = oracle.moe_layer(cinp, shape.k, shape.act, shape.renormalize)
    # routing of the GPU's own ids, bit-exact whatever the near ties
    r = oracle.init_routing(g["ids"].numpy(), shape.E)
    for name in ("counts", "offsets", "sorted_rows", "dest"):
        assert np.array_equal(g[name].numpy(), r[name]), f"{name} differs"
    ties = oracle.near_tie_tokens(ref["logits"], shape.k)
    assert ties.sum() <= max_near_ties(shape.T)
    keep = ~ties
    err = np.abs(g["out"].double().numpy() - ref["out"])[keep]
    assert err.max() <= tol_factor(shape) * rms(ref["out"])


@pytest.mark.parametrize("case,layout", [("gemma4_T8_decode", "kn"), ("qwen3_T512", "kn"),
                                         ("fp8_small_T300", "nk")])
def test_moe_layer_captures_into_a_cuda_graph(case, layout):
    """moe_layer enqueues only kernels, event records and waits (no host
    synchronisation, no allocation), so a stream capture of it replays to the
    eager call's output bit for bit, shared-expert side stream included."""
    shape = LAYER_CASES[case]
    inp = workloads.make_inputs(shape, seed=13, device="cuda")
    cfg = moe.config_from_shape(shape, layout)
    W = packed_weights(inp, layout)
    ws = moe.alloc_workspace(cfg)
    out = torch.empty((shape.T, shape.D), dtype=workloads.torch_dtype(shape.act_dtype), device="cuda")
    s = torch.cuda.Stream()
    args = (cfg, inp["x"], inp["Wg"], inp["logit_bias"], W["W13"], inp["s13"], W["W2"], inp["s2"],
            W["W13s"], inp["s13s"], W["W2s"], inp["s2s"], out, ws)
    with torch.cuda.stream(s):
        moe.moe_layer(*args, stream=s)  # first call: per-device one-time set-up outside the capture
    torch.cuda.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.moe_layer(*args, stream=s)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert moe.moe_read_device_status(ws) == 0


@pytest.mark.parametrize("T,k,D,shared", [(513, 8, 2048, True), (3, 1, 272, False)])
def test_finalize_parity_bf16_rows(T, k, D, shared):
    """fp8-weight layers hand finalize bf16 expert and shared rows."""
    gen = torch.Generator(device="cuda").manual_seed(T + 3 * k)
    R = T * k
    y = torch.randn((R, D), generator=gen, device="cuda").to(torch.bfloat16)
    perm = torch.randperm(R, generator=gen, device="cuda").to(torch.int32)
    w = torch.rand((T, k), generator=gen, device="cuda")
    w = w / w.sum(1, keepdim=True)
    s = torch.randn((T, D), generator=gen, device="cuda").to(torch.bfloat16) if shared else None
    out = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    cfg = moe.make_config(T, D, 16, k, 64, w_dtype="fp8_e4m3_nk")
    ws = _ws_for(cfg)
    moe.moe_finalize(cfg, y, perm, w, s, out, ws)
    assert moe.moe_read_device_status(ws) == 0
    ref = oracle.finalize(oracle.to_f64(y.cpu()), perm.cpu().numpy(), w.cpu().double().numpy(),
                          None if s is None else oracle.to_f64(s.cpu()))
    got = out.cpu().double().numpy()
    assert (np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-5).all()
