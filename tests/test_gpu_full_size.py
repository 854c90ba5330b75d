"""Every configured workload at its full size, in the configuration bench.py
times (default kernel options; fp8 workloads in both weight layouts),
through the C ABI.

The oracle cannot run a whole full-size layer in test time, so each case
checks (1) what holds at any size for every token -- top-k ids bit-exact
and weights within 1e-6 against the oracle's top-k of the GPU's own fp32
logits, the stable counting sort bit-exact against the oracle's
init_routing of the GPU's ids, dest the inverse of sorted_rows -- and (2)
the layer output of a seeded sample of tokens against the fp64 oracle run on
those tokens alone (rows are independent, so out[tokens] of the batch is the
layer applied to x[tokens]), with the same bar as the small-size parity
tests: max |err| <= 2e-2 (fp8: 6e-2) * RMS of the sampled reference, tokens
whose k-th and (k+1)-th oracle logits lie within 1e-4 left out.
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_gating_gb300 as moe
import oracle
import workloads
from tests._lib import ensure_library, max_near_ties, rms, tol_factor

pytestmark = pytest.mark.gpu

# sampled tokens per workload (the first and last token are always added).
# The oracle's cost is dominated by its fp64 copy of each expert a sampled
# token reaches (Ling: 268 MB per expert for W13), so once most experts are
# hit more tokens cost little: the prefill layers take a few hundred.
SAMPLE = {"ling_prefill": 256, "qwen35_prefill": 256, "gemma4_prefill": 128, "ling_decode": 64}
WORKLOADS = sorted(n for n in workloads.CONFIGS if n not in ("toy", "qwen3_prefill"))
# fp8 workloads run in both weight layouts (bench.py times the K-contiguous one)
CASES = [(n, "kn") for n in WORKLOADS] + [(n, "nk") for n in WORKLOADS
                                          if workloads.CONFIGS[n].w_dtype == "fp8_e4m3"]


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return ensure_library()


@pytest.mark.parametrize("name,layout", CASES)
def test_full_size_workload(name, layout):
    shape = workloads.CONFIGS[name]
    T, E, k, R = shape.T, shape.E, shape.k, shape.R
    inp = workloads.make_inputs(shape, seed=11, device="cuda")
    cfg = moe.config_from_shape(shape, layout)
    ws = moe.alloc_workspace(cfg)
    out = torch.empty((T, shape.D), dtype=workloads.torch_dtype(shape.act_dtype), device="cuda")
    W = {n: inp[n] for n in ("W13", "W2", "W13s", "W2s")}
    if layout == "nk":
        W = {n: (None if v is None else moe.pack_weights_nk(v)) for n, v in W.items()}
    moe.moe_layer(cfg, inp["x"], inp["Wg"], inp["logit_bias"], W["W13"], inp["s13"], W["W2"],
                  inp["s2"], W["W13s"], inp["s13s"], W["W2s"], inp["s2s"], out, ws)
    del W
    assert moe.moe_read_device_status(ws) == 0

    view = lambda slot, shp, dt: moe.workspace_view(ws, cfg, slot, shp, dt).cpu()  # noqa: E731
    logits = view("logits", (T, E), torch.float32).double().numpy()
    ids = view("topk_ids", (T, k), torch.int32).numpy()
    w = view("topk_w", (T, k), torch.float32).double().numpy()
    assert np.isfinite(logits).all()

    # (1) routing for every token, given the GPU's logits
    ids_o, w_o = oracle.topk_softmax(logits, k, shape.renormalize)
    assert np.array_equal(ids, ids_o)
    assert np.max(np.abs(w - w_o)) <= 1e-6
    r = oracle.init_routing(ids, E)
    assert np.array_equal(view("counts", (E,), torch.int32).numpy(), r["counts"])
    assert np.array_equal(view("offsets", (E + 1,), torch.int32).numpy(), r["offsets"])
    sorted_rows = view("sorted_rows", (R,), torch.int32).numpy()
    dest = view("dest", (R,), torch.int32).numpy()
    assert np.array_equal(sorted_rows, r["sorted_rows"])
    assert np.array_equal(dest, r["dest"])
    assert np.array_equal(sorted_rows[dest], np.arange(R))

    # (2) sampled tokens against the oracle
    gen = np.random.default_rng(T + E)
    n = min(T, SAMPLE.get(name, 64))
    tokens = np.unique(np.concatenate([[0, T - 1], gen.choice(T, n, replace=False)]))[: n + 2]
    sub = dict(inp)
    sub["x"] = inp["x"].cpu()[torch.from_numpy(tokens)]
    ref = oracle.moe_layer(sub, k, shape.act, shape.renormalize)
    ties = oracle.near_tie_tokens(ref["logits"], k)
    assert ties.sum() <= max_near_ties(len(tokens))
    keep = ~ties
    # every token of the batch: how many have a near tie in the GPU's logits
    # (the oracle's logits exist for the sample only); at most 1 %
    all_ties = oracle.near_tie_tokens(logits, k)
    print(f"{name}/{layout}: {int(all_ties.sum())} of {T} tokens with a near tie")
    assert all_ties.sum() <= max_near_ties(T)
    got = out[torch.from_numpy(tokens).cuda()].double().cpu().numpy()
    assert (np.array_equal(ids[tokens][keep], ref["ids"][keep]))
    assert keep.any()
    err = np.abs(got - ref["out"])[keep]
    scale = rms(ref["out"][keep])
    assert err.max() <= tol_factor(shape) * scale, \
        f"{name}: max|err| {err.max():.3e} > {tol_factor(shape)} * RMS {scale:.3e}"
