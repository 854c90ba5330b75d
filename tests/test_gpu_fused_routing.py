"""The fused routing chain (MOE_OPT_FUSED_ROUTING) against the oracle.

The router projection fused with the top-k softmax (one cluster launch per
128 tokens), through moe_route.  The fused kernel splits the fp32 sum over D
into up to 4 consecutive slices on the CTAs of a cluster and, when E > 256,
the experts into two halves; the CTA that finishes a token adds the partial
rows in slice order.  Routing is checked bit-exact against the oracle's top-k
of the GPU's own logits, the logits against the fp64 projection, with both
settings of the option.  The shapes cover one to four slices, two expert
halves (E = 320 and 512, the second half partly past E), expert counts that
leave the last 64-expert box partly or wholly past E (96, 160, 200), token
counts that leave the last 128-token tile short, and D that is not a multiple
of 64.

init_routing as one cluster of 8 CTAs (histogram, scan and stable scatter,
the histograms exchanged through distributed shared memory), through
moe_permute: counts, offsets, sorted_rows, dest and the permuted rows
bit-exact against the oracle's counting sort, with both settings of the
option, on uniform, skewed, one-expert and half-empty routings, E up to 512,
up to the 65536 expanded rows the cluster sort takes, and a batch with ids out
of range (those rows get dest = -1 and stay out of the sort).
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_gating_gb300 as moe
import oracle
from tests._lib import ensure_library, rms

pytestmark = pytest.mark.gpu

SHAPES = [
    # T, E, k, renorm, bias, D
    (4096, 128, 8, 1, False, 2048),   # Qwen3-MoE prefill shape: 4 slices
    (2048, 128, 8, 1, False, 2816),   # Gemma-4 prefill shape: 4 slices, D % 64 != 0
    (8192, 512, 10, 1, True, 4096),   # Qwen3.5 prefill shape: two expert halves
    (65, 128, 8, 1, True, 2048),      # one short tile, 4 slices
    (300, 96, 6, 0, False, 1000),     # last box partly past E; 3 tiles
    (1000, 160, 8, 1, True, 136),     # a box wholly past E; 3 k-blocks, one slice
    (777, 200, 16, 1, False, 520),    # k = 16
    (129, 320, 8, 0, True, 4096),     # halves of 256 + 64 experts
    (200, 512, 16, 1, False, 8192),   # 8192-wide rows
    (2047, 256, 8, 1, True, 256),
]


def _route(T, E, k, renorm, bias, D):
    gen = torch.Generator(device="cuda").manual_seed(T * 7 + E + k + D)
    x = torch.randn((T, D), generator=gen, device="cuda").to(torch.bfloat16)
    Wg = (0.05 * torch.randn((D, E), generator=gen, device="cuda")).to(torch.bfloat16)
    Wg[:, 5] = Wg[:, 3]  # exact ties: the lower index must win
    Wg[:, 63] = Wg[:, 62]
    Wg[:, E - 1] = Wg[:, 10]
    tz = min(7, T - 1)
    x[tz] = 0  # every logit equal (zero, plus the bias)
    b = (0.01 * torch.randn((E,), generator=gen, device="cuda")) if bias else None
    if bias:
        b[5] = b[3]
        b[63] = b[62]
        b[E - 1] = b[10]
    cfg = moe.make_config(T, D, E, k, 64, renormalize=renorm)
    ws = moe.alloc_workspace(cfg)
    L = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((T, k), -5, dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, x, Wg, b, L, ids, w, ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    return x, Wg, b, L, ids, w, tz


@pytest.mark.parametrize("fused", [2, 0])  # 2: the fused kernel wherever the shape allows
@pytest.mark.parametrize("T,E,k,renorm,bias,D", SHAPES)
def test_router_topk_against_oracle(T, E, k, renorm, bias, D, fused):
    ensure_library()
    old = moe.moe_set_option(moe.MOE_OPT_FUSED_ROUTING, fused)
    try:
        x, Wg, b, L, ids, w, tz = _route(T, E, k, renorm, bias, D)
    finally:
        moe.moe_set_option(moe.MOE_OPT_FUSED_ROUTING, old)
    L_gpu = L.cpu().double().numpy()
    assert np.isfinite(L_gpu).all()
    ids_o, w_o = oracle.topk_softmax(L_gpu, k, renorm)
    assert np.array_equal(ids.cpu().numpy(), ids_o)
    assert np.max(np.abs(w.cpu().double().numpy() - w_o)) <= 1e-6
    L_ref = oracle.router_logits(x.cpu(), Wg.cpu(), b.cpu() if bias else None)
    assert np.max(np.abs(L_gpu - L_ref)) <= 1e-3 * max(1.0, rms(L_ref))
    # duplicated columns give bit-identical logits
    assert np.array_equal(L_gpu[:, 5], L_gpu[:, 3]) and np.array_equal(L_gpu[:, E - 1], L_gpu[:, 10])
    if not bias:
        assert np.array_equal(ids[tz].cpu().numpy(), np.arange(k))


SORT_CASES = [
    # T, E, k, pattern
    (1025, 8, 8, "uniform"),       # 8200 expanded rows: just past the one-launch sort
    (4096, 128, 8, "uniform"),     # Qwen3-MoE prefill
    (6000, 512, 10, "skew"),       # 60000 rows, 512 experts
    (8192, 256, 8, "uniform"),     # 65536 rows: the largest batch the cluster sort takes
    (16384, 256, 8, "uniform"),    # Ling-style prefill: two-kernel sort either way
    (3001, 64, 6, "one_expert"),   # every token's first choice is expert 0
    (2500, 64, 6, "empty_half"),   # experts 32.. never chosen
    (5000, 100, 4, "bad_ids"),     # a few ids out of range
]


def _ids(T, E, k, pattern, gen):
    if pattern == "skew":
        p = 1.0 / torch.arange(1, E + 1, dtype=torch.float64) ** 1.2
        ids = torch.multinomial(p.expand(T, E).contiguous(), k, replacement=False, generator=gen)
    elif pattern == "one_expert":
        ids = torch.argsort(torch.rand((T, E - 1), generator=gen), dim=1)[:, :k] + 1
        ids[:, 0] = 0
    elif pattern == "empty_half":
        ids = torch.argsort(torch.rand((T, E // 2), generator=gen), dim=1)[:, :k]
    else:
        ids = torch.argsort(torch.rand((T, E), generator=gen), dim=1)[:, :k]
    ids = ids.to(torch.int32).contiguous()
    if pattern == "bad_ids":
        flat = ids.view(-1)
        flat[17] = E
        flat[4000] = -1
        flat[-1] = E + 7
    return ids


@pytest.mark.parametrize("fused", [1, 0])
@pytest.mark.parametrize("T,E,k,pattern", SORT_CASES)
def test_cluster_sort_against_oracle(T, E, k, pattern, fused):
    ensure_library()
    gen = torch.Generator().manual_seed(T + E + k)
    ids = _ids(T, E, k, pattern, gen)
    D = 72
    x = torch.randn((T, D), generator=gen).to(torch.bfloat16)
    cfg = moe.make_config(T, D, E, k, 64)
    ws = moe.alloc_workspace(cfg)
    R = T * k
    counts = torch.full((E,), -3, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -3, dtype=torch.int32, device="cuda")
    sorted_rows = torch.full((R,), -3, dtype=torch.int32, device="cuda")
    dest = torch.full((R,), -3, dtype=torch.int32, device="cuda")
    x_perm = torch.zeros((R, D), dtype=torch.bfloat16, device="cuda")
    old = moe.moe_set_option(moe.MOE_OPT_FUSED_ROUTING, fused)
    try:
        moe.moe_permute(cfg, ids.cuda(), x.cuda(), counts, offsets, sorted_rows, dest, x_perm, ws)
        torch.cuda.synchronize()
    finally:
        moe.moe_set_option(moe.MOE_OPT_FUSED_ROUTING, old)
    status = moe.moe_read_device_status(ws)
    flat = ids.view(-1).numpy().astype(np.int64)
    valid = (flat >= 0) & (flat < E)
    if pattern == "bad_ids":
        # the bad ids are flagged (the gather also flags the unused positions
        # past offsets[E], whose sorted_rows entries were never written)
        assert status & moe.MOE_DEV_BAD_EXPERT_ID
        # the oracle's stable counting sort of the valid rows alone
        o = oracle.init_routing(flat[valid], E)
        rows = np.arange(R)[valid]
        order = rows[o["sorted_rows"]]
        d_o = np.full(R, -1, dtype=np.int64)
        d_o[order] = np.arange(order.size)
        n = order.size
        assert np.array_equal(counts.cpu().numpy(), o["counts"])
        assert np.array_equal(offsets.cpu().numpy(), o["offsets"])
        assert np.array_equal(sorted_rows.cpu().numpy()[:n], order)
        assert np.array_equal(dest.cpu().numpy(), d_o)
        assert torch.equal(x_perm[:n].cpu(), x[torch.from_numpy(order // k)])
        return
    assert status == 0
    o = oracle.init_routing(ids.numpy(), E)
    assert np.array_equal(counts.cpu().numpy(), o["counts"])
    assert np.array_equal(offsets.cpu().numpy(), o["offsets"])
    assert np.array_equal(sorted_rows.cpu().numpy(), o["sorted_rows"])
    assert np.array_equal(dest.cpu().numpy(), o["dest"])
    assert torch.equal(x_perm.cpu(), x[torch.from_numpy(o["sorted_rows"] // k)])


LAYER_CASES = [
    # T, E, k, D: the fused router's CTAs (chunks) and rows per chunk in the comment
    (4096, 128, 8, 2048),   # Qwen3-MoE prefill shape: 128 chunks of 256 rows
    (1100, 64, 8, 512),     # 18 chunks of 512 rows, the last one short
    (2100, 320, 8, 1024),   # two expert halves: 68 chunks of 256 rows
    (700, 96, 16, 256),     # one CTA per tile: 6 chunks of 2048 rows
    (1040, 200, 16, 136),   # k = 16 (moe_layer's largest): 9 chunks of 2048 rows, E % 32 != 0
    (9000, 512, 8, 512),    # 72000 rows (past the 8-CTA cluster sort): 142 chunks
]


def _layer_routing(T, E, k, D, mode):
    gen = torch.Generator(device="cuda").manual_seed(T + 3 * E + k + D)
    I = 64
    x = torch.randn((T, D), generator=gen, device="cuda").to(torch.bfloat16)
    Wg = (0.05 * torch.randn((D, E), generator=gen, device="cuda")).to(torch.bfloat16)
    W13 = (0.02 * torch.randn((E, D, 2 * I), generator=gen, device="cuda")).to(torch.bfloat16)
    W2 = (0.02 * torch.randn((E, I, D), generator=gen, device="cuda")).to(torch.bfloat16)
    cfg = moe.make_config(T, D, E, k, I)
    ws = moe.alloc_workspace(cfg)
    out = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    old = moe.moe_set_option(moe.MOE_OPT_FUSED_ROUTING, mode)
    try:
        moe.moe_layer(cfg, x, Wg, None, W13, None, W2, None, None, None, None, None, out, ws)
        torch.cuda.synchronize()
    finally:
        moe.moe_set_option(moe.MOE_OPT_FUSED_ROUTING, old)
    R = T * k
    view = lambda slot, n: moe.workspace_view(ws, cfg, slot, (n,), torch.int32).cpu().numpy()  # noqa: E731
    got = {"ids": view("topk_ids", R), "counts": view("counts", E), "offsets": view("offsets", E + 1),
           "sorted_rows": view("sorted_rows", R), "dest": view("dest", R)}
    return got, out.cpu(), moe.moe_read_device_status(ws)


@pytest.mark.parametrize("T,E,k,D", LAYER_CASES)
def test_layer_sorts_by_router_histograms(T, E, k, D):
    """moe_layer after the fused router: init_routing from the router's
    per-CTA histograms (MOE_OPT_FUSED_ROUTING 2: the fused router wherever the
    shape allows) against the oracle's stable counting sort of the GPU's own
    ids, bit-exact; the layer output bit-identical to the run that sorts with
    the other init_routing kernels (option 3: same router, same permutation)."""
    ensure_library()
    got, out, status = _layer_routing(T, E, k, D, 2)
    assert status == 0
    ids = got["ids"].reshape(T, k)
    assert ((ids >= 0) & (ids < E)).all()
    o = oracle.init_routing(ids, E)
    for key in ("counts", "offsets", "sorted_rows", "dest"):
        assert np.array_equal(got[key], o[key]), key
    got3, out3, status3 = _layer_routing(T, E, k, D, 3)
    assert status3 == 0
    assert np.array_equal(got3["ids"], got["ids"])
    for key in ("counts", "offsets", "sorted_rows", "dest"):
        assert np.array_equal(got3[key], got[key]), key
    assert torch.equal(out3, out)
