"""Checks that pin the CPU oracle to facts outside itself.

Each ``check_*`` function takes the oracle module and raises AssertionError
when the oracle disagrees with a brute-force computation, a textbook or
library routine, an invariant of the method or a value printed on the source
pages.  The pin tests call them on the real oracle; the mutation tests plant
plausible mistakes in the oracle and expect them to fail.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import scipy.special
import torch
import torch.nn.functional as F

import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _brute_topk(L, k):
    """Python sort with key (-logit, index): the lower index wins a tie."""
    T, E = L.shape
    ids = np.zeros((T, k), dtype=np.int64)
    w = np.zeros((T, k))
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-L[t, e], e))[:k]
        ids[t] = order
        m = L[t, order[0]]
        z = [math.exp(L[t, e] - m) for e in order]
        w[t] = [v / sum(z) for v in z]
    return ids, w


def check_topk_brute_force(o):
    rng = _rng(1)
    for E, k in [(7, 3), (8, 2), (16, 5), (5, 5), (9, 1)]:
        # small integer logits force many exact ties
        L = rng.integers(-3, 4, size=(60, E)).astype(np.float64) * 0.5
        ids, w = o.topk_softmax(L, k)
        bids, bw = _brute_topk(L, k)
        assert np.array_equal(ids, bids), "top-k ids differ from brute force"
        assert np.allclose(w, bw, rtol=0, atol=1e-15), "top-k weights differ from brute force"
        L2 = rng.standard_normal((40, E))
        ids, w = o.topk_softmax(L2, k)
        bids, bw = _brute_topk(L2, k)
        assert np.array_equal(ids, bids)
        assert np.allclose(w, bw, rtol=0, atol=1e-15)


def check_topk_all_equal(o):
    L = np.zeros((4, 12))
    ids, w = o.topk_softmax(L, 5)
    assert np.array_equal(ids, np.tile(np.arange(5), (4, 1))), "all-equal logits must give ids 0..k-1"
    assert np.allclose(w, 0.2, rtol=0, atol=1e-15)


def check_topk_full_softmax(o):
    """k = E reduces renormalised top-k gating to the textbook softmax."""
    rng = _rng(2)
    L = rng.standard_normal((30, 9)) * 3
    ids, w = o.topk_softmax(L, 9)
    p = scipy.special.softmax(L, axis=1)
    assert np.allclose(np.take_along_axis(p, ids.astype(np.int64), 1), w, rtol=0, atol=1e-15)
    # without renormalisation the weights are the full softmax probabilities
    ids3, w3 = o.topk_softmax(L, 3, renormalize=False)
    assert np.allclose(np.take_along_axis(p, ids3.astype(np.int64), 1), w3, rtol=0, atol=1e-15)


def check_topk_weight_invariants(o):
    rng = _rng(3)
    L = rng.standard_normal((200, 64)) * 2
    for k in (1, 2, 8, 10):
        ids, w = o.topk_softmax(L, k)
        assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-14), "renormalised weights must sum to 1"
        assert (np.diff(w, axis=1) <= 1e-15).all(), "weights must be non-increasing in slot order"
        assert (w > 0).all()
        sel = np.take_along_axis(L, ids.astype(np.int64), 1)
        assert (np.diff(sel, axis=1) <= 0).all(), "ids must be ordered by descending logit"


def _brute_near_ties(L, k, eps):
    """Per token: sort its logits with Python's sorted(), descending, and
    compare the k-th and (k+1)-th values; no (k+1)-th value (k = E) means no
    near tie."""
    T, E = L.shape
    out = []
    for t in range(T):
        v = sorted((float(a) for a in L[t]), reverse=True)
        out.append(k < E and (v[k - 1] - v[k]) < eps)
    return np.array(out, dtype=bool)


def check_near_ties(o):
    """Which tokens the parity tests leave out: those whose k-th and (k+1)-th
    largest logits differ by less than 1e-4 (strictly), checked on hand-built
    gaps at the boundary and against a brute-force sort on random rows."""
    eps = 1e-4
    below, above = np.nextafter(eps, 0.0), np.nextafter(eps, 1.0)
    # k = 3 of E = 6; the third and fourth logits are `gap` and 0.0, so the
    # gap is exactly the double `gap`; the others are far away
    def row(gap, perm=None):
        r = np.array([5.0, 4.0, gap, 0.0, -3.0, -4.0])
        return r if perm is None else r[perm]
    perm = np.array([3, 5, 0, 2, 4, 1])  # the same values in another order
    L = np.stack([row(eps), row(below), row(above), row(0.0), row(eps, perm), row(below, perm),
                  row(2e-4), row(0.5e-4)])
    want = np.array([False, True, False, True, False, True, False, True])
    got = np.asarray(o.near_tie_tokens(L, 3), dtype=bool)
    assert got.shape == (len(L),)
    assert np.array_equal(got, want), f"near-tie boundary cases: {got} != {want}"
    # ties inside the top k, or below the (k+1)-th, are not near ties
    L2 = np.array([[5.0, 5.0, 3.0, 1.0, 1.0], [2.0, 9.0, 9.0, 9.0, -1.0], [7.0, 1.0, 3.0, 5.0, 1.0]])
    assert np.array_equal(np.asarray(o.near_tie_tokens(L2, 2), dtype=bool), [False, True, False])
    # k = E: there is no (k+1)-th logit, so no token is left out
    assert not np.asarray(o.near_tie_tokens(np.zeros((4, 5)), 5), dtype=bool).any()
    # k = 1: the gap between the largest and the second largest
    L3 = np.array([[1.0, 1.0 - 0.5e-4, 0.0], [1.0, 0.0, 0.5], [0.25, 0.25, 0.25]])
    assert np.array_equal(np.asarray(o.near_tie_tokens(L3, 1), dtype=bool), [True, False, True])
    # random rows, some with values on a grid of eps / 2 so that gaps land on,
    # below and above eps, against the brute-force sort
    rng = _rng(13)
    for E, k in [(8, 2), (16, 5), (7, 6), (9, 1), (12, 12)]:
        R1 = rng.standard_normal((300, E))
        R2 = rng.integers(-6, 7, size=(300, E)) * (eps / 2)
        R3 = rng.integers(-3, 4, size=(300, E)) * eps
        for R in (R1, R2, R3):
            got = np.asarray(o.near_tie_tokens(R, k), dtype=bool)
            assert np.array_equal(got, _brute_near_ties(R, k, eps)), f"near ties differ (E={E}, k={k})"


def check_routing_brute_force(o):
    rng = _rng(4)
    for T, E, k in [(50, 6, 2), (17, 33, 4), (1, 4, 1), (64, 8, 8)]:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        r = o.init_routing(ids, E)
        flat = ids.reshape(-1)
        R = T * k
        want = sorted(range(R), key=lambda q: (flat[q], q))
        assert list(r["sorted_rows"]) == want, "sorted_rows must be the stable sort by expert"
        cnt = [int((flat == e).sum()) for e in range(E)]
        assert list(r["counts"]) == cnt
        assert r["offsets"][0] == 0 and r["offsets"][-1] == R
        assert all(r["offsets"][e + 1] - r["offsets"][e] == cnt[e] for e in range(E))
        assert np.array_equal(r["dest"][r["sorted_rows"]], np.arange(R)), "dest must invert sorted_rows"
        for e in range(E):
            seg = r["sorted_rows"][r["offsets"][e]:r["offsets"][e + 1]]
            assert (flat[seg] == e).all()


def check_permute_round_trip(o):
    rng = _rng(5)
    T, D, E, k = 40, 12, 7, 3
    x = rng.standard_normal((T, D))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    r = o.init_routing(ids, E)
    xp = o.permute(x, r["sorted_rows"], k)
    assert xp.shape == (T * k, D)
    for t in range(T):
        for j in range(k):
            assert np.array_equal(xp[r["dest"][t * k + j]], x[t]), "un-permute(permute(x)) must be x"


def check_swiglu_golden(o):
    g = json.load(open(os.path.join(GOLDEN, "swiglu_chunk_example.json")))
    for case in g["cases"]:
        gu = np.array(case["gate_up"], dtype=np.float64)[None, :]
        I = gu.shape[1] // 2
        # an identity down projection exposes h itself
        W13 = np.eye(2 * I)
        W2 = np.eye(I)
        h, y = o.expert_ffn(gu, W13, W2, o.ACT_SWIGLU)
        assert np.allclose(h[0], case["h"], rtol=0, atol=1e-15), f"swiglu chunk example {case}"
        assert np.allclose(y[0], case["h"], rtol=0, atol=1e-15)


def check_activations_library(o):
    g = np.linspace(-30, 30, 2001)
    tg = torch.from_numpy(g)
    assert np.allclose(o.activation(g, o.ACT_SWIGLU), F.silu(tg).numpy(), rtol=1e-14, atol=1e-300)
    # 1 + tanh(.) cancels for very negative g: both sides are exact to ~1e-16 absolute there
    assert np.allclose(o.activation(g, o.ACT_GEGLU_TANH), F.gelu(tg, approximate="tanh").numpy(),
                       rtol=1e-13, atol=1e-14)


def _dense_mlp_torch(x, W13, W2, act):
    """Dense gated MLP with torch fp64: chunk(x W13, 2) -> act(first) * second -> W2."""
    tx, t13, t2 = (torch.from_numpy(np.asarray(a, np.float64)) for a in (x, W13, W2))
    gate, up = torch.chunk(tx @ t13, 2, dim=-1)
    a = F.silu(gate) if act == "swiglu" else F.gelu(gate, approximate="tanh")
    return ((a * up) @ t2).numpy()


def check_single_expert_is_dense_mlp(o):
    """E = 1, k = 1: the layer reduces to one dense gated MLP (weight 1)."""
    rng = _rng(6)
    T, D, I = 23, 16, 10
    for act in (o.ACT_SWIGLU, o.ACT_GEGLU_TANH):
        x = rng.standard_normal((T, D))
        W13 = rng.standard_normal((1, D, 2 * I)) * 0.3
        W2 = rng.standard_normal((1, I, D)) * 0.3
        inp = {"x": x, "Wg": rng.standard_normal((D, 1)), "W13": W13, "W2": W2}
        out = o.moe_layer(inp, 1, act)["out"]
        ref = _dense_mlp_torch(x, W13[0], W2[0], act)
        assert np.allclose(out, ref, rtol=1e-12, atol=1e-12), "E=1,k=1 must equal the dense MLP"


def _tiny_layer(rng, T=19, D=12, E=6, k=3, I=5, Is=4, fp8=False):
    x = rng.standard_normal((T, D))
    inp = {
        "x": x,
        "Wg": rng.standard_normal((D, E)) * 0.5,
        "logit_bias": rng.standard_normal(E) * 0.1,
        "W13": rng.standard_normal((E, D, 2 * I)) * 0.3,
        "W2": rng.standard_normal((E, I, D)) * 0.3,
    }
    if Is:
        inp["W13s"] = rng.standard_normal((D, 2 * Is)) * 0.3
        inp["W2s"] = rng.standard_normal((Is, D)) * 0.3
    if fp8:
        inp["s13"] = rng.uniform(0.5, 2.0, (E, 2 * I))
        inp["s2"] = rng.uniform(0.5, 2.0, (E, D))
        if Is:
            inp["s13s"] = rng.uniform(0.5, 2.0, 2 * Is)
            inp["s2s"] = rng.uniform(0.5, 2.0, D)
    return inp


def _brute_dense_layer(inp, k, act):
    """Every expert on every token, then masked by the brute-force gates."""
    x = np.asarray(inp["x"], np.float64)
    E = inp["W13"].shape[0]
    L = x @ inp["Wg"] + inp.get("logit_bias", 0.0)
    ids, w = _brute_topk(L, k)
    gates = np.zeros((x.shape[0], E))
    for t in range(x.shape[0]):
        for j in range(k):
            gates[t, ids[t, j]] = w[t, j]

    def w_eff(W, s):
        return W if s is None else W * np.asarray(s)[None, :]

    out = np.zeros_like(x)
    for e in range(E):
        W13 = w_eff(inp["W13"][e], None if inp.get("s13") is None else inp["s13"][e])
        W2 = w_eff(inp["W2"][e], None if inp.get("s2") is None else inp["s2"][e])
        out += gates[:, e:e + 1] * _dense_mlp_torch(x, W13, W2, act)
    if inp.get("W13s") is not None:
        out += _dense_mlp_torch(x, w_eff(inp["W13s"], inp.get("s13s")), w_eff(inp["W2s"], inp.get("s2s")), act)
    return out


def check_layer_vs_dense_then_mask(o):
    rng = _rng(7)
    for act in (o.ACT_SWIGLU, o.ACT_GEGLU_TANH):
        for fp8 in (False, True):
            for (E, k, Is) in [(6, 3, 4), (8, 1, 0), (5, 5, 3)]:
                inp = _tiny_layer(rng, E=E, k=k, Is=Is, fp8=fp8)
                out = o.moe_layer(inp, k, act)["out"]
                ref = _brute_dense_layer(inp, k, act)
                assert np.allclose(out, ref, rtol=1e-11, atol=1e-12), \
                    f"layer != dense-then-mask (act={act}, fp8={fp8}, E={E}, k={k})"


def check_identical_experts(o):
    """All experts equal + renormalised gates: out = FFN(x) + shared(x) whatever the routing."""
    rng = _rng(8)
    inp = _tiny_layer(rng, T=31, E=7, k=3)
    inp["W13"] = np.repeat(inp["W13"][:1], 7, axis=0)
    inp["W2"] = np.repeat(inp["W2"][:1], 7, axis=0)
    out = o.moe_layer(inp, 3, o.ACT_SWIGLU)["out"]
    ref = _dense_mlp_torch(inp["x"], inp["W13"][0], inp["W2"][0], "swiglu") + \
        _dense_mlp_torch(inp["x"], inp["W13s"], inp["W2s"], "swiglu")
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-12), "identical-experts invariant broken"


def check_shared_only(o):
    """Zero routed down projections leave exactly the shared expert's output."""
    rng = _rng(9)
    inp = _tiny_layer(rng)
    inp["W2"] = np.zeros_like(inp["W2"])
    out = o.moe_layer(inp, 3, o.ACT_SWIGLU)["out"]
    ref = _dense_mlp_torch(inp["x"], inp["W13s"], inp["W2s"], "swiglu")
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-13), "shared expert must be added ungated"


def check_fp8_scale_identity(o):
    """(sum_k x q) * s[n] equals sum_k x (q * s[n]) for per-column scales."""
    rng = _rng(10)
    w = torch.from_numpy(rng.standard_normal((64, 48)) * 0.02).float()
    q, s = workloads.quantize_fp8_per_column(w)
    qf, sf = o.to_f64(q), o.to_f64(s)
    x = rng.standard_normal((9, 64))
    a = o.scaled_projection(x, qf, sf)
    b = x @ (qf * sf[None, :])
    assert np.allclose(a, b, rtol=1e-12, atol=1e-15), "per-channel scale must apply to output columns"
    # and the dequantised weights approximate the fp32 weights to e4m3 precision
    assert np.max(np.abs(qf * sf[None, :] - w.double().numpy())) <= 2 ** -4 * np.max(np.abs(w.numpy()))


def check_subset_matches_full(o):
    rng = _rng(11)
    inp = _tiny_layer(rng, T=25)
    full = o.moe_layer(inp, 3, o.ACT_SWIGLU)["out"]
    tok = np.array([0, 7, 24, 3])
    sub = o.moe_layer_tokens(inp, tok, 3, o.ACT_SWIGLU)
    assert np.allclose(sub, full[tok], rtol=1e-13, atol=1e-14)


def check_counts_sum(o):
    rng = _rng(12)
    inp = _tiny_layer(rng, T=33, E=6, k=4)
    res = o.moe_layer(inp, 4, o.ACT_SWIGLU)
    assert res["counts"].sum() == 33 * 4, "per-expert counts must sum to T*k"


# ---------------------------------------------------------------- W8A8 forms
def _e4m3_table():
    """Every finite e4m3 (fn) value with its code, decoded from the bit
    fields: sign, 4 exponent bits (bias 7), 3 fraction bits; exponent field 0
    is subnormal (f / 8 * 2^-6); code 0x7f / 0xff is NaN."""
    vals = []
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        sgn = -1.0 if c & 0x80 else 1.0
        e, f = (c >> 3) & 0xF, c & 7
        mag = (f / 8.0) * 2.0 ** -6 if e == 0 else (1 + f / 8.0) * 2.0 ** (e - 7)
        vals.append((sgn * mag, c))
    return vals


def _brute_e4m3(v):
    """Nearest table value by exhaustive search; a tie goes to the even code
    (fraction LSB 0); beyond 448 saturates."""
    table = _e4m3_table()
    out = np.empty(len(v))
    for i, x in enumerate(v):
        if abs(x) >= 448.0:
            out[i] = math.copysign(448.0, x)
            continue
        best = min(table, key=lambda vc: (abs(vc[0] - x), vc[1] & 1, -abs(vc[0])))
        out[i] = best[0]
        if best[0] == 0.0:
            out[i] = math.copysign(0.0, x)
    return out


def _e4m3_probe_values(rng, n):
    """Random magnitudes over every binade (subnormals included), the exact
    midpoints between neighbouring e4m3 values (ties), the values themselves."""
    mags = sorted({abs(v) for v, _ in _e4m3_table()})
    mids = [(a + b) / 2 for a, b in zip(mags[:-1], mags[1:])]
    r = np.exp(rng.uniform(np.log(2.0 ** -11), np.log(448.0), n))
    v = np.concatenate([r, mids, mags, [0.0, 448.0]])
    sgn = rng.choice([-1.0, 1.0], v.size)
    return (v * sgn).astype(np.float32).astype(np.float64)


def check_e4m3_round(o):
    rng = _rng(14)
    v = _e4m3_probe_values(rng, 3000)
    got = o.e4m3_round(v)
    lib = torch.from_numpy(v).float().to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(got, lib), "e4m3 rounding differs from torch's float8_e4m3fn cast"
    idx = rng.choice(v.size, 600, replace=False)
    assert np.array_equal(got[idx], _brute_e4m3(v[idx])), "e4m3 rounding differs from the code table"
    # beyond the largest finite value: saturation
    assert np.array_equal(o.e4m3_round(np.array([448.5, -460.0, 1e6])), [448.0, -448.0, 448.0])


def check_bf16_round(o):
    rng = _rng(15)
    v = (rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))).astype(np.float32)
    # exact ties: bf16 values with the next bit set and nothing below
    t = (torch.from_numpy(v).to(torch.bfloat16).float().numpy().view(np.uint32) | np.uint32(0x8000))
    v = np.concatenate([v, t.view(np.float32)]).astype(np.float64)
    lib = torch.from_numpy(v).float().to(torch.bfloat16).double().numpy()
    assert np.array_equal(o.bf16_round(v), lib), "bf16 rounding differs from torch's bf16 cast"


def check_quantize_rows(o):
    rng = _rng(16)
    a = rng.standard_normal((50, 40)) * np.exp(rng.uniform(-6, 6, (50, 1)))
    a = torch.from_numpy(a).to(torch.bfloat16).double().numpy()  # bf16 activations
    a[3] = 0.0
    q, sc = o.quantize_rows_e4m3(a)
    assert q.shape == a.shape and sc.shape == (50,)
    amax = np.abs(a).max(axis=1).astype(np.float32)
    want_s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float64)
    assert np.array_equal(sc, want_s), "row scale = amax / 448 in fp32"
    assert sc[3] == 1.0 and not q[3].any()
    live = np.arange(50) != 3
    arg = np.abs(a).argmax(axis=1)
    assert np.array_equal(np.abs(q[np.arange(50), arg])[live], np.full(49, 448.0)), \
        "the largest element of a row maps to +-448"
    assert np.array_equal(q, _brute_e4m3((a.astype(np.float32) / sc.astype(np.float32)[:, None])
                                         .astype(np.float64).ravel()).reshape(a.shape))
    deq = o.dequantize_rows(q, sc)
    rel = np.abs(a) / sc[:, None]
    normal = rel >= 2.0 ** -6
    assert (np.abs(deq - a)[normal] <= 2.0 ** -4 * np.abs(a)[normal] * (1 + 1e-6)).all()
    assert (np.abs(deq - a)[~normal] <= 2.0 ** -10 * np.broadcast_to(sc[:, None], a.shape)[~normal]
            * (1 + 1e-6)).all()


def _brute_w8a8_dense_layer(inp, k, act):
    """Dense-then-mask W8A8: x and h quantised per row through the code table,
    every expert on every token, masked by the brute-force gates."""
    x = np.asarray(inp["x"], np.float64)
    E = inp["W13"].shape[0]
    L = x @ inp["Wg"] + inp.get("logit_bias", 0.0)
    ids, w = _brute_topk(L, k)

    def quant(a):
        out = np.empty_like(a)
        for r in range(a.shape[0]):
            amax = np.float32(np.max(np.abs(a[r])))
            sc = amax / np.float32(448.0) if amax > 0 else np.float32(1.0)
            qv = _brute_e4m3((a[r].astype(np.float32) / sc).astype(np.float64))
            out[r] = qv * np.float64(sc)
        return out

    def ffn(xq, W13, W2, s13, s2):
        W13 = W13 if s13 is None else W13 * np.asarray(s13)[None, :]
        W2 = W2 if s2 is None else W2 * np.asarray(s2)[None, :]
        gu = torch.from_numpy(xq) @ torch.from_numpy(W13)
        gate, up = torch.chunk(gu, 2, dim=-1)
        a = F.silu(gate) if act == "swiglu" else F.gelu(gate, approximate="tanh")
        h = (a * up).to(torch.bfloat16).double().numpy()
        return quant(h) @ W2

    xq = quant(x)
    out = np.zeros_like(x)
    for t in range(x.shape[0]):
        for j in range(k):
            e = ids[t, j]
            out[t] += w[t, j] * ffn(xq[t:t + 1], inp["W13"][e], inp["W2"][e],
                                    None if inp.get("s13") is None else inp["s13"][e],
                                    None if inp.get("s2") is None else inp["s2"][e])[0]
    if inp.get("W13s") is not None:
        out += ffn(xq, inp["W13s"], inp["W2s"], inp.get("s13s"), inp.get("s2s"))
    return out


def check_w8a8_layer(o):
    """The W8A8 layer against a dense-then-mask brute force with the
    activations quantised through the e4m3 code table; the router sees the
    unquantised x; the quantisation error is present and of e4m3 size."""
    rng = _rng(17)
    for act in (o.ACT_SWIGLU, o.ACT_GEGLU_TANH):
        for (E, k, Is) in [(6, 3, 4), (5, 2, 0)]:
            inp = _tiny_layer(rng, T=11, E=E, k=k, Is=Is, fp8=True)
            inp["x"] = torch.from_numpy(inp["x"]).to(torch.bfloat16).double().numpy()
            res = o.moe_layer(inp, k, act, act_quant=o.ACT_QUANT_E4M3_ROW)
            ref = _brute_w8a8_dense_layer(inp, k, act)
            assert np.allclose(res["out"], ref, rtol=1e-11, atol=1e-12), f"W8A8 layer (act={act}, E={E})"
            plain = o.moe_layer(inp, k, act)
            assert np.array_equal(res["ids"], plain["ids"]), "the router projects the unquantised x"
            d = np.abs(res["out"] - plain["out"]).max() / np.sqrt(np.mean(plain["out"] ** 2))
            assert 1e-4 < d < 0.5, f"W8A8 error {d} not of e4m3 size"


ALL_CHECKS = [
    check_topk_brute_force, check_topk_all_equal, check_topk_full_softmax, check_topk_weight_invariants,
    check_routing_brute_force, check_permute_round_trip, check_swiglu_golden, check_activations_library,
    check_single_expert_is_dense_mlp, check_layer_vs_dense_then_mask, check_identical_experts,
    check_shared_only, check_fp8_scale_identity, check_subset_matches_full, check_counts_sum,
    check_near_ties, check_e4m3_round, check_bf16_round, check_quantize_rows, check_w8a8_layer,
]
