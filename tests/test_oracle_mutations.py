"""Plant plausible mistakes in the CPU oracle and check that the pins catch
each one.  Every mistake lives in the oracle, on the CPU."""
import numpy as np
import pytest

import oracle.moe_oracle as o
from tests import _pins

_orig = {name: getattr(o, name) for name in
         ("topk_softmax", "init_routing", "expert_ffn", "finalize", "activation",
          "scaled_projection", "router_logits", "permute", "near_tie_tokens", "quantize_rows_e4m3",
         "e4m3_round", "bf16_round", "dequantize_rows")}


def _swap_gate_up(rows, W13_e, W2_e, act, s13_e=None, s2_e=None, act_quant=None):
    W13_e, W2_e = o.to_f64(W13_e), o.to_f64(W2_e)
    I = W2_e.shape[0]
    gu = o.scaled_projection(rows, W13_e, o.to_f64(s13_e))
    h = o.activation(gu[:, I:], act) * gu[:, :I]
    h_in = h
    if act_quant:
        h = o.bf16_round(h)
        h_in = o.dequantize_rows(*o.quantize_rows_e4m3(h))
    return h, o.scaled_projection(h_in, W2_e, o.to_f64(s2_e))


def _h_not_quantised(rows, W13_e, W2_e, act, s13_e=None, s2_e=None, act_quant=None):
    return _orig["expert_ffn"](rows, W13_e, W2_e, act, s13_e, s2_e, None)


def _ties_to_high_index(L, k, renormalize=True):
    L = np.asarray(L, np.float64)
    E = L.shape[1]
    ids_rev, w = _orig["topk_softmax"](L[:, ::-1], k, renormalize)
    return (E - 1 - ids_rev).astype(np.int32), w


def _no_renormalize(L, k, renormalize=True):
    return _orig["topk_softmax"](L, k, False)


def _drop_shared(y_perm, dest, w, s=None):
    return _orig["finalize"](y_perm, dest, w, None)


def _unweighted_combine(y_perm, dest, w, s=None):
    return _orig["finalize"](y_perm, dest, np.ones_like(np.asarray(w, np.float64)), s)


def _scale_reversed_channels(A, W, scale):
    return _orig["scaled_projection"](A, W, None if scale is None else scale[::-1])


def _reverse_within_expert(ids, E):
    r = _orig["init_routing"](ids, E)
    flat = np.asarray(ids).reshape(-1)
    R = flat.size
    sr = np.array(sorted(range(R), key=lambda q: (flat[q], -q)), dtype=np.int64)
    dest = np.empty(R, dtype=np.int64)
    dest[sr] = np.arange(R)
    r.update(sorted_rows=sr, dest=dest)
    return r


def _dest_not_inverted(ids, E):
    r = _orig["init_routing"](ids, E)
    r["dest"] = r["sorted_rows"].copy()
    return r


def _erf_gelu(g, act):
    if act == o.ACT_GEGLU_TANH:
        import scipy.special
        return 0.5 * g * (1.0 + scipy.special.erf(g / np.sqrt(2.0)))
    return _orig["activation"](g, act)


def _bias_dropped(x, Wg, logit_bias=None):
    return _orig["router_logits"](x, Wg, None)


def _permute_off_by_one(x, sorted_rows, k):
    xx = o.to_f64(x)
    return xx[(np.asarray(sorted_rows) + 1) % (xx.shape[0] * k) // k]


def _ties_next_pair(L, k, eps=1e-4):
    """Compares the (k+1)-th and (k+2)-th logits instead of the k-th and (k+1)-th."""
    L = np.asarray(L, np.float64)
    if k + 1 >= L.shape[1]:
        return np.zeros(L.shape[0], dtype=bool)
    s = -np.sort(-L, axis=1)
    return (s[:, k] - s[:, k + 1]) < eps


def _ties_inclusive(L, k, eps=1e-4):
    """<= in place of <: a gap of exactly eps counts as a near tie."""
    L = np.asarray(L, np.float64)
    if k >= L.shape[1]:
        return np.zeros(L.shape[0], dtype=bool)
    s = -np.sort(-L, axis=1)
    return (s[:, k - 1] - s[:, k]) <= eps


def _ties_all_when_k_is_e(L, k, eps=1e-4):
    """k = E treated as if every token had a near tie."""
    L = np.asarray(L, np.float64)
    if k >= L.shape[1]:
        return np.ones(L.shape[0], dtype=bool)
    return _orig["near_tie_tokens"](L, k, eps)


def _ties_ascending(L, k, eps=1e-4):
    """The k-th and (k+1)-th smallest instead of largest logits."""
    L = np.asarray(L, np.float64)
    if k >= L.shape[1]:
        return np.zeros(L.shape[0], dtype=bool)
    s = np.sort(L, axis=1)
    return (s[:, k] - s[:, k - 1]) < eps


def _quant_per_column(a):
    q, sc = _orig["quantize_rows_e4m3"](np.asarray(a, np.float64).T)
    # a per-column scale, broadcast back as if it were per row (first rows)
    return q.T, np.resize(sc, np.asarray(a).shape[0])


def _quant_max_127(a):
    a32 = np.asarray(a, np.float64).astype(np.float32)
    amax = np.abs(a32).max(axis=1)
    sc = np.where(amax > 0, amax / np.float32(127.0), np.float32(1.0)).astype(np.float32)
    return o.e4m3_round((a32 / sc[:, None]).astype(np.float32)), sc.astype(np.float64)


def _quant_ties_away(v):
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.maximum(a, 2.0 ** -6))
    qn = np.ldexp(1.0, ex - 4)
    r = np.minimum(np.floor(a / qn + 0.5) * qn, 448.0)
    return np.copysign(r, v)


def _bf16_truncate(v):
    v = np.asarray(v, np.float64).astype(np.float32)
    return (v.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)


def _dequant_without_scale(q, sc):
    return np.asarray(q, np.float64)


MUTATIONS = {
    "gate_up_swapped": ("expert_ffn", _swap_gate_up),
    "ties_to_high_index": ("topk_softmax", _ties_to_high_index),
    "no_renormalize": ("topk_softmax", _no_renormalize),
    "shared_dropped": ("finalize", _drop_shared),
    "combine_unweighted": ("finalize", _unweighted_combine),
    "scale_channel_order": ("scaled_projection", _scale_reversed_channels),
    "unstable_within_expert": ("init_routing", _reverse_within_expert),
    "dest_not_inverted": ("init_routing", _dest_not_inverted),
    "erf_instead_of_tanh_gelu": ("activation", _erf_gelu),
    "router_bias_dropped": ("router_logits", _bias_dropped),
    "permute_off_by_one": ("permute", _permute_off_by_one),
    "near_ties_next_pair": ("near_tie_tokens", _ties_next_pair),
    "near_ties_inclusive": ("near_tie_tokens", _ties_inclusive),
    "near_ties_all_when_k_is_e": ("near_tie_tokens", _ties_all_when_k_is_e),
    "near_ties_ascending": ("near_tie_tokens", _ties_ascending),
    "w8a8_quantised_per_column": ("quantize_rows_e4m3", _quant_per_column),
    "w8a8_scale_to_127": ("quantize_rows_e4m3", _quant_max_127),
    "e4m3_ties_away_from_zero": ("e4m3_round", _quant_ties_away),
    "bf16_truncated": ("bf16_round", _bf16_truncate),
    "w8a8_scale_not_applied": ("dequantize_rows", _dequant_without_scale),
    "w8a8_h_not_quantised": ("expert_ffn", _h_not_quantised),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    fn_name, bad = MUTATIONS[name]
    monkeypatch.setattr(o, fn_name, bad)
    caught = []
    for check in _pins.ALL_CHECKS:
        try:
            check(o)
        except AssertionError:
            caught.append(check.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
