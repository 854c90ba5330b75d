"""CPU fp64 oracle of the sparse Mixture-of-Experts FFN layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the test suite, the package smoke check and the
benchmark's CPU-baseline / reference leg use it.  It shares no code with the
CUDA implementation.

It is the plain definition of what the layer computes, written out step by
step in the order and notation of the source pages, with a per-expert loop
and float64 arithmetic throughout (every bf16 / fp32 / e4m3 input converts to
float64 exactly).  A library matmul or sort serves as a single step; there is
no blocking, fusion or reordering beyond the definition.

Steps and the passages they follow
----------------------------------
1. Router projection ``L = x W_g`` -- "千问 3.5 MoE 在 TPU 上的系统优化实战",
   routed sparse MoE paragraph (the router gate projects the token and picks
   the top 10 experts through a softmax distribution); the gate is computed
   from an fp32 copy of the hidden state -- "CANN/cann-recipes-infer：
   Qwen3-MoE优化", section "融合RMSNorm + Cast".
2. Top-k + softmax gating -- Qwen3-MoE page, section "GMM使能和Routing优化"
   (npu_moe_gating_top_k_softmax fuses top-k and softmax); Gemma-4 page §6
   ("MoE Router" row).  Readings: ties go to the lower expert index; the k
   weights are renormalised to sum to one.
3. Routing metadata -- Qwen3-MoE page, "GMM使能和Routing优化"
   (npu_moe_init_routing sorts the expanded rows by expert;
   npu_moe_compute_expert_tokens counts tokens per expert).  Reading: the
   sort is stable in the expanded row index r = t*k + j.
4. Permutation gather -- Qwen3.5 page, SparseCore paragraph (token rows are
   gathered by routing index into one contiguous buffer, no padding).
5. Expert FFN -- Qwen3-MoE page, "MoE TP优化 / 计算分解": each expert is
   down(SiLU(gate(x)) * up(x)); gate and up are concatenated into w13 and the
   fused swiglu splits the last dim in two halves, SiLU(first) * second.
   Gemma-4 page §2: the experts use GEGLU (gelu(gate) * up).
   fp8 weights -- Ling-2.6-1T page §5 "逐通道 direct_scaled_dot": with a
   per-output-channel scale the scale multiplies the finished K reduction,
   out[m, n] = (sum_k A[m, k] W[k, n]) * scale[n].
6. Grouped matmul over experts -- Qwen3-MoE page, "GMM使能和Routing优化"
   (one grouped op instead of a per-expert loop); here the loop is kept on
   purpose because this is the oracle.
7. Finalize -- Qwen3-MoE page, "GMM使能和Routing优化"
   (npu_moe_finalize_routing puts expert outputs back in token order and takes
   the weighted sum).
8. Shared expert / dense MLP -- Qwen3.5 page: y = Router(x) + SharedExpert(x);
   Ling page §1 (the shared expert is a local dense path on every token);
   Gemma-4 page §2 (dense MLP and MoE run in parallel and are added).
9. W8A8 (optional) -- Ling page §5 "激活量化" and "逐通道 direct_scaled_dot":
   activations quantised to fp8 per token with a dynamic scale, fp8 x fp8
   products, per-token and per-channel scales after the reduction.

Every function here is pinned by the CPU tests to something other than itself
(brute force, textbook / library routines, invariants, printed values).
"""
from __future__ import annotations

import math
from typing import Dict, Optional

import numpy as np

ACT_SWIGLU = "swiglu"
ACT_GEGLU_TANH = "geglu_tanh"
ACT_QUANT_E4M3_ROW = "e4m3_row"  # W8A8: activations quantised per row to e4m3


def to_f64(a) -> Optional[np.ndarray]:
    """Exact float64 copy of a torch tensor (any float dtype) or array."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        import torch

        return a.detach().to(device="cpu", dtype=torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------- step 1
def router_logits(x, Wg, logit_bias=None) -> np.ndarray:
    """L[t, e] = sum_d x[t, d] * W_g[d, e]  (+ b_e), in float64."""
    L = to_f64(x) @ to_f64(Wg)
    if logit_bias is not None:
        L = L + to_f64(logit_bias)[None, :]
    return L


# ---------------------------------------------------------------- step 2
def topk_softmax(L, k: int, renormalize: bool = True):
    """Top-k experts per token and their gate weights.

    Experts are ranked by descending logit, the lower index first among equal
    logits; ``ids[t]`` lists the k chosen experts in that order.  With
    renormalisation the weights are the softmax over the k selected logits
    (equivalently: softmax over all E, then divide by the selected mass);
    without it they are the full softmax probabilities of the k experts.
    """
    L = np.asarray(L, dtype=np.float64)
    T, E = L.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    if not np.isfinite(L).all():
        raise ValueError("router logits must be finite")
    order = np.argsort(-L, axis=1, kind="stable")
    ids = order[:, :k]
    top = np.take_along_axis(L, ids, axis=1)
    if renormalize:
        z = np.exp(top - top[:, :1])
        w = z / z.sum(axis=1, keepdims=True)
    else:
        z = np.exp(L - L.max(axis=1, keepdims=True))
        p = z / z.sum(axis=1, keepdims=True)
        w = np.take_along_axis(p, ids, axis=1)
    return ids.astype(np.int32), w


def near_tie_tokens(L, k: int, eps: float = 1e-4) -> np.ndarray:
    """Tokens whose k-th and (k+1)-th largest logits differ by less than eps.

    For these tokens a last-bit difference in the router projection may
    legitimately choose another expert, so id and layer-output comparisons
    leave them out.
    """
    L = np.asarray(L, dtype=np.float64)
    if k >= L.shape[1]:
        return np.zeros(L.shape[0], dtype=bool)
    s = -np.sort(-L, axis=1)
    return (s[:, k - 1] - s[:, k]) < eps


# ---------------------------------------------------------------- W8A8 forms
# "用SGLang-JAX在TPU上优化Ling-2.6-1T" §5, "激活量化": the fused kernel
# quantises the routed tokens' activations from bf16 to fp8 with a dynamic
# per-token scale (before the scatter), and "逐通道 direct_scaled_dot" feeds
# fp8 tokens and fp8 weights to the matrix unit, applying the per-token and
# per-channel scales after the f32 reduction.  Readings (the pages give no
# formula): the scale of a row is its largest |value| over 448, the largest
# e4m3 value; codes are the nearest e4m3 value of value / scale with ties to
# the even code; both divisions are fp32 operations on the bf16 values; the
# intermediate h is carried in bf16 between the two projections (as the bf16
# activations are) and quantised per row the same way before the down
# projection.
E4M3_MAX = 448.0


def _round_binary(v, mant_bits: int, emin: int, vmax: float) -> np.ndarray:
    """Nearest value of a binary floating-point format with `mant_bits`
    fraction bits, smallest normal exponent `emin` (subnormals below it) and
    largest finite value `vmax`; ties to the even significand; magnitudes
    beyond vmax saturate to vmax."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.maximum(a, 2.0 ** emin))  # a = m 2^ex, m in [0.5, 1)
    quantum = np.ldexp(1.0, ex - 1 - mant_bits)  # spacing of the format at a
    r = np.round(a / quantum) * quantum  # a / quantum is exact; np.round: half to even
    r = np.minimum(r, vmax)
    return np.copysign(r, v)


def e4m3_round(v) -> np.ndarray:
    """Nearest e4m3 (fn: 4 exponent bits, bias 7, 3 fraction bits, largest
    finite 448) value of each element, ties to the even code, saturating."""
    return _round_binary(v, 3, -6, E4M3_MAX)


def bf16_round(v) -> np.ndarray:
    """Nearest bf16 value of each element (ties to even)."""
    return _round_binary(v, 7, -126, float(np.finfo(np.float32).max))


def quantize_rows_e4m3(a):
    """Dynamic per-row e4m3 quantisation: returns (q, s) with q [rows, n] the
    e4m3 codes' values and s [rows] the fp32 scales, so that q * s[:, None]
    approximates a.  s = amax / 448 and q = e4m3(a / s), divisions in fp32; a
    row of zeros gets s = 1."""
    a32 = np.asarray(a, dtype=np.float64).astype(np.float32)
    amax = np.abs(a32).max(axis=1) if a32.shape[1] else np.zeros(a32.shape[0], np.float32)
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = e4m3_round((a32 / s[:, None]).astype(np.float32))
    return q, s.astype(np.float64)


def dequantize_rows(q, s) -> np.ndarray:
    return np.asarray(q, np.float64) * np.asarray(s, np.float64)[:, None]


# ---------------------------------------------------------------- step 3
def init_routing(ids, E: int) -> Dict[str, np.ndarray]:
    """Expert histogram, exclusive scan and stable sort of expanded rows.

    Expanded row r = t*k + j holds token t's j-th choice.  ``sorted_rows[p]``
    is the expanded row placed at permuted position p (rows grouped by
    expert, ascending r inside an expert); ``dest`` is the inverse map.
    """
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    R = flat.size
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    sorted_rows = np.argsort(flat, kind="stable").astype(np.int64)
    dest = np.empty(R, dtype=np.int64)
    dest[sorted_rows] = np.arange(R, dtype=np.int64)
    return {"counts": counts, "offsets": offsets, "sorted_rows": sorted_rows, "dest": dest}


# ---------------------------------------------------------------- step 4
def permute(x, sorted_rows, k: int) -> np.ndarray:
    """x_perm[p] = x[sorted_rows[p] // k]."""
    return to_f64(x)[np.asarray(sorted_rows) // k]


# ---------------------------------------------------------------- step 5
def activation(g: np.ndarray, act: str) -> np.ndarray:
    """SiLU(g) = g / (1 + e^-g); tanh-GELU(g) = g/2 (1 + tanh(sqrt(2/pi)(g + 0.044715 g^3)))."""
    with np.errstate(over="ignore"):
        if act == ACT_SWIGLU:
            return g / (1.0 + np.exp(-g))
        if act == ACT_GEGLU_TANH:
            c = math.sqrt(2.0 / math.pi)
            return 0.5 * g * (1.0 + np.tanh(c * (g + 0.044715 * g ** 3)))
    raise ValueError(f"unknown activation {act!r}")


def scaled_projection(A: np.ndarray, W: np.ndarray, scale: Optional[np.ndarray]) -> np.ndarray:
    """(sum_k A[m, k] W[k, n]) * scale[n]; the scale comes after the reduction."""
    out = A @ W
    if scale is not None:
        out = out * scale[None, :]
    return out


def expert_ffn(rows: np.ndarray, W13_e, W2_e, act: str, s13_e=None, s2_e=None,
               act_quant: Optional[str] = None):
    """One expert on a block of rows: h = act(gate) * up; y = h W2.

    W13_e is [D, 2I] with the gate projection in the first I columns and the
    up projection in the last I columns.  Returns (h, y).  With act_quant =
    "e4m3_row" (W8A8) the rows arrive already quantised (q * s) and h is
    rounded to bf16, then quantised per row, before the down projection; the
    returned h is the bf16 h.
    """
    W13_e, W2_e = to_f64(W13_e), to_f64(W2_e)
    I = W2_e.shape[0]
    gu = scaled_projection(rows, W13_e, to_f64(s13_e))
    gate, up = gu[:, :I], gu[:, I:]
    h = activation(gate, act) * up
    h_in = h
    if act_quant == ACT_QUANT_E4M3_ROW:
        h = bf16_round(h)
        h_in = dequantize_rows(*quantize_rows_e4m3(h))
    elif act_quant is not None:
        raise ValueError(f"unknown activation quantisation {act_quant!r}")
    y = scaled_projection(h_in, W2_e, to_f64(s2_e))
    return h, y


# ---------------------------------------------------------------- step 6
def grouped_ffn(x_perm: np.ndarray, offsets, W13, W2, act: str, s13=None, s2=None,
                act_quant: Optional[str] = None):
    """Per-expert loop over the contiguous expert segments of x_perm."""
    offsets = np.asarray(offsets)
    E = len(offsets) - 1
    R = x_perm.shape[0]
    I, D = W2.shape[1], W2.shape[2]
    h = np.zeros((R, I))
    y = np.zeros((R, D))
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        h[a:b], y[a:b] = expert_ffn(
            x_perm[a:b], W13[e], W2[e], act,
            None if s13 is None else s13[e], None if s2 is None else s2[e], act_quant)
    return h, y


# ---------------------------------------------------------------- step 8
def shared_expert(x, W13s, W2s, act: str, s13s=None, s2s=None,
                  act_quant: Optional[str] = None) -> np.ndarray:
    """The always-on expert (or dense MLP) applied to every token (x already
    quantised when act_quant is set)."""
    _, y = expert_ffn(to_f64(x), W13s, W2s, act, s13s, s2s, act_quant)
    return y


# ---------------------------------------------------------------- step 7
def finalize(y_perm: np.ndarray, dest, w, s: Optional[np.ndarray] = None) -> np.ndarray:
    """out[t] = sum_j w[t, j] * y_perm[dest[t*k + j]]  (+ s[t])."""
    w = np.asarray(w, dtype=np.float64)
    T, k = w.shape
    d = np.asarray(dest).reshape(T, k)
    out = np.zeros((T, y_perm.shape[1]))
    for j in range(k):
        out += w[:, j:j + 1] * y_perm[d[:, j]]
    if s is not None:
        out = out + s
    return out


# ---------------------------------------------------------------- layer
def moe_layer(inp: Dict, k: int, act: str, renormalize: bool = True,
              logits: Optional[np.ndarray] = None,
              act_quant: Optional[str] = None) -> Dict[str, np.ndarray]:
    """The whole layer: route, permute, grouped FFN, shared expert, finalize.

    ``inp`` holds x, Wg, logit_bias, W13, W2, s13, s2, W13s, W2s, s13s, s2s
    (torch tensors or arrays; absent / None entries are skipped).  When
    ``logits`` is given it replaces step 1 (used to compare routing against
    an implementation's own fp32 logits).  ``act_quant`` = "e4m3_row" is the
    W8A8 form: the router still projects the bf16 x, while the expert and
    shared-expert FFNs take x quantised per token (before the permutation)
    and h quantised per row.  Returns every intermediate.
    """
    x = to_f64(inp["x"])
    E = inp["W13"].shape[0]
    L = router_logits(x, inp["Wg"], inp.get("logit_bias")) if logits is None else np.asarray(logits, np.float64)
    ids, w = topk_softmax(L, k, renormalize)
    r = init_routing(ids, E)
    x_ffn = x
    if act_quant == ACT_QUANT_E4M3_ROW:
        x_ffn = dequantize_rows(*quantize_rows_e4m3(x))
    elif act_quant is not None:
        raise ValueError(f"unknown activation quantisation {act_quant!r}")
    x_perm = permute(x_ffn, r["sorted_rows"], k)
    h, y_perm = grouped_ffn(x_perm, r["offsets"], inp["W13"], inp["W2"], act,
                            inp.get("s13"), inp.get("s2"), act_quant)
    s = None
    if inp.get("W13s") is not None:
        s = shared_expert(x_ffn, inp["W13s"], inp["W2s"], act, inp.get("s13s"), inp.get("s2s"),
                          act_quant)
    out = finalize(y_perm, r["dest"], w, s)
    res = {"logits": L, "ids": ids, "w": w, "x_perm": x_perm, "h": h, "y_perm": y_perm,
           "shared": s, "out": out}
    res.update(r)
    return res


def moe_layer_tokens(inp: Dict, tokens, k: int, act: str, renormalize: bool = True,
                     act_quant: Optional[str] = None) -> np.ndarray:
    """Layer output for a subset of tokens only.

    Routing, expert FFNs and the combine act on each token independently, so
    out[tokens] of the full batch equals the layer applied to x[tokens].
    """
    tokens = np.asarray(tokens)
    sub = dict(inp)
    x = inp["x"]
    sub["x"] = x[tokens] if not hasattr(x, "detach") else x.detach().cpu()[tokens]
    return moe_layer(sub, k, act, renormalize, act_quant=act_quant)["out"]
