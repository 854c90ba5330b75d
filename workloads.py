"""Seeded synthetic workloads for the sparse MoE FFN layer.

This module is shared by the CPU oracle, the tests and the benchmark.  It only
describes shapes and draws random inputs; it holds none of the layer's
arithmetic (no routing, no activation, no GEMM).

Shapes follow the MoE layers the source pages discuss:
  * Qwen3-MoE (Ascend recipe, "CANN/cann-recipes-infer: Qwen3-MoE" page,
    section "MoE TP"): D=2048, 128 experts, top-8, expert intermediate 768.
  * Gemma-4-26B-A4B ("Gemma-4 模型优化报告", section 2 model structure):
    D=2816, 128 experts, top-8, intermediate 704, GEGLU experts plus a dense
    MLP of intermediate 2112 whose output is added to the MoE output.
  * Qwen3.5-397B ("千问 3.5 MoE 在 TPU 上的系统优化实战", model section):
    D=4096, 512 experts, top-10, intermediate 1024, always-on shared expert.
  * Ling-2.6-1T ("用SGLang-JAX在TPU上优化Ling-2.6-1T", section 1 cost model):
    D=8192, 256 experts, top-8, intermediate 2048, one shared expert,
    per-output-channel fp8 weights.
The token counts (prefill / decode batch) are the ones these pages measure on.
No dataset is used: MoE-layer cost depends on token count and routing only,
so seeded Gaussian inputs of the same shapes stand in for the serving traces.

Input recipe (identical for every config):
  x ~ N(0, 1); W_g, W13, W2 (and the shared expert's) ~ N(0, 0.02);
  cast to the config's dtypes.  fp8 weights are quantised per output column:
  s[n] = max_k |W[k, n]| / 448, q = e4m3(W / s) (round to nearest even).
  The Zipf-skewed config adds a per-expert logit bias b_e = -a * ln(rank_e)
  with rank a seeded random permutation of 1..E, which multiplies each
  expert's softmax mass by a Zipf(a) weight.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import torch

ACT_SWIGLU = "swiglu"
ACT_GEGLU_TANH = "geglu_tanh"

FP8_E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class MoEShape:
    """Static description of one MoE layer workload."""

    name: str
    T: int  # tokens in the batch
    D: int  # hidden size
    E: int  # routed experts
    k: int  # experts per token
    I: int  # routed expert intermediate size
    I_shared: int = 0  # shared expert / dense MLP intermediate (0 = none)
    act: str = ACT_SWIGLU
    w_dtype: str = "bf16"  # "f32" | "bf16" | "fp8_e4m3"
    act_dtype: str = "bf16"  # "f32" | "bf16"
    renormalize: bool = True
    zipf: float = 0.0  # Zipf exponent of the per-expert logit bias (0 = none)

    @property
    def R(self) -> int:
        """Routed (token, slot) rows."""
        return self.T * self.k

    def with_tokens(self, T: int) -> "MoEShape":
        return dataclasses.replace(self, T=T, name=f"{self.name.split('@')[0]}@T{T}")


def _qwen3(T):
    return MoEShape(f"qwen3_moe@T{T}", T, 2048, 128, 8, 768)


def _gemma4(T):
    return MoEShape(f"gemma4_moe@T{T}", T, 2816, 128, 8, 704, I_shared=2112, act=ACT_GEGLU_TANH)


def _qwen35(T):
    return MoEShape(f"qwen35_397b_moe@T{T}", T, 4096, 512, 10, 1024, I_shared=1024, zipf=1.1)


def _ling(T):
    return MoEShape(f"ling_1t_moe@T{T}", T, 8192, 256, 8, 2048, I_shared=2048, w_dtype="fp8_e4m3")


CONFIGS: Dict[str, MoEShape] = {
    "toy": MoEShape("toy", 64, 256, 8, 2, 128, w_dtype="f32", act_dtype="f32"),
    "qwen3_prefill": _qwen3(4096),
    "qwen3_decode": _qwen3(64),
    "gemma4_prefill": _gemma4(2048),
    "gemma4_decode": _gemma4(8),
    "qwen35_prefill": _qwen35(8192),
    "qwen35_decode64": _qwen35(64),
    "qwen35_decode128": _qwen35(128),
    "qwen35_decode256": _qwen35(256),
    "qwen35_decode512": _qwen35(512),
    "ling_prefill": _ling(16384),
    "ling_decode": _ling(512),
}

_TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "fp8_e4m3": torch.float8_e4m3fn}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPES[name]


def quantize_fp8_per_column(w: torch.Tensor):
    """Per-output-column e4m3 quantisation of a [..., K, N] fp32 weight.

    Returns (q, s) with q e4m3 of the same shape and s fp32 of shape [..., N],
    s = amax over K / 448 (columns that are all zero get s = 1).
    """
    amax = w.abs().amax(dim=-2)
    s = torch.where(amax > 0, amax / FP8_E4M3_MAX, torch.ones_like(amax))
    q = (w / s.unsqueeze(-2)).clamp_(-FP8_E4M3_MAX, FP8_E4M3_MAX).to(torch.float8_e4m3fn)
    return q, s.to(torch.float32)


def zipf_logit_bias(E: int, a: float, gen: torch.Generator, device) -> torch.Tensor:
    """b_e = -a ln(rank_e), rank a seeded random permutation of 1..E."""
    rank = torch.randperm(E, generator=gen, device=device).to(torch.float64) + 1.0
    return (-a * torch.log(rank)).to(torch.float32)


def _normal(shape, std, gen, device):
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=gen)
    return t


def make_inputs(shape: MoEShape, seed: int = 0, device="cpu", weights_seed: Optional[int] = None) -> Dict[str, Optional[torch.Tensor]]:
    """Draw one seeded set of layer inputs.

    Tokens and weights use separate generators (``seed`` and ``weights_seed``,
    the latter defaulting to ``seed``) so that a batch of a different size can
    reuse the same weights.  Per-expert weights are drawn expert by expert to
    bound the temporary fp32 footprint.
    """
    device = torch.device(device)
    wseed = seed if weights_seed is None else weights_seed
    gx = torch.Generator(device=device)
    gx.manual_seed(seed * 7919 + 17)
    gw = torch.Generator(device=device)
    gw.manual_seed(wseed * 104729 + 3)

    adt = torch_dtype(shape.act_dtype)
    D, E, I, Is = shape.D, shape.E, shape.I, shape.I_shared
    out: Dict[str, Optional[torch.Tensor]] = {}
    out["x"] = _normal((shape.T, D), 1.0, gx, device).to(adt)
    router_dt = torch.float32 if shape.act_dtype == "f32" else torch.bfloat16
    out["Wg"] = _normal((D, E), 0.02, gw, device).to(router_dt)
    out["logit_bias"] = zipf_logit_bias(E, shape.zipf, gw, device) if shape.zipf > 0 else None

    fp8 = shape.w_dtype == "fp8_e4m3"
    wdt = torch_dtype(shape.w_dtype)
    W13 = torch.empty((E, D, 2 * I), dtype=wdt, device=device)
    W2 = torch.empty((E, I, D), dtype=wdt, device=device)
    s13 = torch.empty((E, 2 * I), dtype=torch.float32, device=device) if fp8 else None
    s2 = torch.empty((E, D), dtype=torch.float32, device=device) if fp8 else None
    for e in range(E):
        a = _normal((D, 2 * I), 0.02, gw, device)
        b = _normal((I, D), 0.02, gw, device)
        if fp8:
            W13[e], s13[e] = quantize_fp8_per_column(a)
            W2[e], s2[e] = quantize_fp8_per_column(b)
        else:
            W13[e] = a.to(wdt)
            W2[e] = b.to(wdt)
    out.update(W13=W13, W2=W2, s13=s13, s2=s2)

    if Is > 0:
        a = _normal((D, 2 * Is), 0.02, gw, device)
        b = _normal((Is, D), 0.02, gw, device)
        if fp8:
            out["W13s"], out["s13s"] = quantize_fp8_per_column(a)
            out["W2s"], out["s2s"] = quantize_fp8_per_column(b)
        else:
            out["W13s"], out["s13s"] = a.to(wdt), None
            out["W2s"], out["s2s"] = b.to(wdt), None
    else:
        out.update(W13s=None, s13s=None, W2s=None, s2s=None)
    return out


# ---------------------------------------------------------------------------
# Algorithmic work counters (measurement bookkeeping, not layer arithmetic).
# ---------------------------------------------------------------------------

def _wbytes(dtype: str) -> int:
    return {"f32": 4, "bf16": 2, "fp8_e4m3": 1}[dtype]


def ffn_gate_up_flops(rows: int, D: int, I: int) -> int:
    """Gate and up projections (two D x I matrices), 2 flops per MAC."""
    return 2 * rows * D * (2 * I)


def ffn_down_flops(rows: int, D: int, I: int) -> int:
    """Down projection (one I x D matrix), 2 flops per MAC."""
    return 2 * rows * I * D


def ffn_flops(rows: int, D: int, I: int) -> int:
    return ffn_gate_up_flops(rows, D, I) + ffn_down_flops(rows, D, I)


def layer_flops(shape: MoEShape) -> int:
    f = ffn_flops(shape.R, shape.D, shape.I) + 2 * shape.T * shape.D * shape.E
    if shape.I_shared:
        f += ffn_flops(shape.T, shape.D, shape.I_shared)
    return f


def expert_weight_bytes(D: int, I: int, w_dtype: str, scales: bool = True) -> int:
    b = 3 * D * I * _wbytes(w_dtype)
    if scales and w_dtype == "fp8_e4m3":
        b += 4 * (2 * I + D)
    return b


def layer_bytes(shape: MoEShape, active_experts: Optional[int] = None) -> int:
    """Minimum HBM traffic of one layer call: every active expert's weights
    once, the shared expert and router weights once, x read once, out written
    once.  Intermediates (permuted rows, h, expert outputs) are excluded."""
    E_act = shape.E if active_experts is None else active_experts
    abytes = _wbytes(shape.act_dtype)
    rbytes = 4 if shape.act_dtype == "f32" else 2
    b = E_act * expert_weight_bytes(shape.D, shape.I, shape.w_dtype)
    if shape.I_shared:
        b += expert_weight_bytes(shape.D, shape.I_shared, shape.w_dtype)
    b += shape.D * shape.E * rbytes
    b += 2 * shape.T * shape.D * abytes
    return b


def expected_active_experts(shape: MoEShape) -> float:
    """Expected count of experts hit at least once under uniform routing."""
    p_miss = (1.0 - shape.k / shape.E) ** shape.T
    return shape.E * (1.0 - p_miss)


def config_summary(shape: MoEShape) -> dict:
    return {
        "workload": shape.name,
        "T": shape.T, "D": shape.D, "E": shape.E, "k": shape.k, "I": shape.I,
        "I_shared": shape.I_shared, "act": shape.act, "w_dtype": shape.w_dtype,
        "act_dtype": shape.act_dtype, "zipf": shape.zipf,
    }


__all__ = [
    "MoEShape", "CONFIGS", "make_inputs", "quantize_fp8_per_column", "zipf_logit_bias",
    "ACT_SWIGLU", "ACT_GEGLU_TANH", "layer_flops", "layer_bytes", "ffn_flops", "ffn_gate_up_flops", "ffn_down_flops",
    "expert_weight_bytes", "expected_active_experts", "torch_dtype", "config_summary",
]
