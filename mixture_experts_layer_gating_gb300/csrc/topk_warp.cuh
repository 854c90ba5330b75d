// Gating top-k softmax of one token by one warp ("CANN/cann-recipes-infer：
// Qwen3-MoE优化", section "GMM使能和Routing优化": gating_top_k_softmax; the
// "Gemma-4 模型优化报告" §6 MoE Router row).  Shared by the stand-alone top-k
// kernel (routing.cu) and the router projection fused with top-k
// (router_sm103.cu), so that both take every decision the same way.
#pragma once

#include <cstdint>

#include "moe_internal.h"

namespace moe {

// Lane l holds the token's projected logits of experts l, l + 32, ... in v
// (EPL = ceil(E / 32) <= 16 entries; entries past E are ignored).  The routine
//  1. adds bias[e] (when bias is given) and, when logits_row is given, writes
//     the final logits there;
//  2. treats a non-finite logit as -inf and flags MOE_DEV_NONFINITE_LOGIT;
//  3. picks the k largest logits in the order (value descending, lower expert
//     index first) by k rounds of warp integer max / min reductions over
//     order-preserving keys (-0 is made +0 first so equal values compare
//     equal; experts past E get key 0, below every finite or -inf logit);
//  4. writes ids_row[j] and w_row[j] for j < k: softmax over the k chosen
//     logits (renorm) or the full-softmax probability of the chosen experts;
//     a token whose every logit is non-finite gets weights 1 / k.
// Returns ids_row[lane] on lanes below k, -1 on the others.
// k <= 32 and E <= 32 * EPL.
template <int EPL>
__device__ __forceinline__ int warp_topk_softmax(float (&v)[EPL], int lane, int E, int k,
                                                  int renorm, const float* __restrict__ bias,
                                                  float* logits_row, int32_t* __restrict__ ids_row,
                                                  float* __restrict__ w_row, int32_t* err) {
  constexpr unsigned kFull = 0xffffffffu;
  bool nonfinite = false;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    float x = -INFINITY;
    if (e < E) {
      x = v[i];
      if (bias) x += bias[e];
      if (logits_row) logits_row[e] = x;
      if (!isfinite(x)) {
        nonfinite = true;
        x = -INFINITY;
      }
    }
    v[i] = x;
  }
  if (__any_sync(kFull, nonfinite) && lane == 0) atomicOr(err, MOE_DEV_NONFINITE_LOGIT);

  uint32_t key[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const uint32_t u = __float_as_uint(v[i] + 0.0f);
    key[i] = (lane + 32 * i < E) ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
  }
  uint32_t taken = 0;
  float my_v = -INFINITY;
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0;  // this lane's best remaining key (the lower index among equal keys)
    int bi = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      if (!((taken >> i) & 1u) && key[i] > bk) {
        bk = key[i];
        bi = i;
      }
    }
    const uint32_t wmax = __reduce_max_sync(kFull, bk);
    const uint32_t be =
        __reduce_min_sync(kFull, bk == wmax ? static_cast<uint32_t>(lane + 32 * bi) : 0xFFFFFFFFu);
    if (static_cast<int>(be & 31u) == lane) taken |= 1u << (be >> 5);
    if (lane == j) {
      my_v = __uint_as_float((wmax & 0x80000000u) ? (wmax & 0x7FFFFFFFu) : ~wmax);
      my_e = static_cast<int>(be);
    }
  }
  const float m = __shfl_sync(kFull, my_v, 0);
  float z = 0.0f;
  float denom;
  if (m == -INFINITY) {  // every logit non-finite: uniform weights
    z = lane < k ? 1.0f : 0.0f;
    denom = static_cast<float>(k);
  } else if (renorm) {
    z = lane < k ? expf(my_v - m) : 0.0f;
    denom = z;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) denom += __shfl_xor_sync(kFull, denom, off);
  } else {
    z = lane < k ? expf(my_v - m) : 0.0f;
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) s += (lane + 32 * i < E) ? expf(v[i] - m) : 0.0f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
    denom = s;
  }
  if (lane < k) {
    ids_row[lane] = my_e;
    w_row[lane] = z / denom;
  }
  return lane < k ? my_e : -1;
}

}  // namespace moe
