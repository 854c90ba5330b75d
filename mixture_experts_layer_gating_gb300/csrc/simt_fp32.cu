// fp32 path of the grouped expert FFN and the router projection, on CUDA
// cores (the tensor core has no full-precision fp32 kind).  It serves the
// all-fp32 configuration; the bf16 / fp8 configurations use the tcgen05
// kernels of gemm_sm103.cu.  Each thread computes a 1 x 4 strip of outputs of
// one row with fp32 FMA accumulation; 64-row x 64-column block tiles with the
// A rows staged through shared memory.
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int TR = 32;   // rows per block
constexpr int TC = 64;   // output columns per block
constexpr int TK = 32;   // reduction chunk

__device__ __forceinline__ int find_group(const int32_t* offsets, int G, int row) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (offsets[mid] <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }
__device__ __forceinline__ float gelu_tanh_f(float g) {
  const float c = 0.7978845608028654f;
  return 0.5f * g * (1.0f + tanhf(c * (g + 0.044715f * g * g * g)));
}

// out[r, c] = sum_k A[r, k] * W[g(r)][k, col_base + c]   for TR x TC tiles.
// MODE 0: gate/up -> h = act(gate) * up (W has 2N columns per group).
// MODE 1: plain projection (+ optional bias).
template <int MODE>
__global__ void simt_group_gemm(const float* __restrict__ A, const int32_t* __restrict__ offsets,
                                int G, int M, int K, const float* __restrict__ W, int N,
                                const float* __restrict__ bias, int act, float* __restrict__ out,
                                int32_t* err) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float As[TR][TK + 1];
  const int row0 = blockIdx.y * TR;
  const int col0 = blockIdx.x * TC;
  const int tr = threadIdx.x / (TC / 4);  // 0..15 -> two rows each
  const int tc = threadIdx.x % (TC / 4);  // 0..15 -> 4 columns each
  const int ldw = (MODE == 0) ? 2 * N : N;
  float accg[2][4] = {}, accu[2][4] = {};
  int rows[2], grp[2];
  bool rvalid[2];
  for (int i = 0; i < 2; ++i) {
    rows[i] = row0 + tr + 16 * i;
    rvalid[i] = rows[i] < M;
    grp[i] = 0;
    if (rvalid[i] && offsets) {
      if (rows[i] >= offsets[G]) rvalid[i] = false;
      else grp[i] = find_group(offsets, G, rows[i]);
    }
  }
  for (int k0 = 0; k0 < K; k0 += TK) {
    for (int idx = threadIdx.x; idx < TR * TK; idx += blockDim.x) {
      const int r = idx / TK, kk = idx % TK;
      const int gr = row0 + r, gk = k0 + kk;
      As[r][kk] = (gr < M && gk < K) ? A[static_cast<size_t>(gr) * K + gk] : 0.0f;
    }
    __syncthreads();
    for (int i = 0; i < 2; ++i) {
      if (!rvalid[i]) continue;
      const float* Wg = W + static_cast<size_t>(grp[i]) * K * ldw;
      for (int kk = 0; kk < TK && k0 + kk < K; ++kk) {
        const float a = As[tr + 16 * i][kk];
        const float* wrow = Wg + static_cast<size_t>(k0 + kk) * ldw;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = col0 + tc * 4 + j;
          if (c < N) {
            accg[i][j] = fmaf(a, wrow[c], accg[i][j]);
            if (MODE == 0) accu[i][j] = fmaf(a, wrow[N + c], accu[i][j]);
          }
        }
      }
    }
    __syncthreads();
  }
  for (int i = 0; i < 2; ++i) {
    if (!rvalid[i]) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = col0 + tc * 4 + j;
      if (c >= N) continue;
      float v;
      if (MODE == 0) {
        const float g = accg[i][j];
        v = (act == MOE_ACT_SWIGLU ? silu_f(g) : gelu_tanh_f(g)) * accu[i][j];
      } else {
        v = accg[i][j] + (bias ? bias[c] : 0.0f);
      }
      out[static_cast<size_t>(rows[i]) * N + c] = v;
    }
  }
}

}  // namespace

cudaError_t launch_simt_router(const float* x, const float* Wg, const float* bias, float* logits,
                               int T, int D, int E, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  dim3 grid((E + TC - 1) / TC, (T + TR - 1) / TR);
  return launch_kernel(simt_group_gemm<1>, grid, dim3(256), 0, s, x, nullptr, 1, T, D, Wg, E, bias,
                       0, logits, nullptr);
}

cudaError_t launch_simt_gate_up(const float* A, const int32_t* offsets, int G, int M, int K,
                                const float* W13, int I, int act, float* h, int32_t* err,
                                cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  dim3 grid((I + TC - 1) / TC, (M + TR - 1) / TR);
  return launch_kernel(simt_group_gemm<0>, grid, dim3(256), 0, s, A, offsets, G, M, K, W13, I,
                       nullptr, act, h, err);
}

cudaError_t launch_simt_down(const float* h, const int32_t* offsets, int G, int M, int I,
                             const float* W2, int N, float* y, int32_t* err, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  dim3 grid((N + TC - 1) / TC, (M + TR - 1) / TR);
  return launch_kernel(simt_group_gemm<1>, grid, dim3(256), 0, s, h, offsets, G, M, I, W2, N,
                       nullptr, 0, y, err);
}

}  // namespace moe
