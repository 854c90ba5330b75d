// Routing-side kernels of the MoE layer: the router projection of small
// batches (CUDA cores), gating top-k softmax, init_routing (histogram,
// exclusive scan, stable scatter: two kernels, or one 8-CTA cluster that
// exchanges its histograms through distributed shared memory, or one
// launch with the gather for small batches), the permutation (gather or token-side
// scatter), the fp8 layers' row forms (fp16 or two-term e4m3 rows with
// power-of-two scales), the one-time fp8 weight transpose and the finalize
// (weighted un-permute + shared-expert add).  All are memory- or
// latency-bound; they move 16-byte vectors and keep every index
// bounds-checked so that bad input data is reported through the error word
// instead of faulting.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cfloat>
#include <climits>

#include "moe_internal.h"
#include "sm103_ptx.cuh"
#include "topk_warp.cuh"

namespace moe {
namespace {

constexpr unsigned FULL = 0xffffffffu;

// ------------------------------------------------------------------------
// gating_top_k_softmax ("CANN/cann-recipes-infer：Qwen3-MoE优化", section
// "GMM使能和Routing优化"; "Gemma-4 模型优化报告" §6 MoE Router row).
// One warp per token; lane l holds experts l, l+32, ... (E <= 512).  k rounds
// of a warp arg-max with the order (higher logit, then lower index).  Weights:
// softmax over the k chosen logits (renormalised) or full-softmax probabilities.
// The router projection may arrive as nsplit fp32 partial planes [nsplit, T, E]
// (split-K); they are summed in plane order, the bias added last, and the final
// logits written to `logits` (which may alias plane 0).
template <int EPL>
__global__ void topk_softmax_kernel(const float* __restrict__ partials, int nsplit,
                                    const float* __restrict__ bias, float* logits, int T, int E,
                                    int k, int renorm, int32_t* __restrict__ ids,
                                    float* __restrict__ w, int32_t* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int warps_per_block = blockDim.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long t = static_cast<long long>(blockIdx.x) * warps_per_block + (threadIdx.x >> 5);
  if (t >= T) return;
  const size_t plane = static_cast<size_t>(T) * E;
  float v[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? partials[t * E + e] : 0.0f;
  }
  // planes summed in order; the loads of up to four planes are issued
  // together (one memory round trip per four planes, not per plane)
  for (int sp0 = 1; sp0 < nsplit; sp0 += 4) {
    float pv[4][EPL];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float* pl = partials + min(sp0 + q, nsplit - 1) * plane + t * E;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        pv[q][i] = (sp0 + q < nsplit && e < E) ? pl[e] : 0.0f;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (sp0 + q < nsplit) {
#pragma unroll
        for (int i = 0; i < EPL; ++i) v[i] += pv[q][i];
      }
    }
  }
  warp_topk_softmax<EPL>(v, lane, E, k, renorm, bias, (nsplit > 1 || bias) ? logits + t * E : nullptr,
                         ids + t * k, w + t * k, err);
}

// ------------------------------------------------------------------------
// Router projection for small batches ("CANN/cann-recipes-infer：Qwen3-MoE优化",
// the gate GEMM in fp32; "千问 3.5 MoE 在 TPU 上的系统优化实战": decode is bound by
// reading weights).  At a few tokens the projection is a matrix-vector product
// per token bounded by reading W_g, and a 128-row tensor-core tile would be
// almost empty, so it runs on the CUDA cores:
//   planes[s][t][e] = sum over d in slice s of x[t][d] * W_g[d][e]
// with slice s = [s*dc, min(D, (s+1)*dc)).  A block takes 64 experts (two per
// lane), one slice and kRouterTok tokens; its kRouterWarps warps split the
// slice into contiguous pieces (fp32 FMA in ascending d inside a piece), and
// the pieces are added in warp order.  The top-k kernel sums the planes in
// plane order and adds the bias.
constexpr int kRouterTok = 4;
constexpr int kRouterWarps = 8;
constexpr int kRouterMaxSlice = 1024;  // d per plane staged in shared memory
constexpr int kRouterUnroll = 16;      // W_g loads in flight per lane

__global__ void __launch_bounds__(kRouterWarps * 32)
    router_small_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ Wg,
                        int T, int D, int E, int dc, float* __restrict__ planes) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float4 xs[kRouterMaxSlice];                   // x[t0 + j][d0 + i], j = 0..3
  __shared__ float2 part[kRouterWarps][kRouterTok][32];  // per-warp sums, two experts a lane
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int s = blockIdx.y;
  const int t0 = blockIdx.z * kRouterTok;
  const int d0 = s * dc;
  const int n = max(0, min(D, d0 + dc) - d0);
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    float v[kRouterTok];
#pragma unroll
    for (int j = 0; j < kRouterTok; ++j)
      v[j] = t0 + j < T ? __bfloat162float(x[static_cast<size_t>(t0 + j) * D + d0 + i]) : 0.0f;
    xs[i] = make_float4(v[0], v[1], v[2], v[3]);
  }
  __syncthreads();
  const int e = blockIdx.x * 64 + 2 * lane;  // this lane's experts e, e + 1
  const int per = (n + kRouterWarps - 1) / kRouterWarps;
  const int i0 = min(n, wid * per), i1 = min(n, i0 + per);
  float a0[kRouterTok] = {0.0f, 0.0f, 0.0f, 0.0f}, a1[kRouterTok] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (e < E) {
    const __nv_bfloat162* wp = reinterpret_cast<const __nv_bfloat162*>(Wg + static_cast<size_t>(d0) * E + e);
    const size_t stride = static_cast<size_t>(E) / 2;  // one W_g row in bf16 pairs
    for (int i = i0; i < i1; i += kRouterUnroll) {
      __nv_bfloat162 w[kRouterUnroll];
#pragma unroll
      for (int u = 0; u < kRouterUnroll; ++u)
        w[u] = i + u < i1 ? wp[static_cast<size_t>(i + u) * stride] : __floats2bfloat162_rn(0.0f, 0.0f);
#pragma unroll
      for (int u = 0; u < kRouterUnroll; ++u) {
        if (i + u < i1) {
          const float2 wf = __bfloat1622float2(w[u]);
          const float4 xv = xs[i + u];
          a0[0] = fmaf(xv.x, wf.x, a0[0]);
          a0[1] = fmaf(xv.y, wf.x, a0[1]);
          a0[2] = fmaf(xv.z, wf.x, a0[2]);
          a0[3] = fmaf(xv.w, wf.x, a0[3]);
          a1[0] = fmaf(xv.x, wf.y, a1[0]);
          a1[1] = fmaf(xv.y, wf.y, a1[1]);
          a1[2] = fmaf(xv.z, wf.y, a1[2]);
          a1[3] = fmaf(xv.w, wf.y, a1[3]);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kRouterTok; ++j) part[wid][j][lane] = make_float2(a0[j], a1[j]);
  __syncthreads();
  if (wid < kRouterTok) {  // warp j writes token t0 + j
    const int t = t0 + wid;
    if (t < T && e < E) {
      float2 sum = part[0][wid][lane];
#pragma unroll
      for (int w = 1; w < kRouterWarps; ++w) {
        sum.x += part[w][wid][lane].x;
        sum.y += part[w][wid][lane].y;
      }
      float* o = planes + (static_cast<size_t>(s) * T + t) * E + e;
      o[0] = sum.x;
      o[1] = sum.y;
    }
  }
}

// ------------------------------------------------------------------------
// init_routing ("CANN/cann-recipes-infer：Qwen3-MoE优化", section
// "GMM使能和Routing优化": npu_moe_init_routing + npu_moe_compute_expert_tokens).
// A stable counting sort of the expanded rows r = t*k + j by expert id, in two
// kernels over segments of `seg` consecutive rows:
//  1. route_hist_kernel: one block per segment writes its expert histogram
//     seg_hist[s][e] (segment-major).
//  2. route_scatter_kernel: one block per segment sums the histograms of all
//     segments (counts), scans them over experts (offsets; block 0 publishes
//     both), adds the histograms of earlier segments (its base position per
//     expert), and scatters its rows in order: the segment is cut into one
//     contiguous piece per warp, per-warp expert counts give each warp's start,
//     and inside a warp equal ids of a 32-row step are ranked with
//     __match_any_sync.  Rows with an id outside [0, E) are skipped (dest -1).
__global__ void route_hist_kernel(const int32_t* __restrict__ ids, int R, int E, int seg,
                                  int32_t* __restrict__ seg_hist, int32_t* err) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ int32_t cnt[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int s = blockIdx.x;
  const int r0 = s * seg, r1 = min(R, r0 + seg);
  bool bad = false;
  for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
    const int e = ids[r];
    if (e < 0 || e >= E) bad = true;
    else atomicAdd(&cnt[e], 1);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(err, MOE_DEV_BAD_EXPERT_ID);
  for (int e = threadIdx.x; e < E; e += blockDim.x) seg_hist[static_cast<size_t>(s) * E + e] = cnt[e];
}

constexpr int kScatterWarps = 8;

__global__ void __launch_bounds__(kScatterWarps * 32)
    route_scatter_kernel(const int32_t* __restrict__ ids, int R, int E, int seg, int nseg,
                         const int32_t* __restrict__ seg_hist, int32_t* __restrict__ counts,
                         int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_rows,
                         int32_t* __restrict__ dest) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ int32_t sm[];
  int32_t* base = sm;                    // [E] first position of this segment's rows of e
  int32_t* wcnt = sm + E;                // [kScatterWarps][E] per-warp counts, then starts
  __shared__ int32_t warp_tot[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int s = blockIdx.x;
  const int nthr = blockDim.x;

  // (a) per expert: rows in earlier segments and in all segments
  int tot_local[2], pre_local[2];  // E <= 512 and 256 threads: at most 2 experts per thread
  const int per = (E + nthr - 1) / nthr;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (i >= per) break;
    const int e = threadIdx.x + i * nthr;
    int pre = 0, tot = 0;
    if (e < E) {
      for (int q = 0; q < nseg; ++q) {
        const int v = seg_hist[static_cast<size_t>(q) * E + e];
        if (q < s) pre += v;
        tot += v;
      }
    }
    pre_local[i] = pre;
    tot_local[i] = tot;
  }
  // (b) exclusive scan of tot over e (thread-major: e = tid + i * nthr)
  //     done as a scan over the flattened order e = 0..E-1 with per = 1 or 2
  //     items per thread; items are visited in e order by a two-pass scan.
  int carry = 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (i >= per) break;
    const int e = threadIdx.x + i * nthr;
    const int v = (e < E) ? tot_local[i] : 0;
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(FULL, incl, d);
      if (lane >= d) incl += y;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    int wbase = 0, all = 0;
    for (int w = 0; w < nthr / 32; ++w) {
      const int t = warp_tot[w];
      if (w < wid) wbase += t;
      all += t;
    }
    const int excl = carry + wbase + incl - v;
    if (e < E) {
      base[e] = excl + pre_local[i];
      if (s == 0) {
        counts[e] = v;
        offsets[e] = excl;
      }
    }
    carry += all;
    __syncthreads();
  }
  if (s == 0 && threadIdx.x == 0) offsets[E] = carry;

  // (c) per-warp counts inside this segment, then per-warp start positions
  for (int i = threadIdx.x; i < kScatterWarps * E; i += nthr) wcnt[i] = 0;
  __syncthreads();
  const int r0 = s * seg, r1 = min(R, r0 + seg);
  const int piece = (seg + kScatterWarps - 1) / kScatterWarps;
  const int w0 = min(r1, r0 + wid * piece), w1 = min(r1, w0 + piece);
  for (int r = w0 + lane; r < w1; r += 32) {
    const int e = ids[r];
    if (e >= 0 && e < E) atomicAdd(&wcnt[wid * E + e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += nthr) {
    int run = base[e];
    for (int w = 0; w < kScatterWarps; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();

  // (d) ordered scatter of each warp's piece
  int32_t* my = wcnt + wid * E;
  const unsigned lt = (1u << lane) - 1u;
  for (int rb = w0; rb < w1; rb += 32) {
    const int r = rb + lane;
    const bool in = r < w1;
    const int e = in ? ids[r] : -1;
    const bool valid = in && e >= 0 && e < E;
    if (in && !valid) dest[r] = -1;
    const int key = valid ? e : -1 - lane;  // invalid rows never match anything
    const unsigned peers = __match_any_sync(FULL, key);
    if (valid) {
      const int pos = my[e] + __popc(peers & lt);
      sorted_rows[pos] = r;
      dest[r] = pos;
    }
    __syncwarp();
    if (valid && (peers & lt) == 0) my[e] += __popc(peers);
    __syncwarp();
  }
}

// ------------------------------------------------------------------------
// init_routing in one launch for larger batches: one cluster of kSortCtas
// CTAs.  CTA c takes the expanded rows [c R / n, (c + 1) R / n), each of its
// warps a contiguous piece of them, and counts them per warp and expert in
// shared memory; after a cluster barrier every CTA reads the others' expert
// histograms through distributed shared memory and adds those of the CTAs
// before it (its base position per expert) and of all of them (counts),
// scans the counts over experts (offsets; CTA 0 publishes both) and scatters
// its rows in order as route_scatter_kernel does.  The same stable counting
// sort as route_hist_kernel + route_scatter_kernel, without their global
// histogram round trip.  A CTA leaves only after every CTA has finished
// reading the others' histograms (split cluster barrier).
constexpr int kSortCtas = 8;
constexpr int kSortWarps = 32;
constexpr int kSortBatch = 8;  // ids per lane held in registers: 256 rows of a warp's piece

__global__ void __launch_bounds__(kSortWarps * 32, 1)
    route_sort_cluster_kernel(const int32_t* __restrict__ ids, int R, int E,
                              int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                              int32_t* __restrict__ sorted_rows, int32_t* __restrict__ dest,
                              int32_t* err) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ int32_t sm[];
  int32_t* wcnt = sm;                      // [kSortWarps][E]: per-warp counts, then starts
  int32_t* cta_tot = sm + kSortWarps * E;  // [E]: this CTA's histogram (read by the others)
  __shared__ int32_t warp_sum[kSortWarps];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nthr = blockDim.x;
  const int c = static_cast<int>(cluster_ctarank());
  const int r0 = static_cast<int>(static_cast<long long>(c) * R / kSortCtas);
  const int r1 = static_cast<int>(static_cast<long long>(c + 1) * R / kSortCtas);

  // (a) per-warp counts of each warp's contiguous piece, then the CTA's
  // histogram.  A warp reads its ids in batches of 32 x kSortBatch rows, all
  // loads of a batch in flight together; a piece of at most one batch keeps
  // its ids in registers for the scatter.
  for (int i = threadIdx.x; i < kSortWarps * E; i += nthr) wcnt[i] = 0;
  const int piece = (r1 - r0 + kSortWarps - 1) / kSortWarps;
  const int w0 = min(r1, r0 + wid * piece), w1 = min(r1, w0 + piece);
  int idv[kSortBatch];
  auto load_batch = [&](int rb) {
#pragma unroll
    for (int j = 0; j < kSortBatch; ++j) {
      const int r = rb + 32 * j + lane;
      idv[j] = r < w1 ? __ldg(ids + r) : -1;
    }
  };
  __syncthreads();
  bool bad = false;
  for (int rb = w0; rb < w1; rb += 32 * kSortBatch) {
    load_batch(rb);
#pragma unroll
    for (int j = 0; j < kSortBatch; ++j) {
      const int r = rb + 32 * j + lane;
      if (r < w1) {
        const int e = idv[j];
        if (e >= 0 && e < E) atomicAdd(&wcnt[wid * E + e], 1);
        else bad = true;
      }
    }
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(err, MOE_DEV_BAD_EXPERT_ID);
  for (int e = threadIdx.x; e < E; e += nthr) {
    int sum = 0;
#pragma unroll 8
    for (int w = 0; w < kSortWarps; ++w) sum += wcnt[w * E + e];
    cta_tot[e] = sum;
  }
  cluster_sync();  // every CTA's histogram is complete

  // (b) per expert e = thread (E <= 512 < threads): rows in earlier CTAs and
  // in all of them; the loads from the other CTAs are issued together
  const int e = threadIdx.x;
  int pre = 0, tot = 0;
  if (e < E) {
    int v[kSortCtas];
#pragma unroll
    for (int q = 0; q < kSortCtas; ++q)
      v[q] = ld_cluster_s32(mapa_shared(&cta_tot[e], static_cast<uint32_t>(q)));
#pragma unroll
    for (int q = 0; q < kSortCtas; ++q) {
      if (q < c) pre += v[q];
      tot += v[q];
    }
  }
  cluster_arrive_release();  // this thread is done with the other CTAs' memory
  // exclusive scan of tot over experts
  int incl = tot;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(FULL, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) warp_sum[wid] = incl;
  __syncthreads();
  int wbase = 0, all = 0;
  for (int w = 0; w < nthr / 32; ++w) {
    const int t = warp_sum[w];
    if (w < wid) wbase += t;
    all += t;
  }
  const int excl = wbase + incl - tot;
  // (c) start position of every warp's rows of each expert
  if (e < E) {
    if (c == 0) {
      counts[e] = tot;
      offsets[e] = excl;
    }
    int run = excl + pre;
#pragma unroll 8
    for (int w = 0; w < kSortWarps; ++w) {
      const int cnt = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += cnt;
    }
  }
  if (c == 0 && threadIdx.x == 0) offsets[E] = all;
  __syncthreads();

  // (d) ordered scatter of each warp's piece, 32 consecutive rows per step;
  // inside a step, equal ids are ranked by lane with __match_any_sync
  int32_t* my = wcnt + wid * E;
  const unsigned lt = (1u << lane) - 1u;
  const bool one_batch = w1 - w0 <= 32 * kSortBatch;
  for (int rb = w0; rb < w1; rb += 32 * kSortBatch) {
    if (!one_batch) load_batch(rb);
#pragma unroll
    for (int j = 0; j < kSortBatch; ++j) {
      if (rb + 32 * j >= w1) break;  // warp-uniform
      const int r = rb + 32 * j + lane;
      const bool in = r < w1;
      const int id = idv[j];
      const bool valid = in && id >= 0 && id < E;
      if (in && !valid) dest[r] = -1;
      const int key = valid ? id : -1 - lane;  // invalid rows never match anything
      const unsigned peers = __match_any_sync(FULL, key);
      if (valid) {
        const int pos = my[id] + __popc(peers & lt);
        sorted_rows[pos] = r;
        dest[r] = pos;
      }
      __syncwarp();
      if (valid && (peers & lt) == 0) my[id] += __popc(peers);
      __syncwarp();
    }
  }
  cluster_wait_acquire();  // no CTA leaves while another may read its histogram
}

// ------------------------------------------------------------------------
// init_routing after the fused router (router_sm103.cu), which also writes
// the expert histogram of each of its CTAs' tokens: chunk_hist[b][e] = rows of
// expert e among the rows [b * chunk_rows, (b + 1) * chunk_rows).  CTA b of
// this grid takes the same rows: it adds, per expert, the histograms of the
// chunks before it (its base position) and of all of them (counts), scans the
// counts over experts (offsets; CTA 0 publishes both), and scatters its rows
// in order as route_scatter_kernel does.  The same stable counting sort as
// the other init_routing kernels, with no cluster or grid-wide wait.  A CTA
// takes cpb consecutive chunks, so that the grid stays at about 32 CTAs:
// with one CTA per chunk (64-128) the sort waited for SMs held by the shared
// expert's GEMMs on the side stream (Gemma-4-style prefill: 460 -> 467 us a
// layer).  A position outside [0, R) (histograms that do not match the ids)
// is never written: the row gets dest = -1 and MOE_DEV_BAD_DEST is flagged.
constexpr int kChunkThreads = 512;
constexpr int kChunkWarps = kChunkThreads / 32;
constexpr int kChunkCtas = 32;        // about this many CTAs
constexpr int kChunkMaxRows = 8192;   // rows of one CTA (its ids in shared memory)

size_t chunk_sort_smem(int E, int cta_rows) {
  const int ngrp = kChunkThreads / (E / 4);
  return (2 * static_cast<size_t>(ngrp) * E + static_cast<size_t>(kChunkWarps) * E + cta_rows) *
         sizeof(int32_t);
}

__global__ void __launch_bounds__(kChunkThreads)
    route_sort_chunks_kernel(const int32_t* __restrict__ ids, int R, int E, int nchunks,
                             int chunk_rows, int cpb, const int32_t* __restrict__ chunk_hist,
                             int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                             int32_t* __restrict__ sorted_rows, int32_t* __restrict__ dest,
                             int32_t* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int c0 = b * cpb;  // first chunk of this CTA
  const long long r0 = static_cast<long long>(c0) * chunk_rows;
  const int n = static_cast<int>(max(0LL, min(static_cast<long long>(cpb) * chunk_rows, R - r0)));
  if (n == 0 && b != 0) return;  // nothing to sort (CTA 0 still publishes counts / offsets)
  extern __shared__ int32_t sm[];
  const int E4 = E >> 2;                  // 16-byte columns of a histogram row (E % 4 == 0)
  const int ngrp = kChunkThreads / E4;    // >= 4 chunk groups (E <= 512)
  int32_t* part = sm;                     // [2][ngrp][E]: partial sums before b / over all
  int32_t* wcnt = part + 2 * ngrp * E;    // [kChunkWarps][E]: per-warp counts, then starts
  int32_t* ids_s = wcnt + kChunkWarps * E;  // [cpb * chunk_rows]: this CTA's expert ids
  __shared__ int32_t warp_sum[kChunkWarps];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;

  // (a) each thread sums four experts over every ngrp-th chunk (16-byte loads)
  {
    const int col = tid % E4, grp = tid / E4;
    if (grp < ngrp) {
      int4 pre = make_int4(0, 0, 0, 0), tot = make_int4(0, 0, 0, 0);
#pragma unroll 8
      for (int c = grp; c < nchunks; c += ngrp) {
        const int4 v = __ldg(reinterpret_cast<const int4*>(chunk_hist + static_cast<size_t>(c) * E) + col);
        tot.x += v.x; tot.y += v.y; tot.z += v.z; tot.w += v.w;
        if (c < c0) {
          pre.x += v.x; pre.y += v.y; pre.z += v.z; pre.w += v.w;
        }
      }
      reinterpret_cast<int4*>(part + grp * E)[col] = pre;
      reinterpret_cast<int4*>(part + (ngrp + grp) * E)[col] = tot;
    }
  }
  for (int i = tid; i < n; i += kChunkThreads) ids_s[i] = ids[r0 + i];
  for (int i = tid; i < kChunkWarps * E; i += kChunkThreads) wcnt[i] = 0;
  __syncthreads();

  // (b) per expert e = thread: base position and count; exclusive scan of
  // the counts over experts
  const int e = tid;
  int pre = 0, tot = 0;
  if (e < E) {
    for (int g = 0; g < ngrp; ++g) {
      pre += part[g * E + e];
      tot += part[(ngrp + g) * E + e];
    }
  }
  int incl = tot;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(FULL, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) warp_sum[wid] = incl;

  // (c) warp w counts its piece of the chunk's rows per expert
  const int piece = (n + kChunkWarps - 1) / kChunkWarps;
  const int w0 = min(n, wid * piece), w1 = min(n, w0 + piece);
  bool bad = false;
  for (int r = w0 + lane; r < w1; r += 32) {
    const int id = ids_s[r];
    if (id >= 0 && id < E) atomicAdd(&wcnt[wid * E + id], 1);
    else bad = true;
  }
  if (__syncthreads_or(bad) && tid == 0) atomicOr(err, MOE_DEV_BAD_EXPERT_ID);
  int wbase = 0, all = 0;
  for (int w = 0; w < kChunkWarps; ++w) {
    const int t = warp_sum[w];
    if (w < wid) wbase += t;
    all += t;
  }
  if (e < E) {
    const int excl = wbase + incl - tot;
    if (b == 0) {
      counts[e] = tot;
      offsets[e] = excl;
    }
    // (d) start position of every warp's rows of expert e
    int run = excl + pre;
    for (int w = 0; w < kChunkWarps; ++w) {
      const int cnt = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += cnt;
    }
  }
  if (b == 0 && tid == 0) offsets[E] = all;
  __syncthreads();

  // (e) ordered scatter, 32 consecutive rows per step; inside a step, equal
  // ids are ranked by lane with __match_any_sync
  int32_t* my = wcnt + wid * E;
  const unsigned lt = (1u << lane) - 1u;
  bool bad_pos = false;
  for (int rb = w0; rb < w1; rb += 32) {
    const int r = rb + lane;
    const bool in = r < w1;
    const int id = in ? ids_s[r] : -1;
    const bool valid = in && id >= 0 && id < E;
    const int key = valid ? id : -1 - lane;  // invalid rows never match anything
    const unsigned peers = __match_any_sync(FULL, key);
    if (valid) {
      const int pos = my[id] + __popc(peers & lt);
      const bool ok = pos >= 0 && pos < R;
      if (ok) sorted_rows[pos] = static_cast<int32_t>(r0 + r);
      dest[r0 + r] = ok ? pos : -1;
      bad_pos |= !ok;
    } else if (in) {
      dest[r0 + r] = -1;
    }
    __syncwarp();
    if (valid && (peers & lt) == 0) my[id] += __popc(peers);
    __syncwarp();
  }
  if (__any_sync(FULL, bad_pos) && lane == 0) atomicOr(err, MOE_DEV_BAD_DEST);
}

// ------------------------------------------------------------------------
// init_routing and the permutation gather in one launch, for small batches
// (R <= kSmallRouteRows expanded rows; decode).  Every CTA loads all R expert
// ids into shared memory and repeats the whole stable counting sort there --
// per-warp histograms over contiguous pieces of the rows, per-expert prefix
// over warps, exclusive scan over experts, ordered scatter with
// __match_any_sync inside each warp -- which at these sizes costs less than
// a kernel boundary.  CTA 0 writes counts / offsets / sorted_rows / dest;
// then all CTAs copy their share of the permuted rows, taking the order from
// their own shared-memory copy.  Same results as route_hist_kernel +
// route_scatter_kernel + permute_gather_kernel (positions past the last
// valid row, which exist only when ids were invalid, get zero rows).
constexpr int kSmallRouteThreads = 1024;

__global__ void __launch_bounds__(kSmallRouteThreads, 1)
    route_permute_small_kernel(const int32_t* __restrict__ ids, int R, int E, int k, int T,
                               int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                               int32_t* __restrict__ sorted_rows, int32_t* __restrict__ dest,
                               const uint4* __restrict__ x, int vec_per_row,
                               uint4* __restrict__ x_perm, const float* __restrict__ tok_scale,
                               float* __restrict__ row_scale, int32_t* err, int extra) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ int32_t sm[];
  int32_t* ids_s = sm;               // [R] expert of each row (-1: invalid)
  int32_t* sorted_s = sm + R;        // [R] row at each permuted position
  int32_t* wcnt = sm + 2 * R;        // [32][E] per-warp counts, then per-warp starts
  int32_t* off_s = wcnt + 32 * E;    // [E + 1] expert offsets
  __shared__ int32_t warp_tot[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const bool writer = blockIdx.x == 0;

  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
  bool bad = false;
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    int e = ids[r];
    if (e < 0 || e >= E) {
      bad = true;
      e = -1;
    }
    ids_s[r] = e;
  }
  if (__syncthreads_or(bad) && writer && threadIdx.x == 0) atomicOr(err, MOE_DEV_BAD_EXPERT_ID);
  // (a) warp w counts rows [w0, w1) per expert
  const int piece = (R + 31) / 32;
  const int w0 = min(R, wid * piece), w1 = min(R, w0 + piece);
  for (int r = w0 + lane; r < w1; r += 32) {
    const int e = ids_s[r];
    if (e >= 0) atomicAdd(&wcnt[wid * E + e], 1);
  }
  __syncthreads();
  // (b) per expert: start of each warp's rows among the expert's rows; total
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
    off_s[e] = run;
  }
  __syncthreads();
  // (c) exclusive scan of the totals over experts (E <= blockDim.x)
  {
    const int e = threadIdx.x;
    const int v = e < E ? off_s[e] : 0;
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(FULL, incl, d);
      if (lane >= d) incl += y;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    int wbase = 0;
    for (int w = 0; w < wid; ++w) wbase += warp_tot[w];
    if (e < E) {
      off_s[e] = wbase + incl - v;
      if (writer) {
        counts[e] = v;
        offsets[e] = wbase + incl - v;
      }
    }
    if (e == E - 1) {
      off_s[E] = wbase + incl;
      if (writer) offsets[E] = wbase + incl;
    }
  }
  __syncthreads();
  // (d) ordered scatter of each warp's piece
  const unsigned lt = (1u << lane) - 1u;
  int32_t* my = wcnt + wid * E;
  for (int rb = w0; rb < w1; rb += 32) {
    const int r = rb + lane;
    const bool in = r < w1;
    const int e = in ? ids_s[r] : -1;
    const bool valid = e >= 0;
    if (in && !valid && writer) dest[r] = -1;
    const int key = valid ? e : -1 - lane;  // invalid rows never match anything
    const unsigned peers = __match_any_sync(FULL, key);
    if (valid) {
      const int pos = off_s[e] + my[e] + __popc(peers & lt);
      sorted_s[pos] = r;
      if (writer) {
        sorted_rows[pos] = r;
        dest[r] = pos;
      }
    }
    __syncwarp();
    if (valid && (peers & lt) == 0) my[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  if (!x) return;
  // (e) gather: one warp per permuted row, grid-strided over all CTAs; with
  // extra = T, rows R + t are copies of the tokens in order (the shared
  // expert's rows when it runs as the last group of the routed GEMMs)
  const int nvalid = off_s[E];
  const long long wstride = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long p = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + wid; p < R + extra;
       p += wstride) {
    uint4* dst = x_perm + p * vec_per_row;
    if (p < R && p >= nvalid) {
      if (row_scale && lane == 0) row_scale[p] = 0.0f;
      for (int v = lane; v < vec_per_row; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const int t = p < R ? sorted_s[p] / k : static_cast<int>(p - R);  // a valid row: t < T
    if (row_scale && lane == 0) row_scale[p] = tok_scale[t];
    const uint4* src = x + static_cast<long long>(t) * vec_per_row;
    int v = lane;
    for (; v + 96 < vec_per_row; v += 128) {
      const uint4 a = src[v], b = src[v + 32], c = src[v + 64], d = src[v + 96];
      dst[v] = a;
      dst[v + 32] = b;
      dst[v + 64] = c;
      dst[v + 96] = d;
    }
    for (; v < vec_per_row; v += 32) dst[v] = src[v];
  }
}

// ------------------------------------------------------------------------
// Permutation gather (the "千问 3.5 MoE 在 TPU 上的系统优化实战" SparseCore
// paragraph: rows gathered by routing index into one contiguous buffer).
// One warp per permuted row, 16-byte vectors.
// extra = T: rows R + t of x_perm are copies of the tokens in order (the
// shared expert's rows when it runs as the last group of the routed GEMMs).
__global__ void permute_gather_kernel(const uint4* __restrict__ x,
                                      const int32_t* __restrict__ sorted_rows, int R, int k, int T,
                                      int vec_per_row, uint4* __restrict__ x_perm,
                                      const float* __restrict__ tok_scale,
                                      float* __restrict__ row_scale, int32_t* err, int extra) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long wstride = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long p = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       p < R + extra; p += wstride) {
    const int r = p < R ? sorted_rows[p] : static_cast<int>((p - R) * k);
    const int t = r / k;
    uint4* dst = x_perm + p * vec_per_row;
    if (r < 0 || t >= T) {
      if (lane == 0) {
        atomicOr(err, MOE_DEV_BAD_DEST);
        if (row_scale) row_scale[p] = 0.0f;
      }
      for (int v = lane; v < vec_per_row; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
      continue;
    }
    if (row_scale && lane == 0) row_scale[p] = tok_scale[t];
    const uint4* src = x + static_cast<long long>(t) * vec_per_row;
    int v = lane;
    for (; v + 96 < vec_per_row; v += 128) {
      const uint4 a = src[v], b = src[v + 32], c = src[v + 64], d = src[v + 96];
      dst[v] = a;
      dst[v + 32] = b;
      dst[v + 64] = c;
      dst[v + 96] = d;
    }
    for (; v < vec_per_row; v += 32) dst[v] = src[v];
  }
  pdl_launch_dependents();  // after the copy: long kernel, see finalize_kernel
}

// The same permutation driven from the token side: each warp item is one
// token's slice of 256 16-byte chunks, read once and written to the token's k
// permuted rows (dest[t*k + j]); positions past the last valid row (only
// when ids were invalid) are zero-filled.  Reads x once instead of k times,
// which matters when x is larger than L2 (every row would come from HBM k
// times).
constexpr int kScatterSlice = 256;

// extra = T: each token's row is also written to R + t (the shared expert's
// rows when it runs as the last group of the routed GEMMs).
__global__ void permute_scatter_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ dest,
                                       const int32_t* __restrict__ nvalid_ptr, int R, int k, int T,
                                       int vec_per_row, uint4* __restrict__ x_perm,
                                       const float* __restrict__ tok_scale,
                                       float* __restrict__ row_scale, int32_t* err, int extra) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long wid = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const long long wstride = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const int nsl = (vec_per_row + kScatterSlice - 1) / kScatterSlice;
  const long long items = static_cast<long long>(T) * nsl;
  for (long long it = wid; it < items; it += wstride) {
    const long long t = it / nsl;
    const int sl = static_cast<int>(it - t * nsl);
    int my_p = -1;
    if (lane < k) {
      const int p = dest[t * k + lane];
      if (p >= R) atomicOr(err, MOE_DEV_BAD_DEST);
      my_p = (p >= 0 && p < R) ? p : -1;  // -1: a row whose id was invalid
    } else if (lane == k && extra > 0) {
      my_p = static_cast<int>(R + t);  // the shared expert's copy
    }
    if (sl == 0 && row_scale && my_p >= 0) row_scale[my_p] = tok_scale[t];
    const int kk = k + (extra > 0 ? 1 : 0);  // destinations of this token
    int pj[17];
#pragma unroll
    for (int j = 0; j < 17; ++j) pj[j] = __shfl_sync(FULL, my_p, j);
    const uint4* src = x + t * vec_per_row;
    const int v1 = min(vec_per_row, (sl + 1) * kScatterSlice);
    int v = sl * kScatterSlice + lane;
    for (; v + 96 < v1; v += 128) {
      const uint4 a = src[v], b = src[v + 32], c = src[v + 64], d = src[v + 96];
#pragma unroll
      for (int j = 0; j < 17; ++j) {
        if (j < kk && pj[j] >= 0) {
          uint4* dst = x_perm + static_cast<long long>(pj[j]) * vec_per_row;
          dst[v] = a;
          dst[v + 32] = b;
          dst[v + 64] = c;
          dst[v + 96] = d;
        }
      }
    }
    for (; v < v1; v += 32) {
      const uint4 a = src[v];
#pragma unroll
      for (int j = 0; j < 17; ++j)
        if (j < kk && pj[j] >= 0) x_perm[static_cast<long long>(pj[j]) * vec_per_row + v] = a;
    }
  }
  // rows past the last valid one (ids that were out of range)
  const int nvalid = max(0, min(R, *nvalid_ptr));
  for (long long p = nvalid + wid; p < R; p += wstride) {
    if (row_scale && lane == 0) row_scale[p] = 0.0f;
    for (int v = lane; v < vec_per_row; v += 32) x_perm[p * vec_per_row + v] = make_uint4(0, 0, 0, 0);
  }
  pdl_launch_dependents();  // after the copy: long kernel, see finalize_kernel
}

// ------------------------------------------------------------------------
// bf16 rows to fp16 rows with an exact power-of-two row scale, for the fp16
// tensor-core path of fp8-weight layers: row t is multiplied by 2^e_t with
// max_d |x[t, d]| * 2^e_t < 2^14, so every bf16 value in the range that
// matters converts exactly (bf16's 8 significant bits fit in fp16's 11), and
// inv_scale[t] = 2^-e_t undoes it exactly after the GEMM.  One warp per row.
__device__ __forceinline__ float exp2_int(int e) {  // exact 2^e for e in [-126, 127]
  return __int_as_float((e + 127) << 23);
}

// 8 consecutive elements of a bf16 or fp32 row as floats
__device__ __forceinline__ void load8f(const __nv_bfloat16* row, int v, float (&f)[8]) {
  const uint4 u = reinterpret_cast<const uint4*>(row)[v];
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ void load8f(const float* row, int v, float (&f)[8]) {
  const float4 a = reinterpret_cast<const float4*>(row)[2 * v];
  const float4 b = reinterpret_cast<const float4*>(row)[2 * v + 1];
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// 8 elements from their raw 16-byte words: two words of fp32, or one of bf16
__device__ __forceinline__ void unpack8(const uint4 (&u)[2], float (&f)[8]) {
  f[0] = __uint_as_float(u[0].x); f[1] = __uint_as_float(u[0].y);
  f[2] = __uint_as_float(u[0].z); f[3] = __uint_as_float(u[0].w);
  f[4] = __uint_as_float(u[1].x); f[5] = __uint_as_float(u[1].y);
  f[6] = __uint_as_float(u[1].z); f[7] = __uint_as_float(u[1].w);
}
__device__ __forceinline__ void unpack8(const uint4 (&u)[1], float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u[0]);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(h[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

// Source rows bf16 (exact conversion) or fp32 (rounded once to fp16's 11
// significant bits, relative to the row maximum's scale).
template <typename Tin>
__global__ void rows_to_fp16_kernel(const Tin* __restrict__ x, int rows, int D,
                                    __half* __restrict__ x16, float* __restrict__ inv_scale) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long wstride = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const int nvec = D / 8;
  for (long long r = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       r < rows; r += wstride) {
    const Tin* src = x + r * D;
    // row maximum: four 8-element loads in flight per lane
    float m = 0.0f;
    for (int v0 = lane; v0 < nvec; v0 += 128) {
      float f[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (v0 + 32 * u < nvec) {
          load8f(src, v0 + 32 * u, f[u]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) f[u][i] = 0.0f;
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[u][i]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, off));
    int e = 0;
    if (m > 0.0f && isfinite(m)) {
      int ex;
      frexpf(m, &ex);  // m < 2^ex
      e = min(100, max(-100, 14 - ex));
    }
    const float sc = exp2_int(e);
    if (lane == 0) inv_scale[r] = exp2_int(-e);
    uint4* dst = reinterpret_cast<uint4*>(x16 + r * D);
#pragma unroll 4
    for (int v = lane; v < nvec; v += 32) {
      float f[8];
      load8f(src, v, f);
      uint4 o;
      __half2* oh = reinterpret_cast<__half2*>(&o);
#pragma unroll
      for (int i = 0; i < 4; ++i) oh[i] = __floats2half2_rn(f[2 * i] * sc, f[2 * i + 1] * sc);
      dst[v] = o;
    }
  }
}

// Two e4m3 values (lo -> low byte) from two floats, round to nearest even,
// saturating to +-448.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// The two e4m3 values of the low 16 bits of w as floats (exact).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t w) {
  uint32_t h;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
      : "=r"(h)
      : "r"(w));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// Rows as two e4m3 terms for the 8-bit tensor-core path: per row a power of
// two 2^e puts the largest |element| in [128, 256); v = x * 2^e, hi =
// e4m3(v), lo = e4m3(v - hi) (v - hi is exact in fp32), so hi + lo = v for
// every bf16 element of magnitude at least 2^-9 of the row's largest, and
// within 2^-10 (scaled units) below that; fp32 sources keep 8 significant
// bits.  Output row r: bytes [0, D) hi, [D, 2D) lo; inv_scale[r] = 2^-e.

// the exponent e of a row whose largest magnitude is m (0 for an all-zero row)
__device__ __forceinline__ int e4m3x2_row_exp(float m) {
  int e = 0;
  if (m > 0.0f && isfinite(m)) {
    int ex;
    frexpf(m, &ex);  // 2^(ex-1) <= m < 2^ex
    e = min(100, max(-100, 8 - ex));
  }
  return e;
}

// hi and lo terms of 8 consecutive elements scaled by sc (8 bytes each)
__device__ __forceinline__ void e4m3x2_terms8(const float (&f)[8], float sc, uint2& hi, uint2& lo) {
  uint32_t hw[2] = {0u, 0u}, lw[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = f[2 * i] * sc, b = f[2 * i + 1] * sc;
    const uint32_t h = f32x2_to_e4m3x2(a, b);
    const float2 hv = e4m3x2_to_f32x2(h);
    const uint32_t l = f32x2_to_e4m3x2(a - hv.x, b - hv.y);
    hw[i >> 1] |= h << (16 * (i & 1));
    lw[i >> 1] |= l << (16 * (i & 1));
  }
  hi = make_uint2(hw[0], hw[1]);
  lo = make_uint2(lw[0], lw[1]);
}

// W8A8 rows (one e4m3 term, dynamic per-row scale): the "用SGLang-JAX在TPU上
// 优化Ling-2.6-1T" §5 activation quantisation.  s = m / 448 for a row whose
// largest |element| is m (1 for an all-zero row), code = e4m3(v / s), both
// divisions correctly rounded in fp32, round to nearest even, saturating.
__device__ __forceinline__ float e4m3_row_scale(float m) {
  return (m > 0.0f && isfinite(m)) ? __fdiv_rn(m, 448.0f) : 1.0f;
}
// the codes of 8 consecutive elements under the row scale s (8 bytes)
__device__ __forceinline__ uint2 e4m3_codes8(const float (&f)[8], float s) {
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i >> 1] |= f32x2_to_e4m3x2(__fdiv_rn(f[2 * i], s), __fdiv_rn(f[2 * i + 1], s)) << (16 * (i & 1));
  return make_uint2(w[0], w[1]);
}

// One warp per row; the row is read twice (maximum, then conversion), the
// second time mostly from cache.  For rows outside the register kernel's range.
// A8: one e4m3 term with the dynamic scale (output rows of D bytes,
// inv_scale[r] = s), else two terms with a power-of-two scale (rows of 2D
// bytes, inv_scale[r] = 2^-e).
template <typename Tin, bool A8>
__global__ void rows_to_e4m3x2_kernel(const Tin* __restrict__ x, int rows, int D,
                                      uint8_t* __restrict__ q, float* __restrict__ inv_scale) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long wstride = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const int nvec = D / 8;
  for (long long r = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       r < rows; r += wstride) {
    const Tin* src = x + r * D;
    // row maximum: four 8-element loads in flight per lane
    float m = 0.0f;
    for (int v0 = lane; v0 < nvec; v0 += 128) {
      float f[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (v0 + 32 * u < nvec) {
          load8f(src, v0 + 32 * u, f[u]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) f[u][i] = 0.0f;
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[u][i]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, off));
    if (A8) {
      const float sr = e4m3_row_scale(m);
      if (lane == 0) inv_scale[r] = sr;
      uint8_t* row = q + r * D;
#pragma unroll 4
      for (int v = lane; v < nvec; v += 32) {
        float f[8];
        load8f(src, v, f);
        *reinterpret_cast<uint2*>(row + 8 * v) = e4m3_codes8(f, sr);
      }
      continue;
    }
    const int e = e4m3x2_row_exp(m);
    const float sc = exp2_int(e);
    if (lane == 0) inv_scale[r] = exp2_int(-e);
    uint8_t* hi_row = q + r * 2 * D;
    uint8_t* lo_row = hi_row + D;
#pragma unroll 4
    for (int v = lane; v < nvec; v += 32) {
      float f[8];
      load8f(src, v, f);
      uint2 hw, lw;
      e4m3x2_terms8(f, sc, hw, lw);
      *reinterpret_cast<uint2*>(hi_row + 8 * v) = hw;
      *reinterpret_cast<uint2*>(lo_row + 8 * v) = lw;
    }
  }
}

// The same rows, each held in registers from its maximum to its conversion,
// so that it is read from memory once: a group of 2^tpr_log2 threads (32 ..
// 256) per row, up to kRegRowVecs 8-element vectors per thread, 256 >>
// tpr_log2 rows per block.  Rows of 1024 .. 8192 elements: with a warp per
// row, the rows in flight on the whole GPU at that length outgrow the L2, and
// the second pass reads them from HBM again.
constexpr int kRegRowVecs = 4;
constexpr int kRegRowBlocksPerSm = 5;  // resident blocks at <= 48 registers, no spills
template <typename Tin, bool A8>
__global__ void __launch_bounds__(256, kRegRowBlocksPerSm) rows_to_e4m3x2_reg_kernel(
    const Tin* __restrict__ x, int rows, int D, int tpr_log2, uint8_t* __restrict__ q,
    float* __restrict__ inv_scale) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red[2][8];  // per-warp maxima, two buffers (one barrier per row)
  const int tpr = 1 << tpr_log2;
  const int rpb = 256 >> tpr_log2;
  const int g = threadIdx.x >> tpr_log2, li = threadIdx.x & (tpr - 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wpr = tpr >> 5;  // warps per row
  const int nvec = D / 8;
  int buf = 0;
  // every thread of the block runs the same iterations (the barrier below)
  for (long long base = static_cast<long long>(blockIdx.x) * rpb; base < rows;
       base += static_cast<long long>(gridDim.x) * rpb) {
    const long long r = base + g;
    const bool valid = r < rows;
    const Tin* src = x + (valid ? r : 0) * D;
    // the row's 8-element vectors as loaded (one or two 16-byte words each)
    constexpr int kWords = sizeof(Tin) == 4 ? 2 : 1;
    uint4 raw[kRegRowVecs][kWords];
#pragma unroll
    for (int j = 0; j < kRegRowVecs; ++j) {
      const int v = li + tpr * j;
#pragma unroll
      for (int w = 0; w < kWords; ++w)
        raw[j][w] = (valid && v < nvec) ? __ldcs(reinterpret_cast<const uint4*>(src) + kWords * v + w)
                                        : make_uint4(0u, 0u, 0u, 0u);
    }
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < kRegRowVecs; ++j) {
      float f[8];
      unpack8(raw[j], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, off));
    if (lane == 0) red[buf][warp] = m;
    __syncthreads();
    m = red[buf][g * wpr];
    for (int w = 1; w < wpr; ++w) m = fmaxf(m, red[buf][g * wpr + w]);
    buf ^= 1;
    if (!valid) continue;
    if (A8) {
      const float sr = e4m3_row_scale(m);
      if (li == 0) inv_scale[r] = sr;
      uint8_t* row = q + r * D;
#pragma unroll
      for (int j = 0; j < kRegRowVecs; ++j) {
        const int v = li + tpr * j;
        if (v < nvec) {
          float f[8];
          unpack8(raw[j], f);
          *reinterpret_cast<uint2*>(row + 8 * v) = e4m3_codes8(f, sr);
        }
      }
      continue;
    }
    const int e = e4m3x2_row_exp(m);
    const float sc = exp2_int(e);
    if (li == 0) inv_scale[r] = exp2_int(-e);
    uint8_t* hi_row = q + r * 2 * D;
    uint8_t* lo_row = hi_row + D;
#pragma unroll
    for (int j = 0; j < kRegRowVecs; ++j) {
      const int v = li + tpr * j;
      if (v < nvec) {
        float f[8];
        unpack8(raw[j], f);
        uint2 hw, lw;
        e4m3x2_terms8(f, sc, hw, lw);
        *reinterpret_cast<uint2*>(hi_row + 8 * v) = hw;
        *reinterpret_cast<uint2*>(lo_row + 8 * v) = lw;
      }
    }
  }
}

// The end of the fused combine: out[t] = round(acc[t] + s[t]) (s fp32, bf16
// or absent), acc the [T, D] fp32 sums the down pass added its weighted rows
// into.  16-byte vectors of 4 elements; one rounding to bf16.
template <typename Ts>
__global__ void combine_round_kernel(const float4* __restrict__ acc, const Ts* __restrict__ s,
                                     long long n4, uint2* __restrict__ out) {
  pdl_wait();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 a = acc[i];
    if (s) {
      float f[4];
      if constexpr (sizeof(Ts) == 4) {
        const float4 v = reinterpret_cast<const float4*>(s)[i];
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
      } else {
        const uint2 u = reinterpret_cast<const uint2*>(s)[i];
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
        f[0] = lo.x; f[1] = lo.y; f[2] = hi.x; f[3] = hi.y;
      }
      a.x += f[0]; a.y += f[1]; a.z += f[2]; a.w += f[3];
    }
    __nv_bfloat162 o0 = __floats2bfloat162_rn(a.x, a.y), o1 = __floats2bfloat162_rn(a.z, a.w);
    out[i] = make_uint2(*reinterpret_cast<uint32_t*>(&o0), *reinterpret_cast<uint32_t*>(&o1));
  }
  pdl_launch_dependents();
}

// W_nk[g][n][c] = W[g][c][n] for one-byte elements: 64 x 64 tiles through
// shared memory, 16-byte loads and stores (K and N multiples of 16).
__global__ void transpose_bytes_kernel(const uint8_t* __restrict__ W, int K, int N,
                                       uint8_t* __restrict__ W_nk) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ uint8_t tile[64][64 + 16];
  const size_t g = blockIdx.z;
  const int c0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const int t = threadIdx.x;  // 256 threads: 64 rows x 4 chunks of 16 bytes
  const int r = t >> 2, ch = (t & 3) * 16;
  const uint8_t* src = W + g * K * static_cast<size_t>(N);
  if (c0 + r < K && n0 + ch < N)
    *reinterpret_cast<uint4*>(&tile[r][ch]) =
        *reinterpret_cast<const uint4*>(src + static_cast<size_t>(c0 + r) * N + n0 + ch);
  __syncthreads();
  uint8_t* dst = W_nk + g * K * static_cast<size_t>(N);
  if (n0 + r < N && c0 + ch < K) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = static_cast<uint32_t>(tile[ch + 4 * i][r]) |
             (static_cast<uint32_t>(tile[ch + 4 * i + 1][r]) << 8) |
             (static_cast<uint32_t>(tile[ch + 4 * i + 2][r]) << 16) |
             (static_cast<uint32_t>(tile[ch + 4 * i + 3][r]) << 24);
    *reinterpret_cast<uint4*>(dst + static_cast<size_t>(n0 + r) * K + c0 + ch) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ------------------------------------------------------------------------
// finalize_routing ("CANN/cann-recipes-infer：Qwen3-MoE优化", section
// "GMM使能和Routing优化") fused with the shared-expert add ("千问 3.5 MoE 在
// TPU 上的系统优化实战": y = Router(x) + SharedExpert(x)).  One warp per
// (token, m 256-column slices): m is chosen so that small batches still
// spread over every SM while large ones keep whole rows per warp; expert
// rows and shared row in fp32 (bf16 for fp8-weight layers), fp32
// accumulation with j ascending, shared row last, one rounding to the output
// type.
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&f)[8]) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void store8(float* p, const float (&f)[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
}

// Ty: the type of the expert rows and the shared row (fp32, or bf16 for
// fp8-weight layers).
template <typename Tt, int KMAX, typename Ty>
__global__ void finalize_kernel(const Ty* __restrict__ y_perm, const int32_t* __restrict__ dest,
                                const float* __restrict__ w, const Ty* __restrict__ s_rows,
                                Tt* __restrict__ out, int T, int k, int D, int R, int m,
                                int32_t* err) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long wstride = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const int nchunk = D / 8;              // 8 output elements per lane and chunk
  const int nslice = (nchunk + 31) / 32;  // 256-column slices of a row
  const int nper = (nslice + m - 1) / m;  // warp items per token: m slices each
  const long long items = static_cast<long long>(T) * nper;
  for (long long it = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       it < items; it += wstride) {
    const long long t = it / nper;
    const int s0 = static_cast<int>(it - t * nper) * m;
    // lanes < k fetch one (position, weight) pair each; a bad position is
    // flagged and replaced by row 0 with weight 0 so every load stays in bounds
    int my_p = 0;
    float my_w = 0.0f;
    if (lane < k) {
      my_p = dest[t * k + lane];
      my_w = w[t * k + lane];
      if (my_p < 0 || my_p >= R) {
        atomicOr(err, MOE_DEV_BAD_DEST);
        my_p = 0;
        my_w = 0.0f;
      }
    }
    int pj[KMAX];
    float wj[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      pj[j] = __shfl_sync(FULL, my_p, j);
      wj[j] = __shfl_sync(FULL, my_w, j);
    }
    for (int c = s0 * 32 + lane; c < min(nslice, s0 + m) * 32 && c < nchunk; c += 32) {
      // issue all k row loads before any arithmetic so they are in flight together
      // (8 elements per row: 32 bytes of fp32, or 16 bytes of bf16)
      constexpr int kVec = sizeof(Ty) == 4 ? 2 : 1;
      uint4 rv[KMAX][kVec];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < k) {
          const uint4* src = reinterpret_cast<const uint4*>(y_perm + static_cast<long long>(pj[j]) * D) + kVec * c;
#pragma unroll
          for (int q = 0; q < kVec; ++q) rv[j][q] = __ldcs(src + q);
        }
      }
      uint4 sv[kVec];
#pragma unroll
      for (int q = 0; q < kVec; ++q) sv[q] = make_uint4(0u, 0u, 0u, 0u);
      if (s_rows) {
        const uint4* src = reinterpret_cast<const uint4*>(s_rows + t * D) + kVec * c;
#pragma unroll
        for (int q = 0; q < kVec; ++q) sv[q] = __ldcs(src + q);
      }
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < k) {
          float f[8];
          unpack8(rv[j], f);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[j], f[i], acc[i]);
        }
      }
      {
        float f[8];
        unpack8(sv, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += f[i];
      }
      store8(out + t * D + c * 8, acc);
    }
  }
  // The next kernel is scheduled once every CTA got here: an earlier trigger
  // lets its CTAs wait beside this (at prefill, long) kernel's, which measured
  // slower; the short routing kernels trigger at their start.
  pdl_launch_dependents();
}

int blocks_for(long long work_items, int per_block, int cap) {
  long long b = (work_items + per_block - 1) / per_block;
  if (b < 1) b = 1;
  if (b > cap) b = cap;
  return static_cast<int>(b);
}

// Launch through launch_kernel (programmatic dependent launch when enabled);
// a failed launch returns its error from the enclosing launcher.
#define MOE_LAUNCH(kern, grid, block, smem, stream, ...)                                  \
  do {                                                                                    \
    const cudaError_t le_ = launch_kernel(kern, dim3(grid), dim3(block), smem, stream, __VA_ARGS__); \
    if (le_ != cudaSuccess) return le_;                                                   \
  } while (0)

}  // namespace

cudaError_t launch_topk_softmax(const float* partials, int nsplit, const float* bias, float* logits,
                                int T, int E, int k, int renorm, int32_t* ids, float* w,
                                int32_t* err, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int threads = 256, wpb = threads / 32;
  const int blocks = (T + wpb - 1) / wpb;
  const int epl = (E + 31) / 32;
  if (epl <= 4)
    MOE_LAUNCH(topk_softmax_kernel<4>, blocks, threads, 0, s, partials, nsplit, bias, logits, T,
               E, k, renorm, ids, w, err);
  else if (epl <= 8)
    MOE_LAUNCH(topk_softmax_kernel<8>, blocks, threads, 0, s, partials, nsplit, bias, logits, T,
               E, k, renorm, ids, w, err);
  else
    MOE_LAUNCH(topk_softmax_kernel<16>, blocks, threads, 0, s, partials, nsplit, bias, logits, T,
               E, k, renorm, ids, w, err);
  return cudaGetLastError();
}

// Up to 64 tokens and 2^25 multiply-adds (x W_g of Qwen3- and Gemma-4-style
// decode batches), with every slice staged in shared memory.
bool router_small_ok(int T, int E, int D, int nsplit) {
  if (T <= 0 || T > 64 || E <= 0 || (E & 1) || nsplit < 1) return false;
  if (static_cast<long long>(T) * D * E > (1ll << 25)) return false;
  return (D + nsplit - 1) / nsplit <= kRouterMaxSlice;
}

cudaError_t launch_router_small(const void* x, const void* Wg, int T, int D, int E, int nsplit,
                                float* planes, cudaStream_t s) {
  if (!router_small_ok(T, E, D, nsplit)) return cudaErrorInvalidValue;
  const int dc = (D + nsplit - 1) / nsplit;
  const dim3 grid((E + 63) / 64, nsplit, (T + kRouterTok - 1) / kRouterTok);
  MOE_LAUNCH(router_small_kernel, grid, kRouterWarps * 32, 0, s,
             static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(Wg), T, D, E,
             dc, planes);
  return cudaGetLastError();
}

cudaError_t launch_init_routing(const int32_t* ids, int R, int E, int32_t* counts, int32_t* offsets,
                                int32_t* sorted_rows, int32_t* dest, int32_t* seg_scratch,
                                int32_t* err, cudaStream_t s, void (*mark)(cudaStream_t)) {
  if (R <= 0) {
    cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s);
    if (e != cudaSuccess) return e;
    return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s);
  }
  const int seg = route_segment_rows(R);
  const int nseg = (R + seg - 1) / seg;
  if (mark) mark(s);
  MOE_LAUNCH(route_hist_kernel, nseg, 256, E * sizeof(int32_t), s, ids, R, E, seg, seg_scratch, err);
  if (mark) mark(s);
  const size_t smem = (1 + kScatterWarps) * E * sizeof(int32_t);
  MOE_LAUNCH(route_scatter_kernel, nseg, kScatterWarps * 32, smem, s, ids, R, E, seg, nseg,
             seg_scratch, counts, offsets, sorted_rows, dest);
  return cudaGetLastError();
}

cudaError_t launch_route_sort_cluster(const int32_t* ids, int R, int E, int32_t* counts,
                                      int32_t* offsets, int32_t* sorted_rows, int32_t* dest,
                                      int32_t* err, cudaStream_t s) {
  if (R <= 0 || E < 1 || E > 512) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(kSortWarps + 1) * E * sizeof(int32_t);
  static bool attr_done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(route_sort_cluster_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>((kSortWarps + 1) * 512 * sizeof(int32_t)));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kSortCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = g_pdl ? 1 : 0;
  cfg.gridDim = dim3(kSortCtas, 1, 1);
  cfg.blockDim = dim3(kSortWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, route_sort_cluster_kernel, ids, R, E, counts, offsets,
                                     sorted_rows, dest, err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_route_sort_chunks(const int32_t* ids, int R, int E, int nchunks, int chunk_rows,
                                     const int32_t* chunk_hist, int32_t* counts, int32_t* offsets,
                                     int32_t* sorted_rows, int32_t* dest, int32_t* err,
                                     cudaStream_t s) {
  if (R <= 0 || E < 8 || E > 512 || (E % 4) || nchunks <= 0 || chunk_rows <= 0 ||
      chunk_rows > kChunkMaxRows || static_cast<long long>(nchunks) * chunk_rows < R || !chunk_hist ||
      (reinterpret_cast<uintptr_t>(chunk_hist) & 15))
    return cudaErrorInvalidValue;
  const int cpb = std::max(1, std::min((nchunks + kChunkCtas - 1) / kChunkCtas,
                                       kChunkMaxRows / chunk_rows));
  const int ctas = (nchunks + cpb - 1) / cpb;
  const size_t smem = chunk_sort_smem(E, cpb * chunk_rows);
  static bool attr_done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    // the largest request: E = 512 (4 chunk groups), kChunkMaxRows rows
    cudaError_t e = cudaFuncSetAttribute(route_sort_chunks_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(chunk_sort_smem(512, kChunkMaxRows)));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = g_pdl ? 1 : 0;
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(kChunkThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, route_sort_chunks_kernel, ids, R, E, nchunks, chunk_rows,
                                     cpb, chunk_hist, counts, offsets, sorted_rows, dest, err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_route_permute_small(const int32_t* ids, int R, int E, int k, int T,
                                       int32_t* counts, int32_t* offsets, int32_t* sorted_rows,
                                       int32_t* dest, const void* x, size_t row_bytes,
                                       void* x_perm, const float* tok_scale, float* row_scale,
                                       int32_t* err, cudaStream_t s, int extra_rows) {
  if (R <= 0 || !small_route(R, E)) return cudaErrorInvalidValue;
  const size_t smem = (2 * static_cast<size_t>(R) + 33 * static_cast<size_t>(E) + 1) * sizeof(int32_t);
  static bool attr_done[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    const size_t max_smem = (2 * static_cast<size_t>(kSmallRouteRows) + 33 * 512 + 1) * sizeof(int32_t);
    cudaError_t e = cudaFuncSetAttribute(route_permute_small_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(max_smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  const int blocks = x ? blocks_for(R + (x ? extra_rows : 0), 32, device_sm_count()) : 1;
  MOE_LAUNCH(route_permute_small_kernel, blocks, kSmallRouteThreads, smem, s, ids, R, E, k, T,
             counts, offsets, sorted_rows, dest, static_cast<const uint4*>(x),
             static_cast<int>(row_bytes / 16), static_cast<uint4*>(x_perm), tok_scale, row_scale,
             err, x ? extra_rows : 0);
  return cudaGetLastError();
}

cudaError_t launch_permute_gather(const void* x, const int32_t* sorted_rows, int R, int k, int T,
                                  size_t row_bytes, void* x_perm, int32_t* err, cudaStream_t s,
                                  const float* tok_scale, float* row_scale, int extra_rows) {
  if (R <= 0) return cudaSuccess;
  const int vec = static_cast<int>(row_bytes / 16);
  const int threads = 256;
  const int blocks = blocks_for(R + extra_rows, threads / 32, device_sm_count() * 16);
  MOE_LAUNCH(permute_gather_kernel, blocks, threads, 0, s, static_cast<const uint4*>(x),
             sorted_rows, R, k, T, vec, static_cast<uint4*>(x_perm), tok_scale, row_scale, err,
             extra_rows);
  return cudaGetLastError();
}

cudaError_t launch_permute_scatter(const void* x, const int32_t* dest, const int32_t* nvalid,
                                   int R, int k, int T, size_t row_bytes, void* x_perm,
                                   int32_t* err, cudaStream_t s, const float* tok_scale,
                                   float* row_scale, int extra_rows) {
  if (R <= 0) return cudaSuccess;
  if (k > 16) return cudaErrorInvalidValue;
  const int vec = static_cast<int>(row_bytes / 16);
  const int threads = 256;
  const long long items = static_cast<long long>(T) * ((vec + kScatterSlice - 1) / kScatterSlice);
  const int blocks = blocks_for(items, threads / 32, device_sm_count() * 16);
  MOE_LAUNCH(permute_scatter_kernel, blocks, threads, 0, s, static_cast<const uint4*>(x), dest,
             nvalid, R, k, T, vec, static_cast<uint4*>(x_perm), tok_scale, row_scale, err,
             extra_rows);
  return cudaGetLastError();
}

cudaError_t launch_rows_to_fp16(const void* x, int rows, int D, void* x16, float* inv_scale,
                                cudaStream_t s, bool src_f32) {
  if (rows <= 0) return cudaSuccess;
  const int threads = 256;
  const int blocks = blocks_for(rows, threads / 32, device_sm_count() * 16);
  if (src_f32)
    MOE_LAUNCH(rows_to_fp16_kernel<float>, blocks, threads, 0, s, static_cast<const float*>(x),
               rows, D, static_cast<__half*>(x16), inv_scale);
  else
    MOE_LAUNCH(rows_to_fp16_kernel<__nv_bfloat16>, blocks, threads, 0, s,
               static_cast<const __nv_bfloat16*>(x), rows, D, static_cast<__half*>(x16), inv_scale);
  return cudaGetLastError();
}

namespace {
template <bool A8>
cudaError_t launch_rows_e4m3(const void* x, int rows, int D, void* q, float* inv_scale,
                             cudaStream_t s, bool src_f32) {
  if (rows <= 0) return cudaSuccess;
  const int threads = 256;
  const int nvec = D / 8;
  if (nvec >= 128 && nvec <= 256 * kRegRowVecs) {
    int tpr_log2 = 5;  // the smallest group that holds the row: 32 .. 256 threads
    while ((1 << tpr_log2) * kRegRowVecs < nvec) ++tpr_log2;
    const int blocks =
        blocks_for(rows, threads >> tpr_log2, device_sm_count() * kRegRowBlocksPerSm);
    if (src_f32)
      MOE_LAUNCH((rows_to_e4m3x2_reg_kernel<float, A8>), blocks, threads, 0, s,
                 static_cast<const float*>(x), rows, D, tpr_log2, static_cast<uint8_t*>(q),
                 inv_scale);
    else
      MOE_LAUNCH((rows_to_e4m3x2_reg_kernel<__nv_bfloat16, A8>), blocks, threads, 0, s,
                 static_cast<const __nv_bfloat16*>(x), rows, D, tpr_log2,
                 static_cast<uint8_t*>(q), inv_scale);
    return cudaGetLastError();
  }
  const int blocks = blocks_for(rows, threads / 32, device_sm_count() * 16);
  if (src_f32)
    MOE_LAUNCH((rows_to_e4m3x2_kernel<float, A8>), blocks, threads, 0, s,
               static_cast<const float*>(x), rows, D, static_cast<uint8_t*>(q), inv_scale);
  else
    MOE_LAUNCH((rows_to_e4m3x2_kernel<__nv_bfloat16, A8>), blocks, threads, 0, s,
               static_cast<const __nv_bfloat16*>(x), rows, D, static_cast<uint8_t*>(q), inv_scale);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_rows_to_e4m3x2(const void* x, int rows, int D, void* q, float* inv_scale,
                                  cudaStream_t s, bool src_f32) {
  return launch_rows_e4m3<false>(x, rows, D, q, inv_scale, s, src_f32);
}

cudaError_t launch_rows_to_e4m3(const void* x, int rows, int D, void* q, float* scale,
                                cudaStream_t s, bool src_f32) {
  return launch_rows_e4m3<true>(x, rows, D, q, scale, s, src_f32);
}

cudaError_t launch_combine_round(const float* acc, const void* s_rows, bool s_bf16, int T, int D,
                                 void* out, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (D % 4) return cudaErrorInvalidValue;
  const long long n4 = static_cast<long long>(T) * D / 4;
  const int threads = 256;
  const int blocks = static_cast<int>(std::min<long long>((n4 + threads - 1) / threads,
                                                          static_cast<long long>(device_sm_count()) * 8));
  if (s_bf16)
    MOE_LAUNCH(combine_round_kernel<__nv_bfloat16>, blocks, threads, 0, s,
               reinterpret_cast<const float4*>(acc), static_cast<const __nv_bfloat16*>(s_rows), n4,
               static_cast<uint2*>(out));
  else
    MOE_LAUNCH(combine_round_kernel<float>, blocks, threads, 0, s, reinterpret_cast<const float4*>(acc),
               static_cast<const float*>(s_rows), n4, static_cast<uint2*>(out));
  return cudaGetLastError();
}

cudaError_t launch_transpose_bytes(const void* W, long long G, int K, int N, void* W_nk,
                                   cudaStream_t s) {
  if (G <= 0) return cudaSuccess;
  const dim3 grid((N + 63) / 64, (K + 63) / 64, static_cast<unsigned>(G));
  MOE_LAUNCH(transpose_bytes_kernel, grid, 256, 0, s, static_cast<const uint8_t*>(W), K, N,
             static_cast<uint8_t*>(W_nk));
  return cudaGetLastError();
}

cudaError_t launch_finalize(int act_dtype, const void* y_perm, const int32_t* dest, const float* w,
                            const void* s_rows, void* out, int T, int k, int D, int R,
                            int32_t* err, cudaStream_t s, bool y_bf16) {
  if (T <= 0) return cudaSuccess;
  const int threads = 256;
  // warp items of m 256-column slices: whole rows (measured fastest) when
  // there are enough tokens for ~16 warps per SM, else rows halved until
  // there are (single slices for decode batches)
  const int nslice = (D / 8 + 31) / 32;
  const long long target = static_cast<long long>(device_sm_count()) * 16;
  int m = nslice;
  while (m > 1 && static_cast<long long>(T) * ((nslice + m - 1) / m) < target) m = (m + 1) / 2;
  const long long items = static_cast<long long>(T) * ((nslice + m - 1) / m);
  const int blocks = blocks_for(items, threads / 32, device_sm_count() * 16);
  const float* y = static_cast<const float*>(y_perm);
  const float* sr = static_cast<const float*>(s_rows);
  const __nv_bfloat16* yb = static_cast<const __nv_bfloat16*>(y_perm);
  const __nv_bfloat16* srb = static_cast<const __nv_bfloat16*>(s_rows);
#define MOE_FIN(KM)                                                               \
  do {                                                                            \
    if (act_dtype == MOE_BF16 && y_bf16) {                                        \
      auto kern = finalize_kernel<__nv_bfloat16, KM, __nv_bfloat16>;              \
      MOE_LAUNCH(kern, blocks, threads, 0, s, yb, dest, w, srb,                   \
                 static_cast<__nv_bfloat16*>(out), T, k, D, R, m, err);           \
    } else if (act_dtype == MOE_BF16) {                                           \
      auto kern = finalize_kernel<__nv_bfloat16, KM, float>;                      \
      MOE_LAUNCH(kern, blocks, threads, 0, s, y, dest, w, sr,                     \
                 static_cast<__nv_bfloat16*>(out), T, k, D, R, m, err);           \
    } else {                                                                      \
      auto kern = finalize_kernel<float, KM, float>;                              \
      MOE_LAUNCH(kern, blocks, threads, 0, s, y, dest, w, sr,                     \
                 static_cast<float*>(out), T, k, D, R, m, err);                   \
    }                                                                             \
  } while (0)
  if (k <= 2) MOE_FIN(2);
  else if (k <= 4) MOE_FIN(4);
  else if (k <= 8) MOE_FIN(8);
  else if (k <= 10) MOE_FIN(10);
  else MOE_FIN(16);
#undef MOE_FIN
  return cudaGetLastError();
}

}  // namespace moe
