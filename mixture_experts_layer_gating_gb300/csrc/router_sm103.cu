// Router projection fused with gating top-k softmax, for batches of more than
// 64 tokens ("CANN/cann-recipes-infer：Qwen3-MoE优化", section "GMM使能和Routing
// 优化": the gate projection and gating_top_k_softmax in one fused operator;
// the gate kept in fp32 as on the "千问 3.5 MoE 在 TPU 上的系统优化实战" page).
//
//   logits[t, e] = sum_d x[t, d] W_g[d, e] (+ bias[e])      (fp32 accumulation)
//   ids[t, :], w[t, :] = top-k of logits[t, :] and its softmax
//
// One thread-block cluster per tile of 128 tokens.  Its C = ck x nh CTAs split
// the reduction over D into ck consecutive slices (ck = 1, 2, 4) and, when
// E > 256, the experts into nh = 2 halves of 256.  Each CTA:
//   warp 0      : TMA producer (one lane) -- x tile 128 tokens x 64 d (K-major)
//                 and the W_g boxes of its experts, 64 d x 64 experts each
//                 (N-major), per stage of a ring in shared memory;
//   warp 1      : TMEM allocator + single-lane tcgen05.mma issuer, M = 128,
//                 N = its experts (64, 128 or 256), K = 16 per instruction,
//                 one fp32 accumulator in TMEM;
//   warps 2..5  : after the last product, read the accumulator (one token row
//                 per thread) and send each row to the CTA of the cluster that
//                 finishes it, into that CTA's shared memory (the stage ring,
//                 no longer needed);
//   warps 6..15 : wait at the cluster barrier;
// then all 16 warps of the CTA finish its 128 / C tokens: the ck partial rows
// added in slice order, the bias added last, the final logits written, and the
// top-k and softmax taken by one warp per token with the same routine as the
// stand-alone top-k kernel; on request (chunk_hist) each CTA also writes the
// expert histogram of its tokens' ids, from which init_routing sorts the rows
// without counting them again.  Two cluster barriers order the hand-over: one
// after every CTA's products (its ring may be overwritten), one after every
// partial row has arrived.  Every mbarrier wait is bounded; a CTA that gives
// up flags MOE_DEV_WAIT_TIMEOUT and still takes part in both barriers.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "moe_internal.h"
#include "sm103_ptx.cuh"
#include "topk_warp.cuh"

namespace moe {
namespace {

constexpr int RT_BM = 128;                       // tokens per tile (TMEM lanes)
constexpr int RT_BK = 64;                        // d per stage (128 bytes of bf16)
constexpr int RT_A_BYTES = RT_BM * RT_BK * 2;    // 16 KB x tile
constexpr int RT_BOX_BYTES = 64 * RT_BK * 2;     // 64 experts x 64 d of W_g, 8 KB
constexpr int RT_RING_BYTES = 192 * 1024;        // stage ring (later: partial rows)
constexpr int RT_MAX_STAGES = 8;
constexpr int RT_THREADS = 512;  // 16 warps: all of them take tokens in the top-k phase
constexpr int RT_WARPS = RT_THREADS / 32;
// Clusters of 8 such CTAs (197 KB of shared memory each) measured slower than
// 4 (Gemma-4-style prefill router, 16 token tiles: 24.4 us with 8 slices);
// at most 4 CTAs per cluster.
constexpr int RT_MAX_CLUSTER = 4;

template <int NB>
struct RtCfg {
  static constexpr int kStageBytes = RT_A_BYTES + NB * 128;  // x tile + NB / 64 W_g boxes
  static constexpr int kStages =
      RT_RING_BYTES / kStageBytes > RT_MAX_STAGES ? RT_MAX_STAGES : RT_RING_BYTES / kStageBytes;
  // partial rows of the cluster's tile at their finishing CTA: 128 / nh rows
  // of nh * NB + 4 floats (the padding spreads a warp's 16-byte row stores
  // over all banks); nh = 2 only with NB = 256
  static_assert(RT_BM * (NB + 4) * 4 <= RT_RING_BYTES, "partial rows fit the ring");
  static_assert((RT_BM / 2) * (2 * 256 + 4) * 4 <= RT_RING_BYTES, "partial rows fit the ring");
};

struct RtCtrl {
  uint64_t full[RT_MAX_STAGES];
  uint64_t empty[RT_MAX_STAGES];
  uint64_t tfull;
  uint32_t tmem_slot;
  int abort;
};

// after the ctrl block: the CTA's expert histogram of its tokens' ids (E <= 512)
constexpr size_t rt_smem_bytes() { return 1024 + RT_RING_BYTES + sizeof(RtCtrl) + 512 * sizeof(int32_t); }
static_assert(rt_smem_bytes() <= 227 * 1024, "shared memory budget");

struct RtParams {
  int T, D, E, k, renorm;
  int ck;  // slices of the reduction over D (CTAs per expert half)
  int nh;  // expert halves: 1, or 2 when E > 256 (then NB = 256)
  const float* bias;
  float* logits;
  int32_t* ids;
  float* w;
  int32_t* err;
  // optional [gridDim.x][E]: row b = expert counts of the ids of CTA b's
  // tokens (the tokens [b * 128 / C, (b + 1) * 128 / C), C CTAs per cluster)
  int32_t* chunk_hist;
};

// NB: experts per CTA (the MMA N); EPL: logits per lane in the top-k warp.
template <int NB, int EPL>
__global__ void __launch_bounds__(RT_THREADS, 1)
    router_topk_kernel(const __grid_constant__ CUtensorMap tmap_x,
                       const __grid_constant__ CUtensorMap tmap_wg, const RtParams p) {
  pdl_wait();
  pdl_launch_dependents();
  constexpr int STAGES = RtCfg<NB>::kStages;
  constexpr int STAGE_BYTES = RtCfg<NB>::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned start, formed as smem_raw + offset (not through an
  // integer round trip) so that the compiler keeps it a shared-memory pointer:
  // the partial rows' loads and the histogram's atomics are then shared-space
  // accesses, not generic ones ordered behind the tokens' global stores
  const uint32_t s_raw = smem_u32(smem_raw);
  uint8_t* base = smem_raw + (((s_raw + 1023u) & ~1023u) - s_raw);
  RtCtrl* ctrl = reinterpret_cast<RtCtrl*>(base + RT_RING_BYTES);
  int32_t* hist = reinterpret_cast<int32_t*>(base + RT_RING_BYTES + sizeof(RtCtrl));
  float* red = reinterpret_cast<float*>(base);  // partial rows, after the products
  volatile int* abort_flag = &ctrl->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int C = p.ck * p.nh;
  const int q = static_cast<int>(cluster_ctarank());
  const int hx = q % p.nh;   // expert half of this CTA
  const int sl = q / p.nh;   // slice of D of this CTA
  const int m0 = static_cast<int>(cluster_id_x()) * RT_BM;  // first token of the tile
  const int KB = (p.D + RT_BK - 1) / RT_BK;
  // balanced slices: every slice has at least one k-block while ck <= KB
  const int kb0 = sl * KB / p.ck, kb1 = (sl + 1) * KB / p.ck;
  const int rpo = RT_BM / C;         // tokens each CTA of the cluster finishes
  const int ld = p.nh * NB + 4;      // floats per partial row
  const int e0 = hx * NB;            // first expert of this CTA

  for (int e = threadIdx.x; e < p.E; e += RT_THREADS) hist[e] = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctrl->full[s], 1);
      mbar_init(&ctrl->empty[s], 1);
    }
    mbar_init(&ctrl->tfull, 1);
    ctrl->abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_wg);
  }
  if (warp == 1) {
    tmem_alloc(&ctrl->tmem_slot, NB);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = ctrl->tmem_slot;

  // W_g boxes of this CTA that hold experts below E (boxes wholly past E are
  // not loaded; their accumulator columns are never read)
  const int nbox = min(NB / 64, (p.E - e0 + 63) / 64);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_normal();
      const uint32_t tx = static_cast<uint32_t>(RT_A_BYTES + nbox * RT_BOX_BYTES);
      uint32_t stage = 0, phase = 0, fill_mask = 0, fill_par = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&ctrl->empty[stage], phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&ctrl->full[stage], tx);
        uint8_t* st = base + stage * STAGE_BYTES;
        tma_load_2d(st, &tmap_x, &ctrl->full[stage], kb * RT_BK, m0, pol);
        for (int j = 0; j < nbox; ++j)
          tma_load_2d(st + RT_A_BYTES + j * RT_BOX_BYTES, &tmap_wg, &ctrl->full[stage],
                      e0 + 64 * j, kb * RT_BK, pol);
        fill_mask |= 1u << stage;
        fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok || *abort_flag) {
        ctrl->abort = 1;
        if (!ok) atomicOr(p.err, MOE_DEV_WAIT_TIMEOUT);
        // let the copies in flight land before the ring is reused or the CTA leaves
        for (int st = 0; st < STAGES; ++st)
          if ((fill_mask >> st) & 1u) mbar_wait_drain(&ctrl->full[st], (fill_par >> st) & 1u);
        drain_grace();
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc_bf16_f32(RT_BM, NB, 0, 1);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&ctrl->full[stage], phase, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint8_t* st = base + stage * STAGE_BYTES;
        // x: K-major, 128-byte rows (a K step of 16 is 32 bytes); W_g: N-major
        // 64-expert boxes 8 KB apart (a K step of 16 rows is 2 KB)
        const uint64_t adesc0 = make_smem_desc_sw128(smem_u32(st), 16, 1024);
        const uint64_t bdesc0 = make_smem_desc_sw128(smem_u32(st + RT_A_BYTES), RT_BOX_BYTES, 1024);
#pragma unroll
        for (int kk = 0; kk < RT_BK / 16; ++kk)
          tc_mma_f16(tmem_base, smem_desc_advance(adesc0, kk * 32), smem_desc_advance(bdesc0, kk * 2048),
                     idesc, ((kb - kb0) | kk) != 0);
        tc_commit(&ctrl->empty[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        tc_commit(&ctrl->tfull);  // arrives once every product above is done
      } else {
        ctrl->abort = 1;
        atomicOr(p.err, MOE_DEV_WAIT_TIMEOUT);
      }
    }
    __syncwarp();
  }

  // ---------------------------------------------------------- accumulator
  bool have_acc = false;
  if (warp >= 2 && warp < 6) {
    have_acc = mbar_wait(&ctrl->tfull, 0, abort_flag);
    if (!have_acc && lane == 0) {
      ctrl->abort = 1;
      atomicOr(p.err, MOE_DEV_WAIT_TIMEOUT);
    }
    __syncwarp();
    tc_fence_after_sync();
  }
  // every CTA of the cluster has finished its products: the rings may be overwritten
  tc_fence_before_sync();
  cluster_sync();
  tc_fence_after_sync();
  if (warp >= 2 && warp < 6) {
    const int quarter = warp & 3;  // TMEM lanes [32 quarter, 32 quarter + 32)
    const int r = quarter * 32 + lane;
    const int owner = r / rpo, local = r - owner * rpo;
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    float* row = red + static_cast<size_t>(sl * rpo + local) * ld + e0;
    const uint32_t dst = mapa_shared(row, static_cast<uint32_t>(owner));
    for (int c = 0; c < nbox * 64; c += 32) {
      uint32_t v[32];
      tmem_ld_32x32b_x32(taddr + c, v);
      tc_wait_ld();
      if (!have_acc) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0u;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        st_cluster_v4(dst + static_cast<uint32_t>((c + 4 * j) * 4), v[4 * j], v[4 * j + 1],
                      v[4 * j + 2], v[4 * j + 3]);
    }
  }
  // every partial row has arrived at its finishing CTA
  tc_fence_before_sync();
  cluster_sync();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, NB);

  // ---------------------------------------------------------- top-k softmax
  for (int i = warp; i < rpo; i += RT_WARPS) {
    const int t = m0 + q * rpo + i;
    if (t >= p.T) break;  // tokens grow with i
    float v[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = lane + 32 * j;
      float s = 0.0f;
      if (e < p.E) {
        s = red[static_cast<size_t>(i) * ld + e];
        for (int z = 1; z < p.ck; ++z) s += red[static_cast<size_t>(z * rpo + i) * ld + e];
      }
      v[j] = s;
    }
    const int id = warp_topk_softmax<EPL>(v, lane, p.E, p.k, p.renorm, p.bias,
                                          p.logits + static_cast<size_t>(t) * p.E,
                                          p.ids + static_cast<size_t>(t) * p.k,
                                          p.w + static_cast<size_t>(t) * p.k, p.err);
    if (id >= 0) atomicAdd(&hist[id], 1);
  }
  if (p.chunk_hist) {
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += RT_THREADS)
      p.chunk_hist[static_cast<size_t>(blockIdx.x) * p.E + e] = hist[e];
  }
}

template <int NB, int EPL>
cudaError_t launch_rt(const CUtensorMap& tx, const CUtensorMap& tw, const RtParams& p, int tiles,
                      cudaStream_t s) {
  auto kern = router_topk_kernel<NB, EPL>;
  constexpr size_t smem = rt_smem_bytes();
  static bool done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) done[dev] = true;
  }
  const int C = p.ck * p.nh;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = g_pdl ? 1 : 0;
  cfg.gridDim = dim3(tiles * C, 1, 1);
  cfg.blockDim = dim3(RT_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tx, tw, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

void router_topk_split(int T, int E, int D, int& ck, int& nh) {
  const int tiles = (T + RT_BM - 1) / RT_BM;
  nh = E > 256 ? 2 : 1;
  const int KB = (D + RT_BK - 1) / RT_BK;
  // about one wave of CTAs on a 152-SM GB300 (a constant, so that the choice
  // depends on the shape alone), slices of at least 4 k-blocks, clusters of
  // at most RT_MAX_CLUSTER CTAs
  const int want = std::max(1, std::min({RT_MAX_CLUSTER / nh, 148 / std::max(1, tiles * nh), KB / 4}));
  ck = 1;
  while (2 * ck <= want) ck *= 2;
}

bool router_topk_ok(int T, int E, int D, int k) {
  // at least one full 64-expert box (W_g rows of 128 bytes or more)
  return T > 0 && E >= 64 && E <= 512 && (E % 8) == 0 && k >= 1 && k <= E && k <= 32 && D >= 1 &&
         (D % 8) == 0;
}

bool router_topk_preferred(int T, int E, int D) {
  // at least 64 CTAs: with fewer token tiles (decode batches up to 512
  // tokens: 4-16 CTAs) the split-K projection over ~64-148 CTAs plus the
  // top-k kernel is faster (Qwen3.5-style decode, 512 tokens: 60 us fused)
  int ck, nh;
  router_topk_split(T, E, D, ck, nh);
  return static_cast<long long>((T + RT_BM - 1) / RT_BM) * ck * nh >= 64;
}

void router_topk_chunks(int T, int E, int D, int k, int& nchunks, int& chunk_rows) {
  int ck, nh;
  router_topk_split(T, E, D, ck, nh);
  nchunks = (T + RT_BM - 1) / RT_BM * ck * nh;
  chunk_rows = RT_BM / (ck * nh) * k;
}

cudaError_t launch_router_topk(const void* x, const void* Wg, const float* bias, int T, int D,
                               int E, int k, int renorm, float* logits, int32_t* ids, float* w,
                               int32_t* err, cudaStream_t s, int32_t* chunk_hist) {
  if (!router_topk_ok(T, E, D, k) || !x || !Wg || !logits || !ids || !w ||
      (reinterpret_cast<uintptr_t>(chunk_hist) & 15))
    return cudaErrorInvalidValue;
  RtParams p;
  p.T = T;
  p.D = D;
  p.E = E;
  p.k = k;
  p.renorm = renorm;
  router_topk_split(T, E, D, p.ck, p.nh);
  p.bias = bias;
  p.logits = logits;
  p.ids = ids;
  p.w = w;
  p.err = err;
  p.chunk_hist = chunk_hist;
  CUtensorMap tx, tw;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(D), static_cast<uint64_t>(T)};
    const uint64_t strides[1] = {static_cast<uint64_t>(D) * 2};
    const uint32_t box[2] = {RT_BK, RT_BM};
    if (!encode_tmap(&tx, x, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(E), static_cast<uint64_t>(D)};
    const uint64_t strides[1] = {static_cast<uint64_t>(E) * 2};
    const uint32_t box[2] = {64, RT_BK};
    if (!encode_tmap(&tw, Wg, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  const int tiles = (T + RT_BM - 1) / RT_BM;
  const int per_cta = E / p.nh;  // experts of one CTA
  if (p.nh == 2) return launch_rt<256, 16>(tx, tw, p, tiles, s);
  if (per_cta <= 64) return launch_rt<64, 2>(tx, tw, p, tiles, s);
  if (per_cta <= 128) return launch_rt<128, 4>(tx, tw, p, tiles, s);
  return launch_rt<256, 8>(tx, tw, p, tiles, s);
}

}  // namespace moe
