// Grouped GEMM over variable-length expert segments on the sm_103a tensor
// core (tcgen05 + TMEM), fed by TMA.
//
// What it computes (per group g with rows [start_g, start_g + cnt_g) of A):
//   gate/up pass : acc = A_g [gate | up]; h = act(gate * s) * (up * s), stored
//                  as a bf16 pair h_hi = bf16(h), h_lo = bf16(h - h_hi)
//   down pass    : out = ((A_hi + A_lo)_g B_g) * s   (fp32 out; two MMAs per
//                  K step so h keeps ~16 significant bits through the GEMM)
//   router pass  : out = A B + bias                 (fp32 out, one group)
// This is the grouped matmul of "CANN/cann-recipes-infer：Qwen3-MoE优化"
// (section "GMM使能和Routing优化": one op computes every expert instead of a
// per-expert loop), with the swiglu of section "MoE TP优化 / 计算分解" fused
// into the epilogue of the gate/up pass (the "千问 3.5 MoE 在 TPU 上的系统优化
// 实战" page fuses SwiGLU into the GMM main loop the same way) and the
// per-output-channel fp8 scale of "用SGLang-JAX在TPU上优化Ling-2.6-1T" §5
// applied after the full K reduction.  Segments are unpadded: a tile that runs
// past its segment computes rows of the next segment and masks their stores
// (the Qwen3.5 page's dynamic bounded slices with minimal padding).
//
// Kernel structure (one persistent CTA per SM, 192 threads; or, in PAIR mode,
// one persistent 2-CTA cluster per SM pair that computes M=256 row tiles with
// tcgen05.mma.cta_group::2 -- each CTA loads its own 128 A rows and half of the
// B columns, so per-SM operand traffic for a 256x256 tile drops by a third):
//   warp 0      : TMA producer (one lane) -- A tile 128 x 64 (K-major; two
//                 of them, hi and lo, in the bf16 down pass) and B tile 64 x 256
//                 (N-major) per stage, 4-stage (3 in the split / fp8 passes) ring.
//   warp 1      : TMEM allocator + single-lane tcgen05.mma issuer,
//                 M=128 N=256 K=16 per instruction, fp32 accumulators in TMEM,
//                 two accumulator buffers (2 x 256 columns).
//   warps 2..5  : epilogue -- tcgen05.ld 32 lanes x 32 columns, activation /
//                 scale, masked stores; one row per thread.
//   warps 6..13 : (fp8 weights only) converters -- TMA brings the raw e4m3
//                 weight boxes; these warps expand them exactly to 16-bit
//                 floats in the swizzled N-major layout the MMA reads, then
//                 arrive on the stage's full barrier (W8A16).  Both passes run
//                 on the fp16 kind: e4m3 -> fp16 is one hardware convert per
//                 pair, and the A rows (x, or h) arrive as fp16 rows carrying
//                 an exact power-of-two row scale that the epilogue removes.
// 2-CTA mode runs a group's last tile "swapped" when it has few rows (at most
// 64 in the gate/up pass, 128 in the down pass): the weights become the
// M = 256 operand (128 features per CTA: gate and matching up features in the
// gate/up pass) and the rows the N operand (N = rows rounded up to 16; the
// down pass stacks h_hi and h_lo rows, N = 2 x that), so a short tail costs a
// short MMA instead of a full 256-row tile.
// Tiles are ordered (group, column tile, row tile) so that the row tiles that
// share a weight slice run at the same time and reuse it from L2.  The tile
// schedule is built on the device from the group offsets, so no host
// synchronisation is needed between routing and the GEMM.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "moe_internal.h"
#include "sm103_ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BN_MAX = 256;
constexpr int A_TILE_BYTES = BM * BK * 2;    // 16 KB
constexpr int B_BOX_BYTES = 64 * BK * 2;     // one 64-column x 64-row bf16 box, 8 KB
constexpr int B_TILE_BYTES = BN_MAX * BK * 2; // 32 KB
constexpr int MAX_STAGES = 8;
constexpr int STAGE_BUDGET = 192 * 1024;
// epilogue staging of the fp32 store pass: one padded 32 x 36 fp32 tile per
// epilogue warp turns a row per thread into 128-byte row segments per store
constexpr int EPI_STAGE_LD = 36;  // padded row (144 bytes: 16-byte aligned rows)
constexpr int EPI_STAGE_FLOATS = 32 * EPI_STAGE_LD;
constexpr int EPI_STAGE_BYTES = 4 * EPI_STAGE_FLOATS * 4;
// groups of one launch: 512 experts, plus the shared expert as one more
// group when it runs inside the routed GEMMs
constexpr int MAX_G = 513;
constexpr uint32_t TMEM_COLS = 512;
constexpr int TQ_DEPTH = 4;  // tile indices in flight between the producer and the other roles
constexpr uint32_t ACC_STRIDE = 256;  // TMEM columns per accumulator buffer

constexpr int RAW_BOX_BYTES = 128 * BK;        // one 128-column x 64-row e4m3 box, 8 KB
constexpr int RAW_TILE_BYTES = 2 * RAW_BOX_BYTES;

template <bool SPLIT, bool FP8, bool PAIR>
struct StageCfg {
  static_assert(!(SPLIT && FP8), "fp8 layers use an unsplit h");
  // Weights expanded from e4m3 on chip run on one-CTA tiles only: 2-CTA tiles
  // measured 40 % slower there, and the one run of an instrumented 2-CTA copy
  // at full Ling size ended in a GPU fault whose cause was not established, so
  // that combination is not compiled.
  static_assert(!(FP8 && PAIR), "no 2-CTA tiles for weights expanded on chip");
  static constexpr int kABytes = (SPLIT ? 2 : 1) * A_TILE_BYTES;  // hi (+ lo) A tiles
  // this CTA's share of the bf16 B tile (all 256 columns, or 128 in a pair)
  static constexpr int kBBytes = PAIR ? B_TILE_BYTES / 2 : B_TILE_BYTES;
  static constexpr int kRawBytes = FP8 ? (PAIR ? RAW_BOX_BYTES : RAW_TILE_BYTES) : 0;
  // stage layout: [A (+ A lo) | B (bf16, MMA operand) | raw e4m3 B]
  static constexpr int kStageBytes = kABytes + kBBytes + kRawBytes;
  static constexpr int kStages =
      STAGE_BUDGET / kStageBytes > MAX_STAGES ? MAX_STAGES : STAGE_BUDGET / kStageBytes;
  // fp8: e4m3 -> fp16 converter warps (6 ..): the expansion limits the fp8
  // passes; 8 warps measured 11 % faster than 4 on the Ling prefill layer, 10
  // no better
  static constexpr int kConvWarps = 8;
  static constexpr int kThreads = FP8 ? (6 + kConvWarps) * 32 : 192;
  static constexpr int kTileM = PAIR ? 2 * BM : BM;  // rows per scheduled tile
};

struct Ctrl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t raw_full[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t xch_full, xch_empty;  // decode gate/up epilogue: up values staged / consumed
  // dynamic tile order: the tile indices handed to every role of the CTA (pair)
  uint64_t tq_full[TQ_DEPTH];
  uint64_t tq_empty[TQ_DEPTH];
  int tq[TQ_DEPTH];
  uint32_t tmem_slot;
  int abort;
  // the schedule's groups in the order their tiles run: position i holds
  // group grp_id[i] (i itself in expert order; heaviest first under LPT)
  int grp_id[MAX_G];
  int grp_start[MAX_G];
  int grp_cnt[MAX_G];
  int tile_start[MAX_G + 1];
};

template <bool SPLIT, bool FP8, bool PAIR>
constexpr size_t smem_bytes() {
  return 1024 + StageCfg<SPLIT, FP8, PAIR>::kStages * StageCfg<SPLIT, FP8, PAIR>::kStageBytes +
         sizeof(Ctrl) + EPI_STAGE_BYTES;
}
static_assert(EPI_STAGE_BYTES >= 4 * 4096 + 1023, "TMA store staging fits the epilogue staging area");
static_assert(smem_bytes<false, false, false>() <= 227 * 1024, "shared memory budget");
static_assert(smem_bytes<true, false, false>() <= 227 * 1024, "shared memory budget");
static_assert(smem_bytes<false, true, false>() <= 227 * 1024, "shared memory budget");
static_assert(smem_bytes<false, false, true>() <= 227 * 1024, "shared memory budget");
static_assert(smem_bytes<true, false, true>() <= 227 * 1024, "shared memory budget");

struct KParams {
  const int32_t* group_offsets;
  int G;
  int M;
  int K;
  int N;              // output columns
  int n_tiles;        // column tiles
  int bn;             // MMA N (accumulator columns per tile)
  int cols_per_tile;  // output columns per tile
  void* out;
  void* out_lo;  // gate/up pass: h_lo
  const float* b_scale;
  const float* bias;
  const float* a_row_scale;  // per-row factor on the accumulator (fp16 A rows), or nullptr
  const int32_t* a_gather;   // gather mode: A row of output row r is a_gather[r] / gather_k
  const void* a_src;         // cp.async gather mode: the [a_rows, K] bf16 A rows
  int gather_k;
  int a_rows;                // rows of the A tensor (gather mode)
  int h_fp32;                // gate/up pass: store h as fp32
  int act;
  int ksplit;  // K split into ksplit parts, each writing its own fp32 output plane
  int kbs;     // k-blocks per split
  int b_wide;  // bf16 B map viewed as [64-column blocks][K][64]: one load per stage
  // 2-CTA tiles: a group's last tile with at most swap_tail rows runs "swapped":
  // weights as the M = 256 operand (128 features per CTA), its rows as N
  int swap_tail;
  int32_t* err;
  // kEpiCombineF32 (fused combine): expanded row of each output row, routing
  // weights, k; out is the [T, N] fp32 accumulator
  const int32_t* comb_rows;
  const float* comb_w;
  int comb_k;
  int lpt;  // 1: groups scheduled heaviest first (most rows; lower index on ties)
  // > 0: the producer also prefetches this CTA's weight box b_prefetch
  // k-blocks ahead into L2 (into the next tile of this CTA near a tile's end)
  int b_prefetch;
  // > 0: the last group (G - 1) is the shared expert: its rows are the last
  // sh_rows rows of A [M - sh_rows, M) and its weights the second weight map
  // (tmap_b2) with per-column scales sh_b_scale
  int sh_rows;
  const float* sh_b_scale;
  // store pass (one plane, no bias): full 32-row warp chunks leave through
  // TMA bulk-tensor stores (tmap_out: the [M, N] output, 128-byte rows per box)
  int tma_out;
  // dynamic tile order: a global counter, zero before the launch, from which
  // the producer of each CTA (the leader of each pair) takes its next tile;
  // nullptr = static round-robin (tile t to CTA / pair t mod grid)
  int32_t* tile_counter;
};

// Fused combine: the token and routing weight of permuted output row `row`.
__device__ __forceinline__ void comb_token(const KParams& p, size_t row, int& t, float& w) {
  if (p.sh_rows > 0 && row >= static_cast<size_t>(p.M - p.sh_rows)) {  // shared expert: weight 1
    t = static_cast<int>(row - static_cast<size_t>(p.M - p.sh_rows));
    w = 1.0f;
    return;
  }
  const int q = p.comb_rows[row];
  t = q / p.comb_k;
  w = p.comb_w[q];
}

// Element type of the store pass's output rows: bf16 for fp8-weight layers
// (expanded on chip or read as e4m3), fp32 otherwise.
template <bool FP8W>
using StoreT = typename std::conditional<FP8W, __nv_bfloat16, float>::type;
__device__ __forceinline__ void store_elem(float* out, size_t i, float v) { out[i] = v; }
__device__ __forceinline__ void store_elem(__nv_bfloat16* out, size_t i, float v) {
  out[i] = __float2bfloat16_rn(v);
}

struct TileInfo {
  int g, row0, rows, n0;
};

template <int TILE_M>
__device__ __forceinline__ TileInfo decode_tile(const Ctrl* c, int G, int t, int n_tiles,
                                                int cols_per_tile) {
  const int q = t / n_tiles;
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (c->tile_start[mid] <= q) lo = mid; else hi = mid - 1;
  }
  TileInfo ti;
  ti.g = c->grp_id[lo];
  const int mt_g = c->tile_start[lo + 1] - c->tile_start[lo];
  const int local = t - c->tile_start[lo] * n_tiles;
  const int nt = local / mt_g;
  const int mt = local - nt * mt_g;
  ti.row0 = c->grp_start[lo] + mt * TILE_M;
  ti.rows = min(TILE_M, c->grp_cnt[lo] - mt * TILE_M);
  ti.n0 = nt * cols_per_tile;
  return ti;
}

// Rows [a, b) of group g, validated (a bad group gets none and sets `bad`);
// with sh_rows > 0 the last group g = G - 1 is the shared expert's rows
// [M - sh_rows, M).
__device__ __forceinline__ void group_rows(const int32_t* offsets, int g, int M, int& a, int& b,
                                           bool& bad, int G = 0, int sh_rows = 0) {
  if (sh_rows > 0 && g == G - 1) {
    a = M - sh_rows;
    b = M;
    return;
  }
  a = 0;
  b = M;
  if (offsets) {
    a = offsets[g];
    b = offsets[g + 1];
  }
  if (a < 0 || b < a || b > M) {
    bad = true;
    a = 0;
    b = 0;
  }
}

// Heaviest-first (LPT) schedule: the groups sorted by row count, descending,
// the lower index first among equal counts, by a bitonic sort of 512 32-bit
// keys (min(count, 2^23 - 1) << 9 | 511 - g; counts beyond 2^23 rows keep
// index order among themselves) held 16 per lane in one warp: position
// i = lane * 16 + r.  Then grp_id / grp_start / grp_cnt / tile_start by
// position.  G <= 512 (a key of 0 is padding: real keys are >= 512 - G).
template <int J>  // one bitonic stage whose partner is r ^ J in this lane
__device__ __forceinline__ void lpt_stage_in_lane(uint32_t (&key)[16], int lane, int k) {
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    if ((r ^ J) > r) {
      const int i = lane * 16 + r;
      const uint32_t a = key[r], b = key[r ^ J];
      const bool swap = ((i & k) == 0) ? (a < b) : (a > b);  // descending blocks first
      key[r] = swap ? b : a;
      key[r ^ J] = swap ? a : b;
    }
  }
}

__device__ __noinline__ void build_schedule_lpt(Ctrl* ctrl, const int32_t* offsets, int G, int M,
                                                int tile_h, int32_t* err, int lane, int sh_rows) {
  uint32_t key[16];
  bool bad = false;
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int g = lane * 16 + r;
    key[r] = 0;  // padding sorts last
    if (g < G) {
      int a, b;
      group_rows(offsets, g, M, a, b, bad, G, sh_rows);
      key[r] = (static_cast<uint32_t>(min(b - a, (1 << 23) - 1)) << 9) | static_cast<uint32_t>(511 - g);
    }
  }
#pragma unroll 1
  for (int k = 2; k <= 512; k <<= 1) {
#pragma unroll 1
    for (int j = k >> 1; j >= 16; j >>= 1) {  // partner in lane ^ (j / 16), same register
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const uint32_t other = __shfl_xor_sync(0xffffffffu, key[r], j >> 4);
        const int i = lane * 16 + r;
        const bool keep_max = (((i & j) == 0) == ((i & k) == 0));
        key[r] = keep_max ? max(key[r], other) : min(key[r], other);
      }
    }
    if (k >= 16) lpt_stage_in_lane<8>(key, lane, k);
    if (k >= 8) lpt_stage_in_lane<4>(key, lane, k);
    if (k >= 4) lpt_stage_in_lane<2>(key, lane, k);
    lpt_stage_in_lane<1>(key, lane, k);
  }
  int local = 0;
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int i = lane * 16 + r;
    if (i < G) {
      const int g = 511 - static_cast<int>(key[r] & 511u);
      int a, b;
      bool bad2 = false;
      group_rows(offsets, g, M, a, b, bad2, G, sh_rows);
      ctrl->grp_id[i] = g;
      ctrl->grp_start[i] = a;
      ctrl->grp_cnt[i] = b - a;
      local += (b - a + tile_h - 1) / tile_h;
    }
  }
  int incl = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  int run = incl - local;
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int i = lane * 16 + r;
    if (i < G) {
      ctrl->tile_start[i] = run;
      run += (ctrl->grp_cnt[i] + tile_h - 1) / tile_h;
    }
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  if (lane == 0) ctrl->tile_start[G] = total;
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(err, MOE_DEV_BAD_OFFSETS);
}

// One warp builds the row-tile schedule of the groups in shared memory:
// grp_start / grp_cnt per group (offsets validated: a bad group gets no rows and
// MOE_DEV_BAD_OFFSETS is flagged) and tile_start[g] = sum_{g' < g} ceil(cnt_g' / tile_h),
// in expert order (grp_id[g] = g), or heaviest first when lpt is set.
// offsets == nullptr: one group of M rows.
__device__ void build_schedule(Ctrl* ctrl, const int32_t* offsets, int G, int M, int tile_h,
                               int32_t* err, int lane, int lpt = 0, int sh_rows = 0) {
  if (lpt && G > 1 && G <= 512) {
    build_schedule_lpt(ctrl, offsets, G, M, tile_h, err, lane, sh_rows);
    return;
  }
  const int per = (G + 31) / 32;  // <= 17 groups per lane (G <= MAX_G)
  const int g0 = min(G, lane * per), g1 = min(G, g0 + per);
  // this lane's offsets[g0 .. g1] first, every load in flight at once (one
  // memory round trip instead of one per group); offsets holds G + 1 entries,
  // or G when the last group is the shared expert's rows
  constexpr int kPer = (MAX_G + 31) / 32;
  static_assert(kPer <= 17, "groups per lane");
  const int n_ofs = (sh_rows > 0) ? G : G + 1;
  int ofs[kPer + 1];
#pragma unroll
  for (int i = 0; i <= kPer; ++i)
    ofs[i] = (offsets && i <= g1 - g0 && g0 + i < n_ofs) ? offsets[g0 + i] : 0;
  int local = 0;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int g = g0 + i;
    if (g < g1) {
      int a = 0, b = M;
      if (sh_rows > 0 && g == G - 1) {
        a = M - sh_rows;
      } else if (offsets) {
        a = ofs[i];
        b = ofs[i + 1];
      }
      if (a < 0 || b < a || b > M) {
        bad = true;
        a = 0;
        b = 0;
      }
      ctrl->grp_id[g] = g;
      ctrl->grp_start[g] = a;
      ctrl->grp_cnt[g] = b - a;
      local += (b - a + tile_h - 1) / tile_h;
    }
  }
  int incl = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  int run = incl - local;
  for (int g = g0; g < g1; ++g) {
    ctrl->tile_start[g] = run;
    run += (ctrl->grp_cnt[g] + tile_h - 1) / tile_h;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  if (lane == 0) ctrl->tile_start[G] = total;
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(err, MOE_DEV_BAD_OFFSETS);
}

// Tile t of a schedule with row tiles of height tile_h, ordered
// (group, column tile, row tile) with the row tile fastest.
__device__ __forceinline__ TileInfo decode_tile_h(const Ctrl* c, int G, int t, int n_tiles,
                                                  int cols_per_tile, int tile_h) {
  const int q = t / n_tiles;
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (c->tile_start[mid] <= q) lo = mid; else hi = mid - 1;
  }
  TileInfo ti;
  ti.g = c->grp_id[lo];
  const int mt_g = c->tile_start[lo + 1] - c->tile_start[lo];
  const int local = t - c->tile_start[lo] * n_tiles;
  const int nt = local / mt_g;
  const int mt = local - nt * mt_g;
  ti.row0 = c->grp_start[lo] + mt * tile_h;
  ti.rows = min(tile_h, c->grp_cnt[lo] - mt * tile_h);
  ti.n0 = nt * cols_per_tile;
  return ti;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }
__device__ __forceinline__ float gelu_tanh_f(float g) {
  const float c = 0.7978845608028654f;  // sqrt(2/pi)
  return 0.5f * g * (1.0f + tanhf(c * (g + 0.044715f * g * g * g)));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Four e4m3 values (bytes of w, low byte first) to four fp16, exactly (every
// e4m3 value is an fp16 value): one hardware conversion per pair, element
// order kept.
__device__ __forceinline__ uint2 e4m3x4_to_f16x4(uint32_t w) {
  uint2 r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
      : "=r"(r.x), "=r"(r.y)
      : "r"(w));
  return r;
}

// Q8: B is e4m3 stored K-contiguous ([G, N, K]): the 8-bit kind::f8f6f4 with
// 128 K elements (128 bytes) per stage and no weight expansion; the A rows are
// two-term e4m3 (hi and lo tiles of the stage, as in SPLIT: W8A16) or, with
// SPLIT off, one e4m3 term with a per-row scale (W8A8).
// CPG: the A rows are gathered by four extra warps (6..9) with 16-byte
// cp.async copies from the unpermuted rows (bf16, one-CTA tiles, gate/up pass).
template <int EPI, bool SPLIT, bool FP8, bool PAIR, bool Q8, bool CPG = false>
__global__ void __launch_bounds__(CPG ? 320 : StageCfg<SPLIT, FP8, PAIR>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_a_lo,
                        const __grid_constant__ CUtensorMap tmap_b,
                        const __grid_constant__ CUtensorMap tmap_b_tail,
                        const __grid_constant__ CUtensorMap tmap_a_tail,
                        const __grid_constant__ CUtensorMap tmap_a_lo_tail,
                        const __grid_constant__ CUtensorMap tmap_b2,
                        const __grid_constant__ CUtensorMap tmap_b2_tail,
                        const __grid_constant__ CUtensorMap tmap_out, const KParams p) {
  pdl_wait();
  static_assert(!Q8 || !FP8, "e4m3 rows meet K-contiguous e4m3 weights, not expanded ones");
  static_assert(!CPG || (!SPLIT && !FP8 && !PAIR && !Q8 && EPI == kEpiGateUpAct),
                "cp.async row gather: bf16 gate/up pass on one-CTA tiles");
  using Cfg = StageCfg<SPLIT, FP8, PAIR>;
  // fp8 weights: fp16 operands; everything else: bf16 operands
  constexpr bool F16 = FP8;
  constexpr int KE = Q8 ? 128 : BK;  // K elements per stage (128 bytes of every operand row)
  constexpr int STAGES = Cfg::kStages;
  constexpr int STAGE_BYTES = Cfg::kStageBytes;
  constexpr int A_BYTES = Cfg::kABytes;
  constexpr int TILE_M = Cfg::kTileM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // stage s: [A hi | A lo (SPLIT) | B], every tile 1024-byte aligned
  auto stage_a = [&](int st) { return base + st * STAGE_BYTES; };
  auto stage_b = [&](int st) { return base + st * STAGE_BYTES + A_BYTES; };
  auto stage_raw = [&](int st) { return base + st * STAGE_BYTES + A_BYTES + Cfg::kBBytes; };
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(base + STAGES * STAGE_BYTES);
  float* epi_stage = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ctrl) + sizeof(Ctrl));
  // the same bytes as 1024-byte-aligned 4 KB staging tiles of the TMA stores,
  // one per epilogue warp (16 KB + alignment within EPI_STAGE_BYTES)
  uint8_t* tma_stage = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(epi_stage) + 1023) & ~static_cast<uintptr_t>(1023));
  volatile int* abort_flag = &ctrl->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.G;
  // PAIR: rank 0 (the leader) issues the MMAs; both CTAs load, convert and drain.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int work0 = PAIR ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int work_stride = PAIR ? static_cast<int>(nclusters_x()) : static_cast<int>(gridDim.x);

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // fp8: the stage is full once the A bytes landed and all converter
      // threads stored their part of the 16-bit B tile
      // (one arrival per converter warp; in a pair both CTAs' converters and
      // A loads report to the leader's barrier)
      // (CPG: the producer's B bytes plus one cp.async arrival per gather thread)
      mbar_init(&ctrl->full[s], FP8 ? 1 + Cfg::kConvWarps * (PAIR ? 2 : 1) : CPG ? 1 + BM : 1);
      mbar_init(&ctrl->empty[s], 1);
      mbar_init(&ctrl->raw_full[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&ctrl->tfull[a], 1);
      mbar_init(&ctrl->tempty[a], 128 * (PAIR ? 2 : 1));
    }
    mbar_init(&ctrl->xch_full, 64);   // swapped gate/up tail: the 64 up-feature threads
    mbar_init(&ctrl->xch_empty, 64);  // ... and the 64 gate-feature threads
    // tile queue: filled by the leader's producer; emptied by the MMA thread,
    // the 4 epilogue warps and the gather / converter warps of a one-CTA tile,
    // or, in a pair, by the leader's MMA thread and epilogue warps and the
    // peer's producer warp and epilogue warps (all on the leader's barrier)
    for (int q = 0; q < TQ_DEPTH; ++q) {
      mbar_init(&ctrl->tq_full[q], 1);
      mbar_init(&ctrl->tq_empty[q], PAIR ? 10 : 5 + (CPG ? 4 : FP8 ? Cfg::kConvWarps : 0));
    }
    ctrl->abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    if (SPLIT) tma_prefetch_desc(&tmap_a_lo);
    tma_prefetch_desc(&tmap_b);
    if (PAIR && EPI == kEpiGateUpAct) tma_prefetch_desc(&tmap_b_tail);
    if (PAIR) tma_prefetch_desc(&tmap_a_tail);
    if (PAIR && SPLIT) tma_prefetch_desc(&tmap_a_lo_tail);
    if (p.sh_rows > 0) {
      tma_prefetch_desc(&tmap_b2);
      if (PAIR) tma_prefetch_desc(&tmap_b2_tail);
    }
    if (p.tma_out) tma_prefetch_desc(&tmap_out);
  }
  if (warp == 1) {
    if (PAIR) {  // collective over one warp of each CTA of the pair
      tmem_alloc_pair(&ctrl->tmem_slot, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&ctrl->tmem_slot, TMEM_COLS);
      tmem_relinquish();
    }
  }
  if (warp == 2) build_schedule(ctrl, p.group_offsets, G, p.M, TILE_M, p.err, lane, p.lpt, p.sh_rows);
  tc_fence_before_sync();
  __syncthreads();
  if (PAIR) cluster_sync();  // the peer's barriers exist before anyone signals them
  tc_fence_after_sync();

  const uint32_t tmem_base = ctrl->tmem_slot;
  const int total_tiles = ctrl->tile_start[G] * p.n_tiles * p.ksplit;
  const int KB = (p.K + KE - 1) / KE;
  // work item t = (output tile t / ksplit, K split t % ksplit)
  auto kb_range = [&](int t, int& kb0, int& kb1) {
    kb0 = (t % p.ksplit) * p.kbs;
    kb1 = min(KB, kb0 + p.kbs);
  };
  // barrier addresses in the leader CTA (cluster window) for the pair protocol
  auto leader_bar = [&](uint64_t* bar) { return PAIR ? mapa_shared(bar, 0) : smem_u32(bar); };
  // ---------------------------------------------------------------- tile order
  // Static: this CTA (pair) takes tiles work0, work0 + work_stride, ...
  // Dynamic (p.tile_counter): the leader's producer takes each next tile from
  // the global counter (one tile ahead, so that the atomic's latency stays off
  // the load path) and hands it to every role of the CTA (pair) through a
  // ring of TQ_DEPTH slots; an index >= total_tiles ends every role's loop.
  const bool dyn = p.tile_counter != nullptr;
  struct Cursor {
    int t;
    int ahead;  // publisher: published, runs next
    int pend;   // publisher: taken from the counter, published at the next tile
    uint32_t qs, qph;
    bool started;
  };
  auto cursor = [&]() { return Cursor{0, 0, 0, 0u, 0u, false}; };
  // consumer: a whole warp (every lane waits, lane 0 arrives) or one thread
  auto next_tile = [&](Cursor& c, bool whole_warp) -> int {
    if (!dyn) {
      c.t = c.started ? c.t + work_stride : work0;
      c.started = true;
      return c.t;
    }
    const bool got = PAIR ? mbar_wait_cluster(&ctrl->tq_full[c.qs], c.qph, abort_flag)
                          : mbar_wait(&ctrl->tq_full[c.qs], c.qph, abort_flag);
    int t = -1;
    if (got) t = *reinterpret_cast<volatile int*>(&ctrl->tq[c.qs]);
    if (whole_warp) __syncwarp();
    if (got && (!whole_warp || lane == 0)) {
      if (PAIR) mbar_arrive_cluster(leader_bar(&ctrl->tq_empty[c.qs]));
      else mbar_arrive(&ctrl->tq_empty[c.qs]);
    }
    if (++c.qs == TQ_DEPTH) {
      c.qs = 0;
      c.qph ^= 1u;
    }
    return t;  // -1: a wait gave up
  };
  // one slot of the queue, in this CTA and (pair) the peer; lane 0 only
  auto push_tile = [&](Cursor& c, int t) -> bool {
    const bool ok = PAIR ? mbar_wait_cluster(&ctrl->tq_empty[c.qs], c.qph ^ 1u, abort_flag)
                         : mbar_wait(&ctrl->tq_empty[c.qs], c.qph ^ 1u, abort_flag);
    if (ok) {
      ctrl->tq[c.qs] = t;
      mbar_arrive(&ctrl->tq_full[c.qs]);
      if (PAIR) {  // the peer's copy of the slot, then its barrier (release.cluster)
        st_cluster_s32(mapa_shared(&ctrl->tq[c.qs], 1), t);
        mbar_arrive_cluster(mapa_shared(&ctrl->tq_full[c.qs], 1));
      }
    }
    if (++c.qs == TQ_DEPTH) {
      c.qs = 0;
      c.qph ^= 1u;
    }
    return ok;
  };
  // publisher (the leader's producer warp; lane 0 takes tiles and publishes):
  // the queue always holds the tile after the current one, so the other roles
  // (the peer's above all) never wait for an index at a tile boundary, and the
  // atomic for the tile after that is in flight while the current tile loads
  auto publish_tile = [&](Cursor& c) -> int {
    if (!dyn) return next_tile(c, true);
    bool ok = true;
    if (lane == 0) {
      if (!c.started) {
        c.started = true;
        c.t = atomicAdd(p.tile_counter, 1);
        ok = push_tile(c, c.t);
        c.ahead = total_tiles;
        if (ok && c.t < total_tiles) {
          c.ahead = atomicAdd(p.tile_counter, 1);
          ok = push_tile(c, c.ahead);
          if (ok && c.ahead < total_tiles) c.pend = atomicAdd(p.tile_counter, 1);
        }
      } else {
        c.t = c.ahead;
        if (c.t < total_tiles) {  // the pending tile was taken when this one was published
          ok = push_tile(c, c.pend);
          c.ahead = c.pend;
          if (ok && c.ahead < total_tiles) c.pend = atomicAdd(p.tile_counter, 1);
        }
      }
    }
    const int t = __shfl_sync(0xffffffffu, c.t, 0);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    return ok ? t : -1;
  };

  const int nbox = p.bn / 64;
  const int nbox_cta = PAIR ? nbox / 2 : nbox;  // bf16 B boxes this CTA loads
  // swapped tail tile (2-CTA mode): the rows are the MMA N operand.  With a
  // split A (bf16 h_hi / h_lo, or two-term e4m3 rows) CTA 0 loads the first
  // plane of the rows and CTA 1 the second, stacked along N (N = 2 x rows
  // rounded up to 16); with one plane (bf16 x, one-term e4m3 rows) each CTA
  // loads half of the rows (N = rows rounded up to 32, a multiple of 16 per
  // CTA).
  auto is_swap = [&](const TileInfo& ti) {
    return PAIR && p.swap_tail > 0 && ti.rows <= p.swap_tail;
  };
  auto swap_rows = [&](const TileInfo& ti) {
    return SPLIT ? (ti.rows + 15) & ~15 : (ti.rows + 31) & ~31;
  };
  // rows each CTA of the pair loads for a swapped tail, from row swap_row0 on
  constexpr bool kSplitRowsAcrossPair = !SPLIT;
  // the shared expert's group (sh_rows > 0): its own weight maps and scales
  auto is_shared_group = [&](int g) { return p.sh_rows > 0 && g == G - 1; };
  // per-column scales of group g (per = 2 for [gate | up], 1 otherwise)
  auto bscale_base = [&](int g, int per) -> const float* {
    if (is_shared_group(g)) return p.sh_b_scale;
    return p.b_scale ? p.b_scale + static_cast<size_t>(g) * per * p.N : nullptr;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Lane 0 waits for free stages, arms the full barrier and loads B (and A,
    // except in gather mode, where every lane fetches 4 of the tile's 128 A
    // rows straight from x with one tile::gather4 per k-block).
    {
      const bool gather = p.a_gather != nullptr && !CPG;  // TMA tile::gather4 rows
      // L2 priorities: A rows (re-read by every column tile) and B weights
      const uint64_t pol_a = l2_policy_evict_normal();
      const uint64_t pol_b = l2_policy_evict_normal();
      // bytes the (leader's) full barrier waits for: A (+ bf16 B) of every CTA
      const uint32_t tx = CPG ? static_cast<uint32_t>(nbox_cta * B_BOX_BYTES)
                              : (PAIR ? 2u : 1u) * (FP8 ? A_BYTES : A_BYTES + nbox_cta * B_BOX_BYTES);
      const int nraw = PAIR ? 1 : (p.bn + 127) / 128;  // raw e4m3 boxes this CTA loads (fp8)
      uint32_t stage = 0, phase = 0;
      // stages filled by this producer and the barrier phase each fill completes
      // (for the drain after an abort)
      uint32_t fill_mask = 0, fill_par = 0;
      bool ok = true;
      Cursor cur = cursor();
      auto next_p = [&]() { return leader ? publish_tile(cur) : next_tile(cur, true); };
      for (;;) {
        if (!ok) break;
        const int t = next_p();
        if (t < 0) {
          ok = false;
          break;
        }
        if (t >= total_tiles) break;
        const TileInfo ti = decode_tile<TILE_M>(ctrl, G, t / p.ksplit, p.n_tiles, p.cols_per_tile);
        const int my_row0 = ti.row0 + static_cast<int>(rank) * BM;
        // the group's weights: the routed tensor at coordinate g, or the shared
        // expert's own tensor (one matrix, coordinate 0)
        const bool shg = is_shared_group(ti.g);
        const CUtensorMap* bmap = shg ? &tmap_b2 : &tmap_b;
        const CUtensorMap* bmap_tail = shg ? &tmap_b2_tail : &tmap_b_tail;
        const int gb = shg ? 0 : ti.g;
        // gather mode: the source rows of this lane's 4 tile rows (rows past the
        // group repeat the tile's first row; their results are never stored)
        int tr[4] = {0, 0, 0, 0};
        if (gather) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int q = 4 * lane + i;
            const int src = p.a_gather[ti.row0 + (q < ti.rows ? q : 0)] / p.gather_k;
            tr[i] = min(max(src, 0), p.a_rows - 1);
          }
        }
        int kb0, kb1;
        kb_range(t, kb0, kb1);
        const bool swap = is_swap(ti);
        // L2 prefetch of this CTA's weight box (k-block kbp of tile tp): the
        // same coordinates as its load below, for the weight layouts read in
        // one box per stage (K-contiguous e4m3, or bf16 viewed as 64-column blocks)
        const int tn = dyn ? total_tiles : t + work_stride;  // the next tile, when known
        TileInfo tin{};
        int kb0n = 0, kb1n = 0;
        if (p.b_prefetch > 0 && tn < total_tiles) {
          tin = decode_tile<TILE_M>(ctrl, G, tn / p.ksplit, p.n_tiles, p.cols_per_tile);
          kb_range(tn, kb0n, kb1n);
        }
        auto prefetch_b = [&](const TileInfo& tp, int kbp) {
          if (PAIR && is_swap(tp)) return;  // swapped tails load other boxes
          const bool shp = is_shared_group(tp.g);
          const CUtensorMap* pm = shp ? &tmap_b2 : &tmap_b;
          const int gp = shp ? 0 : tp.g;
          const int r = static_cast<int>(rank);
          if (Q8) {
            if (EPI == kEpiGateUpAct) tma_prefetch_l2_4d(pm, kbp * KE, tp.n0, PAIR ? r : 0, gp);
            else tma_prefetch_l2_3d(pm, kbp * KE, tp.n0 + (PAIR ? r * (p.bn / 2) : 0), gp);
          } else if (!FP8 && p.b_wide) {
            if (EPI == kEpiGateUpAct) tma_prefetch_l2_5d(pm, 0, kbp * BK, tp.n0 / 64, PAIR ? r : 0, gp);
            else tma_prefetch_l2_4d(pm, 0, kbp * BK, tp.n0 / 64 + (PAIR ? r * nbox_cta : 0), gp);
          }
        };
        // swapped tail: each CTA loads its rows in 32-row boxes (the gate/up
        // pass: rows r * R/2 .. of the tile; the down pass: CTA 0 the h_hi rows,
        // CTA 1 the h_lo rows) and its 128 weight features
        const int swap_boxes =
            swap ? ((kSplitRowsAcrossPair ? swap_rows(ti) / 2 : swap_rows(ti)) + 31) / 32 : 0;
        const uint32_t tile_tx =
            swap ? 2u * (static_cast<uint32_t>(swap_boxes) * 32u * 128u + 2u * B_BOX_BYTES) : tx;
        const int swap_row0 =
            ti.row0 + (kSplitRowsAcrossPair ? static_cast<int>(rank) * (swap_rows(ti) / 2) : 0);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (lane == 0) ok = mbar_wait(&ctrl->empty[stage], phase ^ 1u, abort_flag);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          if (lane == 0 && leader) mbar_arrive_expect_tx(&ctrl->full[stage], tile_tx);
          __syncwarp();
          const uint32_t fbar = leader_bar(&ctrl->full[stage]);
          uint8_t* a_dst = stage_a(stage);
          uint8_t* b_dst = stage_b(stage);
          if (PAIR && swap) {
            if (lane == 0) {
              const CUtensorMap* am = (SPLIT && rank == 1) ? &tmap_a_lo_tail : &tmap_a_tail;
              for (int i = 0; i < swap_boxes; ++i)
                tma_load_2d_pair(a_dst + i * 32 * 128, am, fbar, kb * KE, swap_row0 + 32 * i, pol_a);
              if (Q8) {
                // K-contiguous e4m3 weights: CTA r its 64 gate rows n0 + 64 r .. and
                // the matching 64 up rows, or its 128 output rows n0 + 128 r ..
                if (EPI == kEpiGateUpAct)
                  tma_load_4d_pair(b_dst, bmap_tail, fbar, kb * KE, ti.n0 + 64 * static_cast<int>(rank), 0,
                                   gb, pol_b);
                else
                  tma_load_3d_pair(b_dst, bmap, fbar, kb * KE, ti.n0 + static_cast<int>(rank) * (p.bn / 2),
                                   gb, pol_b);
              } else if (EPI == kEpiGateUpAct) {
                // gate and up features n0 + 64 r .. + 63: one box each
                if (p.b_wide) {
                  tma_load_5d_pair(b_dst, bmap_tail, fbar, 0, kb * BK, ti.n0 / 64 + static_cast<int>(rank),
                                   0, gb, pol_b);
                } else {
                  tma_load_4d_pair(b_dst, bmap_tail, fbar, ti.n0 + 64 * static_cast<int>(rank), 0,
                                   kb * BK, gb, pol_b);
                  tma_load_4d_pair(b_dst + B_BOX_BYTES, bmap_tail, fbar,
                                   ti.n0 + 64 * static_cast<int>(rank), 1, kb * BK, gb, pol_b);
                }
              } else if (p.b_wide) {
                tma_load_4d_pair(b_dst, bmap, fbar, 0, kb * BK,
                                 ti.n0 / 64 + static_cast<int>(rank) * nbox_cta, gb, pol_b);
              } else {
                const int c0 = ti.n0 + static_cast<int>(rank) * 64 * nbox_cta;
                for (int j = 0; j < nbox_cta; ++j)
                  tma_load_3d_pair(b_dst + j * B_BOX_BYTES, bmap, fbar, c0 + 64 * j, kb * BK,
                                   gb, pol_b);
              }
            }
            fill_mask |= 1u << stage;
            fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if (gather) {
            tma_gather4_2d(a_dst + lane * 4 * 128, &tmap_a, &ctrl->full[stage], kb * KE, tr[0],
                           tr[1], tr[2], tr[3], pol_a);
            if (Q8 && SPLIT)  // the lo terms of the same rows
              tma_gather4_2d(a_dst + A_TILE_BYTES + lane * 4 * 128, &tmap_a_lo, &ctrl->full[stage],
                             kb * KE, tr[0], tr[1], tr[2], tr[3], pol_a);
          }
          if (lane == 0) {
          if (!gather && !CPG) {
            if (PAIR) {
              tma_load_2d_pair(a_dst, &tmap_a, fbar, kb * KE, my_row0, pol_a);
              if (SPLIT)
                tma_load_2d_pair(a_dst + A_TILE_BYTES, &tmap_a_lo, fbar, kb * KE, my_row0, pol_a);
            } else {
              tma_load_2d(a_dst, &tmap_a, &ctrl->full[stage], kb * KE, my_row0, pol_a);
              if (SPLIT)
                tma_load_2d(a_dst + A_TILE_BYTES, &tmap_a_lo, &ctrl->full[stage], kb * KE,
                            my_row0, pol_a);
            }
          }
          if (Q8) {
            // e4m3 weights, K contiguous: 128-byte rows of the B tile (the gate/up
            // pass: 128 gate rows then the 128 matching up rows; rank r of a pair
            // its half: the gate rows (0) or the up rows (1), or output rows
            // n0 + r * bn / 2 ..)
            if (EPI == kEpiGateUpAct) {
              if (PAIR)
                tma_load_4d_pair(b_dst, bmap, fbar, kb * KE, ti.n0, static_cast<int>(rank), gb,
                                 pol_b);
              else
                tma_load_4d(b_dst, bmap, &ctrl->full[stage], kb * KE, ti.n0, 0, gb, pol_b);
            } else {
              if (PAIR)
                tma_load_3d_pair(b_dst, bmap, fbar, kb * KE,
                                 ti.n0 + static_cast<int>(rank) * (p.bn / 2), gb, pol_b);
              else
                tma_load_3d(b_dst, bmap, &ctrl->full[stage], kb * KE, ti.n0, gb, pol_b);
            }
          } else if (FP8) {
            // raw e4m3 boxes land on this CTA's own barrier for its converters
            uint8_t* r_dst = stage_raw(stage);
            mbar_arrive_expect_tx(&ctrl->raw_full[stage], nraw * RAW_BOX_BYTES);
            if (EPI == kEpiGateUpAct) {
              if (PAIR) {  // rank 0: gate half, rank 1: up half
                tma_load_4d(r_dst, bmap, &ctrl->raw_full[stage], ti.n0, static_cast<int>(rank),
                            kb * BK, gb, pol_b);
              } else {
                tma_load_4d(r_dst, bmap, &ctrl->raw_full[stage], ti.n0, 0, kb * BK, gb, pol_b);
                tma_load_4d(r_dst + RAW_BOX_BYTES, bmap, &ctrl->raw_full[stage], ti.n0, 1,
                            kb * BK, gb, pol_b);
              }
            } else {
              const int c0 = ti.n0 + (PAIR ? 128 * static_cast<int>(rank) : 0);
              for (int j = 0; j < nraw; ++j)
                tma_load_3d(r_dst + j * RAW_BOX_BYTES, bmap, &ctrl->raw_full[stage],
                            c0 + 128 * j, kb * BK, gb, pol_b);
            }
          } else if (p.b_wide) {
            // one load brings this CTA's whole B share: 64-column blocks
            // n0/64 .. (gate then up in the gate/up pass; rank r its half in a pair)
            if (EPI == kEpiGateUpAct) {
              if (PAIR)
                tma_load_5d_pair(b_dst, bmap, fbar, 0, kb * BK, ti.n0 / 64, static_cast<int>(rank),
                                 gb, pol_b);
              else
                tma_load_5d(b_dst, bmap, &ctrl->full[stage], 0, kb * BK, ti.n0 / 64, 0, gb,
                            pol_b);
            } else {
              if (PAIR)
                tma_load_4d_pair(b_dst, bmap, fbar, 0, kb * BK,
                                 ti.n0 / 64 + static_cast<int>(rank) * nbox_cta, gb, pol_b);
              else
                tma_load_4d(b_dst, bmap, &ctrl->full[stage], 0, kb * BK, ti.n0 / 64, gb, pol_b);
            }
          } else if (EPI == kEpiGateUpAct) {
            if (PAIR) {  // rank 0: gate columns n0..n0+127, rank 1: up columns
              for (int j = 0; j < 2; ++j)
                tma_load_4d_pair(b_dst + j * B_BOX_BYTES, bmap, fbar, ti.n0 + 64 * j,
                                 static_cast<int>(rank), kb * BK, gb, pol_b);
            } else {
              // gate columns n0..n0+127 into boxes 0,1; up columns into boxes 2,3
              for (int j = 0; j < 2; ++j) {
                tma_load_4d(b_dst + j * B_BOX_BYTES, bmap, &ctrl->full[stage], ti.n0 + 64 * j,
                            0, kb * BK, gb, pol_b);
                tma_load_4d(b_dst + (2 + j) * B_BOX_BYTES, bmap, &ctrl->full[stage],
                            ti.n0 + 64 * j, 1, kb * BK, gb, pol_b);
              }
            }
          } else {
            if (PAIR) {  // rank r: columns n0 + r*bn/2 ...
              const int c0 = ti.n0 + static_cast<int>(rank) * 64 * nbox_cta;
              for (int j = 0; j < nbox_cta; ++j)
                tma_load_3d_pair(b_dst + j * B_BOX_BYTES, bmap, fbar, c0 + 64 * j, kb * BK,
                                 gb, pol_b);
            } else {
              for (int j = 0; j < nbox; ++j)
                tma_load_3d(b_dst + j * B_BOX_BYTES, bmap, &ctrl->full[stage], ti.n0 + 64 * j,
                            kb * BK, gb, pol_b);
            }
          }
          if (p.b_prefetch > 0) {  // this CTA's weight box b_prefetch k-blocks ahead
            const int kbp = kb + p.b_prefetch;
            if (kbp < kb1) prefetch_b(ti, kbp);
            else if (tn < total_tiles && kb0n + (kbp - kb1) < kb1n) prefetch_b(tin, kb0n + (kbp - kb1));
          }
          }  // lane 0
          fill_mask |= 1u << stage;
          fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (lane == 0 && (!ok || *abort_flag)) {
        ctrl->abort = 1;
        if (!ok) atomicOr(p.err, MOE_DEV_WAIT_TIMEOUT);
        // let this CTA's copies in flight land before it leaves: wait (bounded)
        // for the phase of every stage filled (its bytes; in a pair the leader's
        // barrier counts both CTAs' bytes), then a short grace period
        for (int st = 0; st < STAGES; ++st) {
          if (!((fill_mask >> st) & 1u)) continue;
          const uint32_t par = (fill_par >> st) & 1u;
          if (FP8) mbar_wait_drain(&ctrl->raw_full[st], par);
          if (leader) mbar_wait_drain(&ctrl->full[st], par);
        }
        drain_grace();
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      const uint32_t idesc = F16 ? make_idesc_f16_f32(TILE_M, p.bn, 0, 1)
                                 : make_idesc_bf16_f32(TILE_M, p.bn, 0, 1);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      Cursor cur = cursor();
      for (;;) {
        if (!ok) break;
        const int t = next_tile(cur, false);
        if (t < 0) {
          ok = false;
          break;
        }
        if (t >= total_tiles) break;
        if (!mbar_wait(&ctrl->tempty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * ACC_STRIDE;
        int kb0, kb1;
        kb_range(t, kb0, kb1);
        const TileInfo ti = decode_tile<TILE_M>(ctrl, G, t / p.ksplit, p.n_tiles, p.cols_per_tile);
        const bool swap = is_swap(ti);
        // swapped tail: A = weights (N-major boxes: MN-major operand), B = rows
        // (K-major), N = rows (gate/up) or 2 x rows (down: h_hi | h_lo)
        const uint32_t idesc_swap =
            Q8 ? make_idesc_e4m3_f32(TILE_M, (SPLIT ? 2 : 1) * swap_rows(ti))
               : make_idesc_bf16_f32(TILE_M, (SPLIT ? 2 : 1) * swap_rows(ti), 1, 0);
        const uint32_t idesc_q8 = make_idesc_e4m3_f32(TILE_M, p.bn);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&ctrl->full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          // A rows written by the gather warps' cp.async (generic proxy), read
          // by the tensor core (async proxy)
          if (CPG) fence_proxy_async_smem();
          if (PAIR && swap && Q8) {
            // weights (K-major, 128 rows per CTA) as the M = 256 operand; the
            // hi rows (CTA 0) and lo rows (CTA 1), or each CTA's half of the
            // one-term rows, as N
            const uint64_t wdesc0 = make_smem_desc_sw128(smem_u32(stage_b(stage)), 16, 1024);
            const uint64_t rdesc0 = make_smem_desc_sw128(smem_u32(stage_a(stage)), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < KE / 32; ++kk)
              tc_mma_f8_pair(d_tmem, smem_desc_advance(wdesc0, kk * 32), smem_desc_advance(rdesc0, kk * 32),
                             idesc_swap, ((kb - kb0) | kk) != 0);
            tc_commit_pair_multicast(&ctrl->empty[stage], 0x3);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if (PAIR && swap) {
            const uint64_t wdesc0 = make_smem_desc_sw128(smem_u32(stage_b(stage)), B_BOX_BYTES, 1024);
            const uint64_t rdesc0 = make_smem_desc_sw128(smem_u32(stage_a(stage)), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              tc_mma_f16_pair(d_tmem, smem_desc_advance(wdesc0, kk * 2048),
                              smem_desc_advance(rdesc0, kk * 32), idesc_swap,
                              ((kb - kb0) | kk) != 0);
            tc_commit_pair_multicast(&ctrl->empty[stage], 0x3);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if (Q8) {
            // A hi / lo and B all K-major with 128-byte rows; a K step of 32
            // e4m3 is 32 bytes.  acc += hi * B, then += lo * B (one-term rows:
            // the hi product only).
            const uint64_t adesc0 = make_smem_desc_sw128(smem_u32(stage_a(stage)), 16, 1024);
            const uint64_t bdesc0 = make_smem_desc_sw128(smem_u32(stage_b(stage)), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < KE / 32; ++kk) {
              const uint64_t bdesc = smem_desc_advance(bdesc0, kk * 32);
              const uint64_t ahi = smem_desc_advance(adesc0, kk * 32);
              const uint64_t alo = smem_desc_advance(adesc0, A_TILE_BYTES + kk * 32);
              if (PAIR) {
                tc_mma_f8_pair(d_tmem, ahi, bdesc, idesc_q8, ((kb - kb0) | kk) != 0);
                if (SPLIT) tc_mma_f8_pair(d_tmem, alo, bdesc, idesc_q8, 1);
              } else {
                tc_mma_f8(d_tmem, ahi, bdesc, idesc_q8, ((kb - kb0) | kk) != 0);
                if (SPLIT) tc_mma_f8(d_tmem, alo, bdesc, idesc_q8, 1);
              }
            }
            if (PAIR) tc_commit_pair_multicast(&ctrl->empty[stage], 0x3);
            else tc_commit(&ctrl->empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          // A: K-major, 128-byte rows; a K step of 16 bf16 is 32 bytes.
          // B: N-major, 64-column boxes 8 KB apart; a K step of 16 rows is 2 KB.
          const uint64_t adesc0 = make_smem_desc_sw128(smem_u32(stage_a(stage)), 16, 1024);
          const uint64_t bdesc0 = make_smem_desc_sw128(smem_u32(stage_b(stage)), B_BOX_BYTES, 1024);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t adesc = smem_desc_advance(adesc0, kk * 32);
            const uint64_t bdesc = smem_desc_advance(bdesc0, kk * 2048);
            if (PAIR) tc_mma_f16_pair(d_tmem, adesc, bdesc, idesc, ((kb - kb0) | kk) != 0);
            else tc_mma_f16(d_tmem, adesc, bdesc, idesc, ((kb - kb0) | kk) != 0);
            if (SPLIT) {
              const uint64_t adesc_lo = smem_desc_advance(adesc0, A_TILE_BYTES + kk * 32);
              if (PAIR) tc_mma_f16_pair(d_tmem, adesc_lo, bdesc, idesc, 1);
              else tc_mma_f16(d_tmem, adesc_lo, bdesc, idesc, 1);
            }
          }
          if (PAIR) tc_commit_pair_multicast(&ctrl->empty[stage], 0x3);
          else tc_commit(&ctrl->empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (PAIR) tc_commit_pair_multicast(&ctrl->tfull[acc], 0x3);
        else tc_commit(&ctrl->tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        ctrl->abort = 1;
        atomicOr(p.err, MOE_DEV_WAIT_TIMEOUT);
      }
    }
    __syncwarp();
  } else if (warp >= 6) {
    // ------------------------------------------------------------ row gather
    // Warps 6..9 fill the A tiles: warp w the rows 32 w .. 32 w + 31, eight
    // lanes per row, so that one copy instruction reads four whole 128-byte
    // row segments (k-block kb of source row x[a_gather[row] / k]) and lane
    // l copies piece l % 8 of row 32 w + 4 j + l / 8 (j = 0..7) into the
    // 128-byte-swizzled K-major layout the MMA reads (piece c of row r at
    // c ^ (r & 7)).  Columns past K are zeros; rows past the group are not
    // loaded (their results are never stored).  Each thread then arrives on
    // the stage's full barrier once its copies have landed.
    if (CPG) {
      const int gw = warp - 6;
      const int piece = lane & 7;
      const __nv_bfloat16* src_base = static_cast<const __nv_bfloat16*>(p.a_src);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      Cursor cur = cursor();
      for (;;) {
        if (!ok) break;
        const int t = next_tile(cur, true);
        if (t < 0) {
          ok = false;
          break;
        }
        if (t >= total_tiles) break;
        const TileInfo ti = decode_tile<TILE_M>(ctrl, G, t / p.ksplit, p.n_tiles, p.cols_per_tile);
        const __nv_bfloat16* src_row[8];
        uint32_t live = 0;  // bit j: row 32 gw + 4 j + lane / 8 is inside the group
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int r = 32 * gw + 4 * jj + (lane >> 3);
          src_row[jj] = src_base;
          if (r < ti.rows) {
            const int src = p.a_gather[ti.row0 + r] / p.gather_k;
            src_row[jj] = src_base + static_cast<size_t>(min(max(src, 0), p.a_rows - 1)) * p.K;
            live |= 1u << jj;
          }
        }
        int kb0, kb1;
        kb_range(t, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (lane == 0) ok = mbar_wait(&ctrl->empty[stage], phase ^ 1u, abort_flag);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          const int kc = kb * BK + 8 * piece;  // K is a multiple of 8: a piece is all in or all out
          const uint32_t nbytes = kc < p.K ? 16u : 0u;
          const int koff = kc < p.K ? kc : 0;
          const uint32_t a0 = smem_u32(stage_a(stage));
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const uint32_t r = static_cast<uint32_t>(32 * gw + 4 * jj + (lane >> 3));
            if ((live >> jj) & 1u)
              cp_async_16(a0 + r * 128u + ((static_cast<uint32_t>(piece) ^ (r & 7u)) << 4),
                          src_row[jj] + koff, nbytes);
          }
          cp_async_mbar_arrive_noinc(&ctrl->full[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && lane == 0) {
        ctrl->abort = 1;
        atomicOr(p.err, MOE_DEV_WAIT_TIMEOUT);
      }
      cp_async_wait_all();  // this thread's copies land before the CTA may leave
    }
    // ------------------------------------------------------------ fp8 converters
    if (FP8) {
      constexpr int NCONV = Cfg::kConvWarps * 32;
      const int tid = threadIdx.x - 6 * 32;  // 0 .. NCONV - 1
      const int nraw = PAIR ? 1 : (p.bn + 127) / 128;
      // 16-byte chunk q = tid + NCONV * i of the stage's raw boxes (512 per box):
      // its offset in the raw boxes and those of its two fp16 chunks
      constexpr int kConvIters = 2 * 512 / NCONV;
      static_assert(2 * 512 % NCONV == 0, "converter threads divide the raw chunks");
      const int conv_iters = nraw * 512 / NCONV;
      uint32_t conv_src[kConvIters], conv_dst0[kConvIters], conv_dst1[kConvIters];
#pragma unroll
      for (int i = 0; i < kConvIters; ++i) {
        const int q = tid + NCONV * i;
        const int b = q >> 9, r = (q >> 3) & 63, cc = q & 7;
        conv_src[i] = b * RAW_BOX_BYTES + r * 128 + ((cc ^ (r & 7)) << 4);
        const int j = 2 * b + (cc >> 2);  // 64-column fp16 box
        const int lc = 2 * (cc & 3);      // first logical 16-byte chunk in the row
        conv_dst0[i] = j * B_BOX_BYTES + r * 128 + ((lc ^ (r & 7)) << 4);
        conv_dst1[i] = j * B_BOX_BYTES + r * 128 + (((lc + 1) ^ (r & 7)) << 4);
      }
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      Cursor cur = cursor();
      for (;;) {
        if (!ok) break;
        const int t = next_tile(cur, true);
        if (t < 0) {
          ok = false;
          break;
        }
        if (t >= total_tiles) break;
        int kb0, kb1;
        kb_range(t, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&ctrl->raw_full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          const uint8_t* raw = stage_raw(stage);
          uint8_t* dst = stage_b(stage);
          // raw box b: 64 rows x 128 bytes (128 e4m3 columns), 128-byte swizzled;
          // each thread expands 16-byte raw chunks into two 16-byte fp16 chunks of
          // the N-major fp16 boxes (64 columns each) the MMA descriptor reads.
          // The chunk offsets depend only on the thread (computed once, above).
#pragma unroll
          for (int i = 0; i < kConvIters; ++i) {
            if (i < conv_iters) {
              const uint4 v = *reinterpret_cast<const uint4*>(raw + conv_src[i]);
              const uint2 o0 = e4m3x4_to_f16x4(v.x), o1 = e4m3x4_to_f16x4(v.y);
              const uint2 o2 = e4m3x4_to_f16x4(v.z), o3 = e4m3x4_to_f16x4(v.w);
              *reinterpret_cast<uint4*>(dst + conv_dst0[i]) = make_uint4(o0.x, o0.y, o1.x, o1.y);
              *reinterpret_cast<uint4*>(dst + conv_dst1[i]) = make_uint4(o2.x, o2.y, o3.x, o3.y);
            }
          }
          fence_proxy_async_smem();  // generic-proxy stores -> tensor core reads
          __syncwarp();
          if (lane == 0) {
            if (PAIR) mbar_arrive_cluster(leader_bar(&ctrl->full[stage]));
            else mbar_arrive(&ctrl->full[stage]);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && tid == 0) {
        ctrl->abort = 1;
        atomicOr(p.err, MOE_DEV_WAIT_TIMEOUT);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes [32*quarter, 32*quarter + 32)
    const int row_in_tile = quarter * 32 + lane;
    uint32_t acc = 0, acc_phase = 0, xch_phase = 0;
    Cursor cur = cursor();
    for (;;) {
      const int t = next_tile(cur, true);
      if (t < 0) {
        if (lane == 0) {
          ctrl->abort = 1;
          atomicOr(p.err, MOE_DEV_WAIT_TIMEOUT);
        }
        break;
      }
      if (t >= total_tiles) break;
      TileInfo ti = decode_tile<TILE_M>(ctrl, G, t / p.ksplit, p.n_tiles, p.cols_per_tile);
      ti.row0 += static_cast<int>(rank) * BM;  // this CTA's 128 rows of the tile
      ti.rows -= static_cast<int>(rank) * BM;
      const size_t plane = static_cast<size_t>(t % p.ksplit) * p.M * p.N;
      if (!mbar_wait(&ctrl->tfull[acc], acc_phase, abort_flag)) {
        if (lane == 0) {
          ctrl->abort = 1;
          atomicOr(p.err, MOE_DEV_WAIT_TIMEOUT);
        }
        break;
      }
      __syncwarp();
      tc_fence_after_sync();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * ACC_STRIDE;
      if (PAIR) {
        // ti was shifted to this CTA's half above; the swapped test uses the
        // whole tile's rows
        TileInfo tw = ti;
        tw.row0 -= static_cast<int>(rank) * BM;
        tw.rows += static_cast<int>(rank) * BM;
        if (is_swap(tw)) {
          const int R = swap_rows(tw);  // accumulator columns per plane
          bool ok = true;
          // split rows (two-term e4m3): columns [0, R) hold the hi products
          // of rows 0..R-1, [R, 2R) their lo products
          auto load_cols = [&](int c, uint32_t (&v)[32]) {
            tmem_ld_32x32b_x32(taddr + c, v);
            if (SPLIT) {
              uint32_t lo[32];
              tmem_ld_32x32b_x32(taddr + R + c, lo);
              tc_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(lo[j]));
            } else {
              tc_wait_ld();
            }
          };
          if (EPI == kEpiGateUpAct) {
            // lanes 0..63: gate features, 64..127: the matching up features of
            // output columns n0 + 64 r + (0..63); up values pass through shared memory
            float* up = epi_stage;  // [R <= 64][64]
            const int fl = quarter * 32 + lane;
            const bool is_up = quarter >= 2;
            const int f = ti.n0 + 64 * static_cast<int>(rank) + (fl & 63);
            if (is_up) {
              ok = mbar_wait(&ctrl->xch_empty, xch_phase ^ 1u, abort_flag);
              if (ok) {
#pragma unroll 1
                for (int c = 0; c < R; c += 32) {
                  uint32_t v[32];
                  load_cols(c, v);
#pragma unroll
                  for (int j = 0; j < 32; ++j)
                    if (c + j < R) up[(c + j) * 64 + (fl - 64)] = __uint_as_float(v[j]);
                }
              }
              mbar_arrive(&ctrl->xch_full);
            } else {
              ok = mbar_wait(&ctrl->xch_full, xch_phase, abort_flag);
              __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
              __nv_bfloat16* out_lo = reinterpret_cast<__nv_bfloat16*>(p.out_lo);
              const float* sg = bscale_base(ti.g, 2);
              const float gs = (sg && f < p.N) ? sg[f] : 1.0f;
              const float us = (sg && f < p.N) ? sg[p.N + f] : 1.0f;
#pragma unroll 1
              for (int c = 0; c < R && ok; c += 32) {
                uint32_t v[32];
                load_cols(c, v);
                if (f < p.N) {
#pragma unroll 4
                  for (int j = 0; j < 32; ++j) {
                    if (c + j >= tw.rows) break;
                    const size_t row = static_cast<size_t>(tw.row0 + c + j);
                    const float rs = p.a_row_scale ? p.a_row_scale[row] : 1.0f;
                    const float g = __uint_as_float(v[j]) * rs * gs;
                    const float u = up[(c + j) * 64 + fl] * rs * us;
                    const float hf = ((p.act == MOE_ACT_SWIGLU) ? silu_f(g) : gelu_tanh_f(g)) * u;
                    if (p.h_fp32) {
                      reinterpret_cast<float*>(p.out)[row * p.N + f] = hf;
                    } else {
                      const __nv_bfloat16 hi = __float2bfloat16_rn(hf);
                      out[row * p.N + f] = hi;
                      if (out_lo) out_lo[row * p.N + f] = __float2bfloat16_rn(hf - __bfloat162float(hi));
                    }
                  }
                }
              }
              mbar_arrive(&ctrl->xch_empty);  // the up values may be rewritten
            }
            xch_phase ^= 1u;
          } else {
            // lanes = output features n0 + 128 r + (0..127); columns j (h_hi rows,
            // or hi e4m3 terms) and R + j (h_lo rows, lo terms) add up to row j's
            // result (one plane: column j alone)
            const int f = ti.n0 + 128 * static_cast<int>(rank) + quarter * 32 + lane;
            const float* sb = bscale_base(ti.g, 1);
            const float cs = (sb && f < p.N) ? sb[f] : 1.0f;
#pragma unroll 1
            for (int c = 0; c < R; c += 32) {
              uint32_t hi[32], lo[32];
              tmem_ld_32x32b_x32(taddr + c, hi);
              if (SPLIT) {
                tmem_ld_32x32b_x32(taddr + R + c, lo);
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) lo[j] = 0u;  // +0.0f
              }
              tc_wait_ld();
              if (f < p.N) {
#pragma unroll 4
                for (int j = 0; j < 32; ++j) {
                  if (c + j >= tw.rows) break;
                  const size_t row = static_cast<size_t>(tw.row0 + c + j);
                  const float rs = p.a_row_scale ? p.a_row_scale[row] : 1.0f;
                  const float v = (__uint_as_float(hi[j]) + __uint_as_float(lo[j])) * rs * cs;
                  if (EPI == kEpiCombineF32) {
                    int t;
                    float w;
                    comb_token(p, row, t, w);
                    atomicAdd(reinterpret_cast<float*>(p.out) + static_cast<size_t>(t) * p.N + f, v * w);
                  } else {
                    store_elem(reinterpret_cast<StoreT<FP8 || Q8>*>(p.out), plane + row * p.N + f, v);
                  }
                }
              }
            }
          }
          tc_fence_before_sync();
          mbar_arrive_cluster(leader_bar(&ctrl->tempty[acc]));
          if (!ok) {
            if (lane == 0) {
              ctrl->abort = 1;
              atomicOr(p.err, MOE_DEV_WAIT_TIMEOUT);
            }
            break;
          }
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1u;
          }
          continue;
        }
      }
      const bool valid = row_in_tile < ti.rows;
      const size_t out_row = static_cast<size_t>(ti.row0 + row_in_tile);

      // per-warp staging tile: stg[row_in_warp * 33 + col]
      float* stg = epi_stage + (warp - 2) * EPI_STAGE_FLOATS;
      const int wrow0 = ti.row0 + quarter * 32;                 // first row of this warp
      const int wrows = min(32, max(0, ti.rows - quarter * 32));  // valid rows of this warp
      if (EPI == kEpiGateUpAct) {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
        __nv_bfloat16* out_lo = reinterpret_cast<__nv_bfloat16*>(p.out_lo);
        const float* sg = bscale_base(ti.g, 2);
        const float rs =
            (p.a_row_scale && valid)
                ? p.a_row_scale[p.a_gather ? p.a_gather[out_row] / p.gather_k : out_row]
                : 1.0f;
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t gr[32], ur[32];
          tmem_ld_32x32b_x32(taddr + c, gr);
          tmem_ld_32x32b_x32(taddr + 128 + c, ur);
          tc_wait_ld();
          const int col = ti.n0 + c;
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int cc = col + 8 * v;
              if (cc < p.N) {
                uint32_t packed[4], packed_lo[4];
                float hfull[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  float hv[2], lo[2];
#pragma unroll
                  for (int h2 = 0; h2 < 2; ++h2) {
                    const int idx = 8 * v + 2 * i + h2;
                    float g = __uint_as_float(gr[idx]) * rs;
                    float u = __uint_as_float(ur[idx]) * rs;
                    if (sg) {
                      g *= sg[cc + 2 * i + h2];
                      u *= sg[p.N + cc + 2 * i + h2];
                    }
                    const float a = (p.act == MOE_ACT_SWIGLU) ? silu_f(g) : gelu_tanh_f(g);
                    const float hf = a * u;
                    hfull[2 * i + h2] = hf;
                    hv[h2] = __bfloat162float(__float2bfloat16_rn(hf));
                    lo[h2] = hf - hv[h2];  // exact in fp32
                  }
                  packed[i] = pack_bf16x2(hv[0], hv[1]);
                  packed_lo[i] = pack_bf16x2(lo[0], lo[1]);
                }
                if (p.h_fp32) {
                  float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) +
                                                        out_row * p.N + cc);
                  o[0] = make_float4(hfull[0], hfull[1], hfull[2], hfull[3]);
                  o[1] = make_float4(hfull[4], hfull[5], hfull[6], hfull[7]);
                } else {
                  *reinterpret_cast<uint4*>(out + out_row * p.N + cc) =
                      make_uint4(packed[0], packed[1], packed[2], packed[3]);
                  if (out_lo)
                    *reinterpret_cast<uint4*>(out_lo + out_row * p.N + cc) =
                        make_uint4(packed_lo[0], packed_lo[1], packed_lo[2], packed_lo[3]);
                }
              }
            }
          }
        }
      } else {  // kEpiStoreF32: (acc * row scale * scale[col]) + bias[col]
        // this split's output plane (bf16 rows for fp8-weight layers)
        using OutT = StoreT<FP8 || Q8>;
        OutT* out = reinterpret_cast<OutT*>(p.out) + plane;
        const float* sc = bscale_base(ti.g, 1);
        const float rs = (p.a_row_scale && valid) ? p.a_row_scale[out_row] : 1.0f;
        // after the transpose lane l owns 4 columns (4 * (l % 8) ..) of rows
        // l / 8, l / 8 + 4, ...: one warp store writes 4 rows x 128 bytes
        const int sub = lane >> 3, c4 = (lane & 7) * 4;
        const bool vec = (p.N % 4) == 0;
        if (EPI == kEpiCombineF32) {
          // fused combine: the token and weight of the 8 rows this lane adds
          int ct[8];
          float cw[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            ct[i] = 0;
            cw[i] = 0.0f;
            if (sub + 4 * i < wrows) comb_token(p, static_cast<size_t>(wrow0 + sub + 4 * i), ct[i], cw[i]);
          }
          float* acc = reinterpret_cast<float*>(p.out);
#pragma unroll 1
          for (int c = 0; c < p.bn; c += 32) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + c, r);
            tc_wait_ld();
            const int col = ti.n0 + c;
            if (col >= p.N) continue;  // warp-uniform
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<float4*>(stg + lane * EPI_STAGE_LD + 4 * j) =
                  make_float4(__uint_as_float(r[4 * j]) * rs, __uint_as_float(r[4 * j + 1]) * rs,
                              __uint_as_float(r[4 * j + 2]) * rs, __uint_as_float(r[4 * j + 3]) * rs);
            __syncwarp();
            const int cl = col + c4;
            float cs[4] = {1.f, 1.f, 1.f, 1.f};
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (sc && cl + i < p.N) cs[i] = sc[cl + i];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int rr = sub + 4 * i;
              if (rr < wrows) {
                const float4 v = *reinterpret_cast<const float4*>(stg + rr * EPI_STAGE_LD + c4);
                float* arow = acc + static_cast<size_t>(ct[i]) * p.N;
                const float w = cw[i];
                if (vec && cl + 4 <= p.N) {
                  atomicAdd(reinterpret_cast<float4*>(arow + cl),
                            make_float4(v.x * cs[0] * w, v.y * cs[1] * w, v.z * cs[2] * w, v.w * cs[3] * w));
                } else {
                  if (cl < p.N) atomicAdd(arow + cl, v.x * cs[0] * w);
                  if (cl + 1 < p.N) atomicAdd(arow + cl + 1, v.y * cs[1] * w);
                  if (cl + 2 < p.N) atomicAdd(arow + cl + 2, v.z * cs[2] * w);
                  if (cl + 3 < p.N) atomicAdd(arow + cl + 3, v.w * cs[3] * w);
                }
              }
            }
          }
        } else {
        // TMA stores (p.tma_out): a warp holding 32 valid rows writes its chunk
        // of 128-byte rows (32 fp32 or 64 bf16 columns) into its 4 KB staging
        // tile with the 128-byte swizzle (16-byte piece q of row r at q ^ (r & 7):
        // conflict-free) and one lane stores the box; a warp with fewer rows (a
        // group's last tile) takes the masked row stores below
        constexpr int CW = (FP8 || Q8) ? 64 : 32;  // output columns per box
        const bool full_warp = p.tma_out && wrows == 32;
        uint8_t* tst = tma_stage + (warp - 2) * 4096;
#pragma unroll 1
        for (int c0 = 0; c0 < p.bn; c0 += CW) {
          if (c0 + CW > p.bn) break;  // bn is a multiple of 64
          uint32_t rv[CW];
          tmem_ld_32x32b_x32(taddr + c0, *reinterpret_cast<uint32_t(*)[32]>(&rv[0]));
          if (CW == 64) tmem_ld_32x32b_x32(taddr + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&rv[CW - 32]));
          tc_wait_ld();
          if (ti.n0 + c0 >= p.N) continue;  // warp-uniform
          if (p.tma_out) {
            if (lane == 0) bulk_wait_read0();  // the last store has read the staging tile
            __syncwarp();
          }
          if (full_warp) {
            // lane l: the column scales of columns n0 + c0 + l (+ 32)
            float csl[CW / 32];
#pragma unroll
            for (int h = 0; h < CW / 32; ++h) {
              const int cc = ti.n0 + c0 + 32 * h + lane;
              csl[h] = (sc && cc < p.N) ? sc[cc] : 1.0f;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {  // 16-byte piece q of this lane's row
              uint4 w;
              uint32_t* wv = reinterpret_cast<uint32_t*>(&w);
              if (CW == 32) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const int j = 4 * q + i;
                  wv[i] = __float_as_uint(__uint_as_float(rv[j]) * rs * __shfl_sync(0xffffffffu, csl[0], j));
                }
              } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const int j = 8 * q + 2 * i;
                  const float a = __uint_as_float(rv[j]) * rs *
                                  __shfl_sync(0xffffffffu, csl[j >> 5], j & 31);
                  const float b = __uint_as_float(rv[j + 1]) * rs *
                                  __shfl_sync(0xffffffffu, csl[(j + 1) >> 5], (j + 1) & 31);
                  wv[i] = pack_bf16x2(a, b);
                }
              }
              *reinterpret_cast<uint4*>(tst + lane * 128 + ((q ^ (lane & 7)) << 4)) = w;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmap_out, tst, ti.n0 + c0, wrow0);
              bulk_commit();
            }
            continue;
          }
        // masked row stores: each 32-column piece staged (fp32) in this warp's
        // own 4 KB tile with the same swizzle, then written out as 4 rows x 128
        // bytes per warp store (the tile is this warp's alone, so no other
        // warp's bulk store can be reading it)
#pragma unroll
        for (int c1 = 0; c1 < CW; c1 += 32) {
          const int c = c0 + c1;
          const int col = ti.n0 + c;
          if (col >= p.N) continue;  // warp-uniform
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(tst + lane * 128 + ((j ^ (lane & 7)) << 4)) = make_float4(
                __uint_as_float(rv[c1 + 4 * j]) * rs, __uint_as_float(rv[c1 + 4 * j + 1]) * rs,
                __uint_as_float(rv[c1 + 4 * j + 2]) * rs, __uint_as_float(rv[c1 + 4 * j + 3]) * rs);
          __syncwarp();
          const int cl = col + c4;
          float cs[4] = {1.f, 1.f, 1.f, 1.f}, cb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (cl + i < p.N) {
              if (sc) cs[i] = sc[cl + i];
              if (p.bias) cb[i] = p.bias[cl + i];
            }
          }
#pragma unroll 2
          for (int rr = sub; rr < wrows; rr += 4) {
            const float4 v = *reinterpret_cast<const float4*>(tst + rr * 128 + (((lane & 7) ^ (rr & 7)) << 4));
            OutT* orow = out + static_cast<size_t>(wrow0 + rr) * p.N;
            const float o0 = v.x * cs[0] + cb[0], o1 = v.y * cs[1] + cb[1];
            const float o2 = v.z * cs[2] + cb[2], o3 = v.w * cs[3] + cb[3];
            if (vec && cl + 4 <= p.N) {
              if (FP8 || Q8)
                *reinterpret_cast<uint2*>(orow + cl) = make_uint2(pack_bf16x2(o0, o1), pack_bf16x2(o2, o3));
              else
                *reinterpret_cast<float4*>(orow + cl) = make_float4(o0, o1, o2, o3);
            } else {
              if (cl < p.N) store_elem(orow, cl, o0);
              if (cl + 1 < p.N) store_elem(orow, cl + 1, o1);
              if (cl + 2 < p.N) store_elem(orow, cl + 2, o2);
              if (cl + 3 < p.N) store_elem(orow, cl + 3, o3);
            }
          }
        }
        }
        }  // not the fused combine
      }
      tc_fence_before_sync();
      if (PAIR) mbar_arrive_cluster(leader_bar(&ctrl->tempty[acc]));
      else mbar_arrive(&ctrl->tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (p.tma_out && lane == 0) bulk_wait0();  // this lane's output stores are done
    __syncwarp();
  }

  // ---------------------------------------------------------------- teardown
  // the next kernel may be scheduled once every CTA got here (not earlier:
  // its waiting CTAs would sit beside this persistent kernel's for its whole run)
  pdl_launch_dependents();
  tc_fence_before_sync();
  __syncthreads();
  // a pair finishes together: the leader's MMAs read the peer's shared memory
  // and the peer arrives on the leader's barriers
  if (PAIR) cluster_sync();
  if (warp == 1) {
    tc_fence_after_sync();
    if (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}


// ==========================================================================
// Swap-AB grouped GEMM for decode-size groups (a handful of rows per expert).
// The weights become the M = 128 operand (N-major in shared memory, exactly
// the boxes the prefill kernel loads as its B tile) and the group's rows the
// N = 16 / 32 / 64 operand, so each stage is ~24 KB of which 16 KB are
// weights: 6-8 stages keep plenty of weight bytes in flight per SM while each
// active expert's weights stream through once.  The accumulator is
// feature x token (TMEM lane = output feature); the gate/up pass puts 64 gate
// and the 64 matching up features in one tile and pairs them through shared
// memory in the epilogue.
constexpr int DEC_M = 128;                               // MMA M: weight features per tile
constexpr int DEC_NT_MAX = 64;                           // MMA N: rows per tile, at most
constexpr int DEC_W_BYTES = DEC_M * BK * 2;              // 16-bit weight tile, two 64-feature boxes
constexpr int DEC_TOK_BYTES = DEC_NT_MAX * BK * 2;       // row tile (one plane)
constexpr int DEC_RAW_BOX_BYTES = 64 * BK;               // 64 e4m3 features x 64 K, unswizzled
// two accumulators of <= 128 columns (the split down pass stacks the h_hi
// and h_lo rows along N: 2 * rows columns)
constexpr uint32_t DEC_TMEM_COLS = 256;
constexpr int DEC_ACC_STRIDE = 128;
constexpr int DEC_UP_FLOATS = DEC_NT_MAX * 64;           // up values of a gate/up tile

template <bool SPLIT, bool FP8>
struct DecCfg {
  static_assert(!(SPLIT && FP8), "fp8 layers use an unsplit h");
  static constexpr int kTokBytes = (SPLIT ? 2 : 1) * DEC_TOK_BYTES;
  static constexpr int kRawBytes = FP8 ? 2 * DEC_RAW_BOX_BYTES : 0;
  // stage layout: [weights (MMA A) | rows (+ lo rows) (MMA B) | raw e4m3 weights]
  static constexpr int kStageBytes = DEC_W_BYTES + kTokBytes + kRawBytes;
  static constexpr int kStages =
      STAGE_BUDGET / kStageBytes > MAX_STAGES ? MAX_STAGES : STAGE_BUDGET / kStageBytes;
  // fp8: e4m3 -> fp16 converter warps (6 ..); 8 measured slower here (each
  // stage expands only 8 KB of weights)
  static constexpr int kConvWarps = 4;
  static constexpr int kThreads = FP8 ? (6 + kConvWarps) * 32 : 192;
};

template <bool SPLIT, bool FP8>
constexpr size_t dec_smem_bytes() {
  return 1024 + DecCfg<SPLIT, FP8>::kStages * DecCfg<SPLIT, FP8>::kStageBytes + sizeof(Ctrl) +
         DEC_UP_FLOATS * 4;
}
static_assert(dec_smem_bytes<false, false>() <= 227 * 1024, "shared memory budget");
static_assert(dec_smem_bytes<true, false>() <= 227 * 1024, "shared memory budget");
static_assert(dec_smem_bytes<false, true>() <= 227 * 1024, "shared memory budget");

// KParams as for the prefill kernel, read as: M rows (tokens) grouped by
// group_offsets, K reduction, N output features, bn = rows per tile (MMA N),
// cols_per_tile = output features per tile (64 gate/up, 128 down),
// a_row_scale per row.
// Q8: two-term e4m3 rows (the hi rows, then the lo rows, stacked along N as in
// SPLIT) and e4m3 weights stored K-contiguous ([G, N, K]), K-major as the
// M = 128 operand: kind::f8f6f4, 128 K elements per stage, no expansion.
template <int EPI, bool SPLIT, bool FP8, bool Q8>
__global__ void __launch_bounds__(DecCfg<SPLIT, FP8>::kThreads, 1)
    grouped_gemm_decode_kernel(const __grid_constant__ CUtensorMap tmap_rows,
                               const __grid_constant__ CUtensorMap tmap_rows_lo,
                               const __grid_constant__ CUtensorMap tmap_w, const KParams p) {
  pdl_wait();
  static_assert(!Q8 || !FP8, "e4m3 rows meet K-contiguous e4m3 weights, not expanded ones");
  constexpr int KE = Q8 ? 128 : BK;  // K elements per stage (128 bytes of every operand row)
  using Cfg = DecCfg<SPLIT, FP8>;
  constexpr int STAGES = Cfg::kStages;
  constexpr int STAGE_BYTES = Cfg::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  auto stage_w = [&](int st) { return base + st * STAGE_BYTES; };
  auto stage_rows = [&](int st) { return base + st * STAGE_BYTES + DEC_W_BYTES; };
  auto stage_raw = [&](int st) { return base + st * STAGE_BYTES + DEC_W_BYTES + Cfg::kTokBytes; };
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(base + STAGES * STAGE_BYTES);
  float* up_stage = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ctrl) + sizeof(Ctrl));
  volatile int* abort_flag = &ctrl->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.G;
  const int NT = p.bn;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctrl->full[s], FP8 ? 1 + Cfg::kConvWarps : 1);
      mbar_init(&ctrl->empty[s], 1);
      mbar_init(&ctrl->raw_full[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&ctrl->tfull[a], 1);
      mbar_init(&ctrl->tempty[a], 128);
    }
    mbar_init(&ctrl->xch_full, 64);   // the 64 up-feature threads
    mbar_init(&ctrl->xch_empty, 64);  // the 64 gate-feature threads
    ctrl->abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_rows);
    if (SPLIT) tma_prefetch_desc(&tmap_rows_lo);
    tma_prefetch_desc(&tmap_w);
  }
  if (warp == 1) {
    tmem_alloc(&ctrl->tmem_slot, DEC_TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 2) build_schedule(ctrl, p.group_offsets, G, p.M, NT, p.err, lane, p.lpt, p.sh_rows);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  const uint32_t tmem_base = ctrl->tmem_slot;
  const int total_tiles = ctrl->tile_start[G] * p.n_tiles;
  const int KB = (p.K + KE - 1) / KE;
  const uint32_t rows_bytes = static_cast<uint32_t>(NT) * BK * 2;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_rows = l2_policy_evict_normal();
      const uint64_t pol_w = l2_policy_evict_normal();
      const uint32_t tx = (SPLIT ? 2u : 1u) * rows_bytes + (FP8 ? 0u : DEC_W_BYTES);
      uint32_t stage = 0, phase = 0;
      uint32_t fill_mask = 0, fill_par = 0;  // as in the 128-row kernel
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const TileInfo ti = decode_tile_h(ctrl, G, t, p.n_tiles, p.cols_per_tile, NT);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&ctrl->empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&ctrl->full[stage], tx);
          tma_load_2d(stage_rows(stage), &tmap_rows, &ctrl->full[stage], kb * KE, ti.row0, pol_rows);
          if (SPLIT)
            tma_load_2d(stage_rows(stage) + NT * 128, &tmap_rows_lo, &ctrl->full[stage],
                        kb * KE, ti.row0, pol_rows);
          if (Q8) {
            // 128 weight rows of 128 bytes (64 gate rows, then the 64 matching up
            // rows; or 128 consecutive output features)
            if (EPI == kEpiGateUpAct)
              tma_load_4d(stage_w(stage), &tmap_w, &ctrl->full[stage], kb * KE, ti.n0, 0, ti.g,
                          pol_w);
            else
              tma_load_3d(stage_w(stage), &tmap_w, &ctrl->full[stage], kb * KE, ti.n0, ti.g, pol_w);
            fill_mask |= 1u << stage;
            fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          uint8_t* wdst = FP8 ? stage_raw(stage) : stage_w(stage);
          uint64_t* wbar = FP8 ? &ctrl->raw_full[stage] : &ctrl->full[stage];
          const int wbox = FP8 ? DEC_RAW_BOX_BYTES : DEC_W_BYTES / 2;
          if (FP8) mbar_arrive_expect_tx(&ctrl->raw_full[stage], 2 * DEC_RAW_BOX_BYTES);
          if (EPI == kEpiGateUpAct) {  // 64 gate features, then the 64 matching up features
            tma_load_4d(wdst, &tmap_w, wbar, ti.n0, 0, kb * BK, ti.g, pol_w);
            tma_load_4d(wdst + wbox, &tmap_w, wbar, ti.n0, 1, kb * BK, ti.g, pol_w);
          } else {  // 128 consecutive output features
            tma_load_3d(wdst, &tmap_w, wbar, ti.n0, kb * BK, ti.g, pol_w);
            tma_load_3d(wdst + wbox, &tmap_w, wbar, ti.n0 + 64, kb * BK, ti.g, pol_w);
          }
          fill_mask |= 1u << stage;
          fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok || *abort_flag) {
        ctrl->abort = 1;
        if (!ok) atomicOr(p.err, MOE_DEV_WAIT_TIMEOUT);
        for (int st = 0; st < STAGES; ++st) {  // copies in flight land first
          if (!((fill_mask >> st) & 1u)) continue;
          const uint32_t par = (fill_par >> st) & 1u;
          if (FP8) mbar_wait_drain(&ctrl->raw_full[st], par);
          mbar_wait_drain(&ctrl->full[st], par);
        }
        drain_grace();
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // split down pass: the h_lo rows follow the h_hi rows in the stage, so one
      // MMA with N = 2 * NT covers both (accumulator columns NT.. hold the lo
      // products; the epilogue adds them): half the MMA instructions, which
      // at these N are what bounds the pass
      const int mma_n = SPLIT ? 2 * NT : NT;
      const uint32_t idesc = Q8    ? make_idesc_e4m3_f32(DEC_M, mma_n)
                             : FP8 ? make_idesc_f16_f32(DEC_M, mma_n, 1, 0)
                                   : make_idesc_bf16_f32(DEC_M, mma_n, 1, 0);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        if (!mbar_wait(&ctrl->tempty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * DEC_ACC_STRIDE;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&ctrl->full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t bdesc0 = make_smem_desc_sw128(smem_u32(stage_rows(stage)), 16, 1024);
          if (Q8) {
            // A = weights and B = rows, both K-major 128-byte rows; K step of 32 e4m3 = 32 bytes
            const uint64_t adesc0 = make_smem_desc_sw128(smem_u32(stage_w(stage)), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < KE / 32; ++kk)
              tc_mma_f8(d_tmem, smem_desc_advance(adesc0, kk * 32), smem_desc_advance(bdesc0, kk * 32),
                        idesc, (kb | kk) != 0);
          } else {
            // A = weights, N-major: 64-feature groups 8 KB apart, K step of 16 rows = 2 KB
            // B = rows, K-major: 128-byte rows, K step of 16 = 32 bytes
            const uint64_t adesc0 =
                make_smem_desc_sw128(smem_u32(stage_w(stage)), DEC_W_BYTES / 2, 1024);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              tc_mma_f16(d_tmem, smem_desc_advance(adesc0, kk * 2048),
                         smem_desc_advance(bdesc0, kk * 32), idesc, (kb | kk) != 0);
          }
          tc_commit(&ctrl->empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&ctrl->tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        ctrl->abort = 1;
        atomicOr(p.err, MOE_DEV_WAIT_TIMEOUT);
      }
    }
    __syncwarp();
  } else if (warp >= 6) {
    // ------------------------------------------------------------ fp8 converters
    if (FP8) {
      const int tid = threadIdx.x - 6 * 32;
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&ctrl->raw_full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          const uint8_t* raw = stage_raw(stage);
          uint8_t* dst = stage_w(stage);
          // raw box b: 64 rows (K) x 64 bytes (64 e4m3 features), unswizzled;
          // each 16-byte chunk becomes two 16-byte fp16 chunks of the 128B-swizzled
          // 64-feature box b of the weight tile
          constexpr int NCONV = Cfg::kConvWarps * 32;
          static_assert(512 % NCONV == 0, "converter threads divide the stage's 512 chunks");
#pragma unroll
          for (int i = 0; i < 512 / NCONV; ++i) {
            const int q = tid + NCONV * i;
            const int b = q >> 8, r = (q >> 2) & 63, c = q & 3;
            const uint4 v = *reinterpret_cast<const uint4*>(raw + b * DEC_RAW_BOX_BYTES + r * 64 + c * 16);
            const uint2 o0 = e4m3x4_to_f16x4(v.x), o1 = e4m3x4_to_f16x4(v.y);
            const uint2 o2 = e4m3x4_to_f16x4(v.z), o3 = e4m3x4_to_f16x4(v.w);
            uint8_t* row = dst + b * (DEC_W_BYTES / 2) + r * 128;
            *reinterpret_cast<uint4*>(row + (((2 * c) ^ (r & 7)) << 4)) = make_uint4(o0.x, o0.y, o1.x, o1.y);
            *reinterpret_cast<uint4*>(row + (((2 * c + 1) ^ (r & 7)) << 4)) =
                make_uint4(o2.x, o2.y, o3.x, o3.y);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctrl->full[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && tid == 0) {
        ctrl->abort = 1;
        atomicOr(p.err, MOE_DEV_WAIT_TIMEOUT);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int fl = quarter * 32 + lane;  // feature of the tile held by this thread
    uint32_t acc = 0, acc_phase = 0, xch_phase = 0;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
      const TileInfo ti = decode_tile_h(ctrl, G, t, p.n_tiles, p.cols_per_tile, NT);
      if (!mbar_wait(&ctrl->tfull[acc], acc_phase, abort_flag)) {
        if (lane == 0) {
          ctrl->abort = 1;
          atomicOr(p.err, MOE_DEV_WAIT_TIMEOUT);
        }
        break;
      }
      __syncwarp();
      tc_fence_after_sync();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * DEC_ACC_STRIDE;
      uint32_t v[DEC_NT_MAX];
      tmem_ld_32x32b_x32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      if (NT > 32) tmem_ld_32x32b_x32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tc_wait_ld();
      if (SPLIT) {
        // h = h_hi + h_lo: row j's lo products are in column NT + j
        if (NT <= 16) {  // already loaded: columns 16..31
#pragma unroll
          for (int j = 0; j < 16; ++j)
            v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(v[16 + j]));
        } else {
#pragma unroll
          for (int q = 0; q < DEC_NT_MAX / 32; ++q) {
            if (32 * q < NT) {
              uint32_t lo[32];
              tmem_ld_32x32b_x32(taddr + NT + 32 * q, lo);
              tc_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j)
                v[32 * q + j] = __float_as_uint(__uint_as_float(v[32 * q + j]) + __uint_as_float(lo[j]));
            }
          }
        }
      }
      const int rows = ti.rows;
      bool ok = true;
      if (EPI == kEpiGateUpAct) {
        // up features (TMEM lanes 64..127) pass their values to the gate
        // features (lanes 0..63) of the same index through shared memory;
        // both hand-overs are mbarriers with bounded waits
        const bool is_up = quarter >= 2;
        const int f = ti.n0 + (fl & 63);  // output feature (gate and up share the index)
        if (is_up) {
          ok = mbar_wait(&ctrl->xch_empty, xch_phase ^ 1u, abort_flag);
          if (ok) {
#pragma unroll
            for (int j = 0; j < DEC_NT_MAX; ++j)
              if (j < rows) up_stage[j * 64 + (fl - 64)] = __uint_as_float(v[j]);
          }
          mbar_arrive(&ctrl->xch_full);
        } else {
          ok = mbar_wait(&ctrl->xch_full, xch_phase, abort_flag);
        }
        if (ok && !is_up && f < p.N) {
          const float* sg = p.b_scale ? p.b_scale + static_cast<size_t>(ti.g) * 2 * p.N : nullptr;
          const float gs = sg ? sg[f] : 1.0f, us = sg ? sg[p.N + f] : 1.0f;
#pragma unroll 4
          for (int j = 0; j < DEC_NT_MAX; ++j) {
            if (j >= rows) break;
            const size_t row = static_cast<size_t>(ti.row0 + j);
            const float rs = p.a_row_scale ? p.a_row_scale[row] : 1.0f;
            const float g = __uint_as_float(v[j]) * rs * gs;
            const float u = up_stage[j * 64 + fl] * rs * us;
            const float hf = ((p.act == MOE_ACT_SWIGLU) ? silu_f(g) : gelu_tanh_f(g)) * u;
            if (p.h_fp32) {
              reinterpret_cast<float*>(p.out)[row * p.N + f] = hf;
            } else {
              const __nv_bfloat16 hi = __float2bfloat16_rn(hf);
              reinterpret_cast<__nv_bfloat16*>(p.out)[row * p.N + f] = hi;
              if (p.out_lo)
                reinterpret_cast<__nv_bfloat16*>(p.out_lo)[row * p.N + f] =
                    __float2bfloat16_rn(hf - __bfloat162float(hi));
            }
          }
        }
        if (!is_up) mbar_arrive(&ctrl->xch_empty);  // up_stage may be rewritten
        xch_phase ^= 1u;
      } else {
        const int f = ti.n0 + fl;
        if (f < p.N) {
          const float cs = p.b_scale ? p.b_scale[static_cast<size_t>(ti.g) * p.N + f] : 1.0f;
#pragma unroll 4
          for (int j = 0; j < DEC_NT_MAX; ++j) {
            if (j >= rows) break;
            const size_t row = static_cast<size_t>(ti.row0 + j);
            const float rs = p.a_row_scale ? p.a_row_scale[row] : 1.0f;
            if (EPI == kEpiCombineF32) {
              int t;
              float w;
              comb_token(p, row, t, w);
              atomicAdd(reinterpret_cast<float*>(p.out) + static_cast<size_t>(t) * p.N + f,
                        __uint_as_float(v[j]) * rs * cs * w);
            } else {
              store_elem(reinterpret_cast<StoreT<FP8 || Q8>*>(p.out), row * p.N + f,
                         __uint_as_float(v[j]) * rs * cs);
            }
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&ctrl->tempty[acc]);
      if (!ok) {
        if (lane == 0) {
          ctrl->abort = 1;
          atomicOr(p.err, MOE_DEV_WAIT_TIMEOUT);
        }
        break;
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    __syncwarp();
  }

  pdl_launch_dependents();  // at the end, as in the 128-row kernel
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, DEC_TMEM_COLS);
  }
}

}  // namespace

// ------------------------------------------------------------------ host side
namespace {
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}
}  // namespace

bool encode_tmap(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapDataType dt,
                 CUtensorMapSwizzle swz) {
  auto fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t gd[5];
  cuuint64_t gs[4];
  cuuint32_t bx[5];
  cuuint32_t es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
  CUresult r = fn(m, dt, rank, const_cast<void*>(ptr), gd, gs, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

// The store pass's output as a TMA store target: [M, N] rows of fp32 (or
// bf16 when out_bf16), 32 rows x 128 bytes per box, 128-byte swizzle.  Only
// for one-plane outputs without bias (kp.tma_out); otherwise kp.tma_out stays
// 0 and the map is unused.
constexpr bool kTmaStoreEpilogue = true;
void make_out_map(const GroupedGemmArgs& a, KParams& kp, bool out_bf16, CUtensorMap& tout) {
  kp.tma_out = 0;
  if (!kTmaStoreEpilogue || a.epilogue != kEpiStoreF32 || kp.ksplit != 1 || a.bias || !a.out ||
      (reinterpret_cast<uintptr_t>(a.out) & 15u))
    return;
  const uint64_t eb = out_bf16 ? 2 : 4;
  const uint64_t dims[2] = {static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.M)};
  const uint64_t strides[1] = {static_cast<uint64_t>(a.N) * eb};
  if (strides[0] % 16) return;
  const uint32_t box[2] = {out_bf16 ? 64u : 32u, 32u};
  if (encode_tmap(&tout, a.out, 2, dims, strides, box,
                  out_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
    kp.tma_out = 1;
}

template <int EPI, bool SPLIT, bool FP8, bool PAIR, bool Q8 = false, bool CPG = false>
cudaError_t launch_epi(const CUtensorMap& ta, const CUtensorMap& ta_lo, const CUtensorMap& tb,
                       const CUtensorMap& tb_tail, const CUtensorMap& ta_tail,
                       const CUtensorMap& ta_lo_tail, const CUtensorMap& tb2,
                       const CUtensorMap& tb2_tail, const CUtensorMap& tout, const KParams& kp,
                       long long max_tiles,
                       cudaStream_t s) {
  constexpr size_t smem = smem_bytes<SPLIT, FP8, PAIR>();
  constexpr int threads = CPG ? 320 : StageCfg<SPLIT, FP8, PAIR>::kThreads;
  auto kern = grouped_gemm_kernel<EPI, SPLIT, FP8, PAIR, Q8, CPG>;
  // the attribute is per device: set it once for each device this process uses
  static bool done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) done[dev] = true;
  }
  if (!PAIR) {
    const int grid =
        static_cast<int>(std::max<long long>(1, std::min<long long>(device_sm_count(), max_tiles)));
    return launch_kernel(kern, dim3(grid), dim3(threads), smem, s, ta, ta_lo, tb, tb_tail, ta_tail,
                         ta_lo_tail, tb2, tb2_tail, tout, kp);
  }
  // one persistent 2-CTA cluster per SM pair that can hold one
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = g_pdl ? 1 : 0;
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // cluster shape only for the occupancy query
  static int max_clusters[64] = {0};
  if (dev < 0 || dev >= 64 || max_clusters[dev] == 0) {
    cfg.gridDim = dim3(2 * (device_sm_count() / 2), 1, 1);
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess || n < 1) n = device_sm_count() / 2;
    if (dev >= 0 && dev < 64) max_clusters[dev] = n;
    else max_clusters[0] = n;
  }
  const int nclu = static_cast<int>(std::max<long long>(
      1, std::min<long long>(max_clusters[(dev >= 0 && dev < 64) ? dev : 0], max_tiles)));
  cfg.gridDim = dim3(2 * nclu, 1, 1);
  cfg.numAttrs = 2;
  cudaError_t e =
      cudaLaunchKernelEx(&cfg, kern, ta, ta_lo, tb, tb_tail, ta_tail, ta_lo_tail, tb2, tb2_tail, tout, kp);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int g_pair_tiles = 3;      // set through moe_set_option(MOE_OPT_PAIR_TILES, .)
int g_decode_kernel = 1;   // set through moe_set_option(MOE_OPT_DECODE_KERNEL, .)
int g_pdl = 1;             // set through moe_set_option(MOE_OPT_PDL, .)
int g_tile_order = 0;      // set through moe_set_option(MOE_OPT_TILE_ORDER, .)
int g_b_prefetch = 0;      // set through moe_set_option(MOE_OPT_B_PREFETCH, .)

namespace {

// The persistent grid: one CTA (cluster) per tile at most, and at most
// a.max_ctas CTAs when the caller caps it (the shared expert's GEMMs beside the
// routed path: MOE_OPT_SHARED_CTAS).
long long cap_grid(long long tiles, const GroupedGemmArgs& a, bool pair) {
  if (a.max_ctas <= 0) return tiles;
  return std::min<long long>(tiles, std::max(1, pair ? a.max_ctas / 2 : a.max_ctas));
}
template <int EPI, bool SPLIT, bool FP8, bool Q8 = false>
cudaError_t launch_dec(const CUtensorMap& tr, const CUtensorMap& tr_lo, const CUtensorMap& tw,
                       const KParams& kp, long long max_tiles, cudaStream_t s) {
  constexpr size_t smem = dec_smem_bytes<SPLIT, FP8>();
  constexpr int threads = DecCfg<SPLIT, FP8>::kThreads;
  auto kern = grouped_gemm_decode_kernel<EPI, SPLIT, FP8, Q8>;
  static bool done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) done[dev] = true;
  }
  const int grid =
      static_cast<int>(std::max<long long>(1, std::min<long long>(device_sm_count(), max_tiles)));
  return launch_kernel(kern, dim3(grid), dim3(threads), smem, s, tr, tr_lo, tw, kp);
}

// Swap-AB launch for decode-size groups, e4m3 rows and K-contiguous e4m3
// weights: nt rows per tile (two-term rows: 2 nt MMA columns, hi rows then lo
// rows; one-term rows: nt).
cudaError_t launch_grouped_gemm_decode_q8(const GroupedGemmArgs& a, int nt, cudaStream_t s) {
  CUtensorMap tr, tr_lo, tw;
  const uint64_t K = static_cast<uint64_t>(a.K), N = static_cast<uint64_t>(a.N);
  const uint64_t M = static_cast<uint64_t>(a.M), G = static_cast<uint64_t>(a.G);
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const bool one = a.a_e4m3 != 0;  // one-term rows [M, K]; else two-term [M, 2K]
  {
    const uint64_t dims[2] = {K, M};
    const uint64_t strides[1] = {one ? K : 2 * K};
    const uint32_t box[2] = {128, static_cast<uint32_t>(nt)};
    if (!encode_tmap(&tr, a.A, 2, dims, strides, box, u8)) return cudaErrorInvalidValue;
    if (one) tr_lo = tr;
    else if (!encode_tmap(&tr_lo, static_cast<const uint8_t*>(a.A) + K, 2, dims, strides, box, u8))
      return cudaErrorInvalidValue;
  }
  KParams kp{};
  kp.group_offsets = a.group_offsets;
  kp.G = a.G;
  kp.M = a.M;
  kp.K = a.K;
  kp.N = a.N;
  kp.out = a.out;
  kp.b_scale = a.b_scale;
  kp.a_row_scale = a.a_row_scale;
  kp.h_fp32 = a.h_fp32;
  kp.act = a.act;
  kp.err = a.err;
  kp.comb_rows = a.comb_rows;
  kp.comb_w = a.comb_w;
  kp.comb_k = a.comb_k;
  kp.lpt = g_tile_order == 1 && a.group_offsets != nullptr && a.G > 1;
  kp.tile_counter = a.tile_counter;
  kp.b_prefetch = g_b_prefetch;
  kp.sh_rows = a.sh_rows;
  kp.sh_b_scale = a.sh_b_scale;
  kp.bn = nt;
  kp.ksplit = 1;
  kp.kbs = (a.K + 127) / 128;
  if (a.epilogue == kEpiGateUpAct) {  // [G][2][N][K]: 64 gate rows, then the 64 up rows
    const uint64_t dims[4] = {K, N, 2, G};
    const uint64_t strides[3] = {K, N * K, 2 * N * K};
    const uint32_t box[4] = {128, 64, 2, 1};
    if (!encode_tmap(&tw, a.B, 4, dims, strides, box, u8)) return cudaErrorInvalidValue;
    kp.cols_per_tile = 64;
  } else {  // [G][N][K]: 128 output features
    const uint64_t dims[3] = {K, N, G};
    const uint64_t strides[2] = {K, N * K};
    const uint32_t box[3] = {128, 128, 1};
    if (!encode_tmap(&tw, a.B, 3, dims, strides, box, u8)) return cudaErrorInvalidValue;
    kp.cols_per_tile = 128;
  }
  kp.n_tiles = (a.N + kp.cols_per_tile - 1) / kp.cols_per_tile;
  const long long max_tiles = cap_grid(
      (static_cast<long long>((a.M + nt - 1) / nt) + a.G) * static_cast<long long>(kp.n_tiles), a, false);
  if (a.epilogue == kEpiCombineF32)
    return one ? launch_dec<kEpiCombineF32, false, false, true>(tr, tr_lo, tw, kp, max_tiles, s)
               : launch_dec<kEpiCombineF32, true, false, true>(tr, tr_lo, tw, kp, max_tiles, s);
  if (one)
    return a.epilogue == kEpiGateUpAct
               ? launch_dec<kEpiGateUpAct, false, false, true>(tr, tr_lo, tw, kp, max_tiles, s)
               : launch_dec<kEpiStoreF32, false, false, true>(tr, tr_lo, tw, kp, max_tiles, s);
  if (a.epilogue == kEpiGateUpAct)
    return launch_dec<kEpiGateUpAct, true, false, true>(tr, tr_lo, tw, kp, max_tiles, s);
  return launch_dec<kEpiStoreF32, true, false, true>(tr, tr_lo, tw, kp, max_tiles, s);
}

// Swap-AB launch for decode-size groups: nt rows per tile.
cudaError_t launch_grouped_gemm_decode(const GroupedGemmArgs& a, int nt, cudaStream_t s) {
  if (a.a_e4m3x2 || a.a_e4m3) return launch_grouped_gemm_decode_q8(a, nt, s);
  CUtensorMap tr, tr_lo, tw;
  const CUtensorMapDataType adt =
      a.a_fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.K) * 2};
    const uint32_t box[2] = {BK, static_cast<uint32_t>(nt)};
    if (!encode_tmap(&tr, a.A, 2, dims, strides, box, adt)) return cudaErrorInvalidValue;
    if (a.A_lo && !encode_tmap(&tr_lo, a.A_lo, 2, dims, strides, box)) return cudaErrorInvalidValue;
    if (!a.A_lo) tr_lo = tr;
  }
  const uint64_t N = static_cast<uint64_t>(a.N), K = static_cast<uint64_t>(a.K);
  const uint64_t eb = a.b_fp8 ? 1 : 2;
  const CUtensorMapDataType bdt =
      a.b_fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  // 64 features per box: 128 swizzled bytes (bf16), or 64 plain bytes (e4m3)
  const CUtensorMapSwizzle bsw = a.b_fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
  KParams kp{};
  kp.group_offsets = a.group_offsets;
  kp.G = a.G;
  kp.M = a.M;
  kp.K = a.K;
  kp.N = a.N;
  kp.out = a.out;
  kp.out_lo = a.out_lo;
  kp.b_scale = a.b_scale;
  kp.a_row_scale = a.a_row_scale;
  kp.h_fp32 = a.h_fp32;
  kp.act = a.act;
  kp.err = a.err;
  kp.comb_rows = a.comb_rows;
  kp.comb_w = a.comb_w;
  kp.comb_k = a.comb_k;
  kp.lpt = g_tile_order == 1 && a.group_offsets != nullptr && a.G > 1;
  kp.tile_counter = a.tile_counter;
  kp.b_prefetch = g_b_prefetch;
  kp.sh_rows = a.sh_rows;
  kp.sh_b_scale = a.sh_b_scale;
  kp.bn = nt;
  kp.ksplit = 1;
  kp.kbs = (a.K + BK - 1) / BK;
  if (a.epilogue == kEpiGateUpAct) {
    const uint64_t dims[4] = {N, 2, K, static_cast<uint64_t>(a.G)};
    const uint64_t strides[3] = {N * eb, 2 * N * eb, K * 2 * N * eb};
    const uint32_t box[4] = {64, 1, BK, 1};
    if (!encode_tmap(&tw, a.B, 4, dims, strides, box, bdt, bsw)) return cudaErrorInvalidValue;
    kp.cols_per_tile = 64;
  } else {
    const uint64_t dims[3] = {N, K, static_cast<uint64_t>(a.G)};
    const uint64_t strides[2] = {N * eb, K * N * eb};
    const uint32_t box[3] = {64, BK, 1};
    if (!encode_tmap(&tw, a.B, 3, dims, strides, box, bdt, bsw)) return cudaErrorInvalidValue;
    kp.cols_per_tile = 128;
  }
  kp.n_tiles = (a.N + kp.cols_per_tile - 1) / kp.cols_per_tile;
  const long long max_tiles = cap_grid(
      (static_cast<long long>((a.M + nt - 1) / nt) + a.G) * static_cast<long long>(kp.n_tiles), a, false);
  if (a.epilogue == kEpiGateUpAct)
    return a.b_fp8 ? launch_dec<kEpiGateUpAct, false, true>(tr, tr_lo, tw, kp, max_tiles, s)
                   : launch_dec<kEpiGateUpAct, false, false>(tr, tr_lo, tw, kp, max_tiles, s);
  if (a.epilogue == kEpiCombineF32) {  // bf16 h pairs only
    if (a.b_fp8 || !a.A_lo) return cudaErrorNotSupported;
    return launch_dec<kEpiCombineF32, true, false>(tr, tr_lo, tw, kp, max_tiles, s);
  }
  if (a.b_fp8) return launch_dec<kEpiStoreF32, false, true>(tr, tr_lo, tw, kp, max_tiles, s);
  return a.A_lo ? launch_dec<kEpiStoreF32, true, false>(tr, tr_lo, tw, kp, max_tiles, s)
                : launch_dec<kEpiStoreF32, false, false>(tr, tr_lo, tw, kp, max_tiles, s);
}

// 128-row (or 2-CTA 256-row) tiles for e4m3 rows and K-contiguous e4m3
// weights: kind::f8f6f4; two-term rows put the hi and lo products into one
// accumulator, one-term rows (W8A8) one product.
cudaError_t launch_grouped_gemm_q8(const GroupedGemmArgs& a, cudaStream_t s) {
  if (!a.b_fp8 || a.A_lo || a.ksplit > 1 || a.bias) return cudaErrorInvalidValue;
  if (a.epilogue == kEpiCombineF32 && (!a.comb_rows || !a.comb_w || a.comb_k < 1))
    return cudaErrorInvalidValue;
  if (a.a_gather && (a.a_rows < 1 || a.gather_k < 1)) return cudaErrorInvalidValue;
  if (a.G < 1 || a.G > MAX_G) return cudaErrorInvalidValue;
  const uint64_t K = static_cast<uint64_t>(a.K), N = static_cast<uint64_t>(a.N);
  const uint64_t M = static_cast<uint64_t>(a.M), G = static_cast<uint64_t>(a.G);
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  KParams kp{};
  kp.group_offsets = a.group_offsets;
  kp.G = a.G;
  kp.M = a.M;
  kp.K = a.K;
  kp.N = a.N;
  kp.out = a.out;
  kp.b_scale = a.b_scale;
  kp.a_row_scale = a.a_row_scale;
  kp.a_gather = a.a_gather;
  kp.a_src = a.A;
  kp.gather_k = a.gather_k;
  kp.a_rows = a.a_rows;
  kp.h_fp32 = a.h_fp32;
  kp.act = a.act;
  kp.err = a.err;
  kp.comb_rows = a.comb_rows;
  kp.comb_w = a.comb_w;
  kp.comb_k = a.comb_k;
  kp.lpt = g_tile_order == 1 && a.group_offsets != nullptr && a.G > 1;
  kp.tile_counter = a.tile_counter;
  kp.b_prefetch = g_b_prefetch;
  kp.sh_rows = a.sh_rows;
  kp.sh_b_scale = a.sh_b_scale;
  kp.ksplit = 1;
  kp.kbs = (a.K + 127) / 128;
  if (a.epilogue == kEpiGateUpAct) {
    kp.bn = 256;
    kp.cols_per_tile = 128;
  } else {
    kp.bn = static_cast<int>(std::min<uint64_t>(BN_MAX, (N + 63) / 64 * 64));
    kp.cols_per_tile = kp.bn;
  }
  kp.n_tiles = (a.N + kp.cols_per_tile - 1) / kp.cols_per_tile;
  // Policy as for bf16 (3: 2-CTA tiles with swapped tails from 150 rows per
  // group on average).  Ling-style prefill (~512 rows per group), layer time:
  // 12.0-12.1 ms on 2-CTA tiles with swapped tails, 12.4 ms on 128-row tiles,
  // 12.65 ms on 2-CTA tiles without swapped tails.
  const bool pair_policy =
      g_pair_tiles == 1 || g_pair_tiles == 2 ||
      (g_pair_tiles == 3 && static_cast<long long>(a.M) >= 150ll * a.G);
  const bool pair = a.pair_ok && !a.a_gather && kp.bn == 256 && pair_policy;
  // 2-CTA tiles: a group's last tile with at most 64 (gate/up) or 128 (down)
  // rows runs swapped (weights as the M = 256 operand, hi and lo rows as N)
  kp.swap_tail = (pair && g_pair_tiles != 2) ? (a.epilogue == kEpiGateUpAct ? 64 : 128) : 0;
  CUtensorMap ta, ta_lo, tb, ta_tail, ta_lo_tail, tb_tail;
  const bool one = a.a_e4m3 != 0;  // one-term rows [M, K]; else two-term [M, 2K] (hi | lo)
  {
    const uint64_t dims[2] = {K, M};
    const uint64_t strides[1] = {one ? K : 2 * K};
    const uint32_t box[2] = {128, BM};
    const uint8_t* lo = static_cast<const uint8_t*>(a.A) + K;
    if (a.a_gather) {
      // row gather from the [a_rows, .] rows: one-row boxes, 4 rows per load
      const uint64_t gdims[2] = {K, static_cast<uint64_t>(a.a_rows)};
      const uint32_t gbox[2] = {128, 1};
      if (!encode_tmap(&ta, a.A, 2, gdims, strides, gbox, u8)) return cudaErrorInvalidValue;
      if (one) ta_lo = ta;
      else if (!encode_tmap(&ta_lo, lo, 2, gdims, strides, gbox, u8)) return cudaErrorInvalidValue;
    } else {
      if (!encode_tmap(&ta, a.A, 2, dims, strides, box, u8)) return cudaErrorInvalidValue;
      if (one) ta_lo = ta;
      else if (!encode_tmap(&ta_lo, lo, 2, dims, strides, box, u8)) return cudaErrorInvalidValue;
    }
    const uint32_t tbox[2] = {128, 32};  // swapped tails: 32-row boxes
    if (!encode_tmap(&ta_tail, a.A, 2, dims, strides, tbox, u8)) return cudaErrorInvalidValue;
    if (one) ta_lo_tail = ta_tail;
    else if (!encode_tmap(&ta_lo_tail, lo, 2, dims, strides, tbox, u8)) return cudaErrorInvalidValue;
  }
  // the weight maps of a tensor of ng matrices: the routed experts, or the
  // shared expert's one matrix (the last group when sh_rows > 0)
  auto make_b = [&](const void* Bp, uint64_t ng, CUtensorMap& mb, CUtensorMap& mb_tail) {
    if (a.epilogue == kEpiGateUpAct) {  // [G][2][N][K]: gate rows, then up rows
      const uint64_t dims[4] = {K, N, 2, ng};
      const uint64_t strides[3] = {K, N * K, 2 * N * K};
      const uint32_t box[4] = {128, 128, pair ? 1u : 2u, 1};
      const uint32_t tbox[4] = {128, 64, 2, 1};  // swapped tails: 64 gate + 64 up rows per CTA
      return encode_tmap(&mb, Bp, 4, dims, strides, box, u8) &&
             encode_tmap(&mb_tail, Bp, 4, dims, strides, tbox, u8);
    }
    const uint64_t dims[3] = {K, N, ng};  // [G][N][K]
    const uint64_t strides[2] = {K, N * K};
    const uint32_t box[3] = {128, static_cast<uint32_t>(pair ? kp.bn / 2 : kp.bn), 1};
    if (!encode_tmap(&mb, Bp, 3, dims, strides, box, u8)) return false;
    mb_tail = mb;
    return true;
  };
  CUtensorMap tb2, tb2_tail;
  if (!make_b(a.B, G - (a.sh_rows > 0 ? 1 : 0), tb, tb_tail)) return cudaErrorInvalidValue;
  if (a.sh_rows > 0) {
    if (!make_b(a.sh_B, 1, tb2, tb2_tail)) return cudaErrorInvalidValue;
  } else {
    tb2 = tb;
    tb2_tail = tb_tail;
  }
  const int tile_m = pair ? 2 * BM : BM;
  const long long max_tiles = cap_grid((static_cast<long long>((a.M + tile_m - 1) / tile_m) + a.G) *
                                           static_cast<long long>(kp.n_tiles), a, pair);
  CUtensorMap tout = ta;
  make_out_map(a, kp, /*out_bf16=*/true, tout);
#define MOE_LAUNCH_Q8(E_, S_, P_) \
  launch_epi<E_, S_, false, P_, true>(ta, ta_lo, tb, tb_tail, ta_tail, ta_lo_tail, tb2, tb2_tail, tout, \
                                      kp, max_tiles, s)
  if (one) {
    if (a.epilogue == kEpiGateUpAct)
      return pair ? MOE_LAUNCH_Q8(kEpiGateUpAct, false, true) : MOE_LAUNCH_Q8(kEpiGateUpAct, false, false);
    if (a.epilogue == kEpiStoreF32)
      return pair ? MOE_LAUNCH_Q8(kEpiStoreF32, false, true) : MOE_LAUNCH_Q8(kEpiStoreF32, false, false);
    if (a.epilogue == kEpiCombineF32)
      return pair ? MOE_LAUNCH_Q8(kEpiCombineF32, false, true) : MOE_LAUNCH_Q8(kEpiCombineF32, false, false);
    return cudaErrorInvalidValue;
  }
  if (a.epilogue == kEpiCombineF32)
    return pair ? MOE_LAUNCH_Q8(kEpiCombineF32, true, true) : MOE_LAUNCH_Q8(kEpiCombineF32, true, false);
  if (a.epilogue == kEpiGateUpAct)
    return pair ? MOE_LAUNCH_Q8(kEpiGateUpAct, true, true) : MOE_LAUNCH_Q8(kEpiGateUpAct, true, false);
  if (a.epilogue == kEpiStoreF32)
    return pair ? MOE_LAUNCH_Q8(kEpiStoreF32, true, true) : MOE_LAUNCH_Q8(kEpiStoreF32, true, false);
#undef MOE_LAUNCH_Q8
  return cudaErrorInvalidValue;
}

}  // namespace

int router_k_split(int T, int E, int D) {
  // aim for about 148 work items (one wave on a GB300's 152 SMs; a constant, so
  // that the workspace size depends on the shape alone) without making a
  // split shorter than 4 k-blocks; at most 8 partial planes
  const int tiles = ((T + BM - 1) / BM) * ((E + BN_MAX - 1) / BN_MAX);
  const int KB = (D + BK - 1) / BK;
  int ks = std::max(1, std::min({8, 148 / std::max(1, tiles), KB / 4}));
  const int kbs = (KB + ks - 1) / ks;
  return (KB + kbs - 1) / kbs;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  static int cached[64] = {0};
  if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
  int n = 1;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

cudaError_t launch_grouped_gemm(const GroupedGemmArgs& a, cudaStream_t s) {
  if (a.M <= 0) return cudaSuccess;
  if (a.epilogue == kEpiCombineF32 && (!a.comb_rows || !a.comb_w || a.comb_k < 1 || a.ksplit > 1))
    return cudaErrorInvalidValue;
  // the shared expert as the last group: 128-row / 2-CTA tiles only, its own
  // weight tensor, no row gather or split-K; weights expanded on chip excluded
  if (a.sh_rows > 0 && (!a.sh_B || a.a_gather || a.ksplit > 1 || a.sh_rows > a.M || a.G < 2 ||
                        (a.b_fp8 && !a.a_e4m3x2 && !a.a_e4m3)))
    return cudaErrorInvalidValue;
  // Swap-AB kernel (weights as the 128-row operand) where it measured faster
  // than 128-row tiles on GB300, with 16 rows per tile: a single group of at
  // most 64 rows (the shared expert at decode: more, smaller tiles), at most
  // one row per group on average, and up to 4 rows per group when there are
  // at most 256 groups (Qwen3-MoE decode: 223 -> 213 us); 64 rows per tile for
  // fp8 weights at up to 16 rows per group.  Elsewhere 128-row tiles already
  // stream the weights at close to HBM peak (Qwen3.5-style decode: 92-100 %).
  // fp8 weights (expanded on chip, or read as e4m3 by the 8-bit kind) take
  // 64-row decode tiles up to 16 rows per group: Ling-style decode (16 rows
  // per group) measured 2201 us per layer on them against 2380 us on 128-row
  // tiles and 2606 us on 16-row decode tiles with e4m3 rows.
  const long long Mg = a.M, Gg = a.G;
  if ((a.a_e4m3x2 || a.a_e4m3) && (!a.b_fp8 || a.a_fp16 || (a.a_e4m3x2 && a.a_e4m3)))
    return cudaErrorInvalidValue;
  int nt = 0;
  if (g_decode_kernel == 2) nt = DEC_NT_MAX;
  else if (g_decode_kernel == 3) nt = 16;
  else if (Gg == 1 && Mg <= 64) nt = 16;
  else if (Mg <= Gg) nt = 16;
  else if (!a.b_fp8 && Gg <= 256 && Mg <= 4 * Gg) nt = 16;
  else if (a.b_fp8 && Mg <= 16 * Gg) nt = DEC_NT_MAX;
  if (g_decode_kernel && nt && a.decode_ok && !a.a_gather && a.ksplit <= 1 && a.G <= MAX_G &&
      a.sh_rows == 0 &&
      (a.epilogue == kEpiGateUpAct || a.epilogue == kEpiStoreF32 || a.epilogue == kEpiCombineF32)) {
    if (!a.a_e4m3x2 && !a.a_e4m3 && (a.a_fp16 != 0) != (a.b_fp8 != 0)) return cudaErrorInvalidValue;
    if (a.b_fp8 && a.A_lo) return cudaErrorNotSupported;
    return launch_grouped_gemm_decode(a, nt, s);
  }
  if (a.a_e4m3x2 || a.a_e4m3) return launch_grouped_gemm_q8(a, s);
  if (a.b_fp8 && a.A_lo) return cudaErrorNotSupported;
  // fp16 A rows exactly when the weights are fp8
  if ((a.a_fp16 != 0) != (a.b_fp8 != 0)) return cudaErrorInvalidValue;
  if (a.G < 1 || a.G > MAX_G) return cudaErrorInvalidValue;
  CUtensorMap ta, ta_lo, tb;
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.K) * 2};
    const uint32_t box[2] = {BK, BM};
    const CUtensorMapDataType adt =
        a.a_fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (a.a_gather) {
      // row gather from an [a_rows, K] tensor: one-row boxes, 4 rows per load
      if (a.A_lo || a.a_rows < 1 || a.gather_k < 1) return cudaErrorInvalidValue;
      const uint64_t gdims[2] = {static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.a_rows)};
      const uint32_t gbox[2] = {BK, 1};
      if (!encode_tmap(&ta, a.A, 2, gdims, strides, gbox, adt)) return cudaErrorInvalidValue;
    } else if (!encode_tmap(&ta, a.A, 2, dims, strides, box, adt)) {
      return cudaErrorInvalidValue;
    }
    if (a.A_lo && !encode_tmap(&ta_lo, a.A_lo, 2, dims, strides, box)) return cudaErrorInvalidValue;
    if (!a.A_lo) ta_lo = ta;
  }
  KParams kp;
  kp.group_offsets = a.group_offsets;
  kp.G = a.G;
  kp.M = a.M;
  kp.K = a.K;
  kp.N = a.N;
  kp.out = a.out;
  kp.out_lo = a.out_lo;
  kp.b_scale = a.b_scale;
  kp.bias = a.bias;
  kp.a_row_scale = a.a_row_scale;
  kp.a_gather = a.a_gather;
  kp.a_src = a.A;
  kp.gather_k = a.gather_k;
  kp.a_rows = a.a_rows;
  kp.h_fp32 = a.h_fp32;
  kp.act = a.act;
  kp.err = a.err;
  kp.comb_rows = a.comb_rows;
  kp.comb_w = a.comb_w;
  kp.comb_k = a.comb_k;
  kp.lpt = g_tile_order == 1 && a.group_offsets != nullptr && a.G > 1;
  kp.tile_counter = a.tile_counter;
  kp.b_prefetch = g_b_prefetch;
  kp.sh_rows = a.sh_rows;
  kp.sh_b_scale = a.sh_b_scale;
  {
    const int KB = (a.K + BK - 1) / BK;
    int ks = std::max(1, std::min(a.ksplit, KB));
    if (a.epilogue != kEpiStoreF32) ks = 1;
    kp.kbs = (KB + ks - 1) / ks;
    kp.ksplit = (KB + kp.kbs - 1) / kp.kbs;  // no empty split
    if (kp.ksplit != ks && a.ksplit > 1) return cudaErrorInvalidValue;
  }
  const uint64_t N = static_cast<uint64_t>(a.N), K = static_cast<uint64_t>(a.K);
  const uint64_t eb = a.b_fp8 ? 1 : 2;  // weight element bytes
  const CUtensorMapDataType bdt =
      a.b_fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t box_n = a.b_fp8 ? 128 : 64;  // 128 bytes of columns either way
  if (a.epilogue == kEpiGateUpAct) {
    kp.bn = 256;
    kp.cols_per_tile = 128;
  } else {
    const uint64_t gran = a.b_fp8 ? 128 : 64;
    kp.bn = static_cast<int>(std::min<uint64_t>(BN_MAX, (N + gran - 1) / gran * gran));
    kp.cols_per_tile = kp.bn;
  }
  kp.n_tiles = (a.N + kp.cols_per_tile - 1) / kp.cols_per_tile;
  // 2-CTA tiles need a full 256-column B tile and no split-K.  Policy
  // (moe_set_option(MOE_OPT_PAIR_TILES, .)): 3 (default) = with swapped tails
  // when there are at least 150 rows per group on average (measured faster on
  // the Qwen3.5 and Qwen3 prefill layers and the shared experts, slower at
  // ~128 rows per group, where 256-row tiles are half empty); 1 = always, 2 =
  // always without swapped tails, 0 = never.  Never for fp8 weights: there
  // they measured 40 % slower, and a 2-CTA fp8 run at full Ling size with
  // eight converter warps per CTA ended in a GPU fault whose cause was not found.
  const bool pair_policy =
      g_pair_tiles == 1 || g_pair_tiles == 2 ||
      (g_pair_tiles == 3 && static_cast<long long>(a.M) >= 150ll * a.G);
  const bool pair = a.pair_ok && !a.a_gather && !a.b_fp8 && kp.bn == 256 && kp.ksplit == 1 &&
                    pair_policy;
  // bf16 weights with N a multiple of 64: view each expert's [K, N] (gate/up:
  // [K, 2, N]) matrix as 64-column blocks, [block][K][64], so that one TMA load
  // brings all the blocks of a stage in the layout the MMA reads (box 0 at
  // offset 0, box j at j * 8 KB).  Otherwise one load per 64-column box.
  kp.b_wide = (!a.b_fp8 && N % 64 == 0) ? 1 : 0;
  // 2-CTA tiles: a group's last tile with few rows runs swapped (rows as the
  // MMA N); the gate/up pass then loads one gate and one up block per CTA
  kp.swap_tail = (pair && g_pair_tiles != 2) ? (a.epilogue == kEpiGateUpAct ? 64 : 128) : 0;
  // the weight maps of a tensor of ng matrices: the routed experts, or the
  // shared expert's one matrix (the last group when sh_rows > 0)
  auto make_b = [&](const void* Bp, uint64_t G64, CUtensorMap& mb, CUtensorMap& mb_tail) {
    bool ok;
    if (kp.b_wide && a.epilogue == kEpiGateUpAct) {
      const uint64_t dims[5] = {64, K, N / 64, 2, G64};
      const uint64_t strides[4] = {2 * N * eb, 64 * eb, N * eb, K * 2 * N * eb};
      const uint32_t box[5] = {64, BK, 2, pair ? 1u : 2u, 1};
      ok = encode_tmap(&mb, Bp, 5, dims, strides, box, bdt);
    } else if (kp.b_wide) {
      const uint64_t dims[4] = {64, K, N / 64, G64};
      const uint64_t strides[3] = {N * eb, 64 * eb, K * N * eb};
      const uint32_t nb = static_cast<uint32_t>(kp.bn / 64) / (pair ? 2u : 1u);
      const uint32_t box[4] = {64, BK, nb, 1};
      ok = encode_tmap(&mb, Bp, 4, dims, strides, box, bdt);
    } else if (a.epilogue == kEpiGateUpAct) {
      const uint64_t dims[4] = {N, 2, K, G64};
      const uint64_t strides[3] = {N * eb, 2 * N * eb, K * 2 * N * eb};
      const uint32_t box[4] = {box_n, 1, BK, 1};
      ok = encode_tmap(&mb, Bp, 4, dims, strides, box, bdt);
    } else {
      const uint64_t dims[3] = {N, K, G64};
      const uint64_t strides[2] = {N * eb, K * N * eb};
      const uint32_t box[3] = {box_n, BK, 1};
      ok = encode_tmap(&mb, Bp, 3, dims, strides, box, bdt);
    }
    mb_tail = mb;
    if (ok && kp.swap_tail && kp.b_wide && a.epilogue == kEpiGateUpAct) {
      const uint64_t dims[5] = {64, K, N / 64, 2, G64};
      const uint64_t strides[4] = {2 * N * eb, 64 * eb, N * eb, K * 2 * N * eb};
      const uint32_t box[5] = {64, BK, 1, 2, 1};
      ok = encode_tmap(&mb_tail, Bp, 5, dims, strides, box, bdt);
    }
    return ok;
  };
  CUtensorMap tb_tail, tb2, tb2_tail;
  if (!make_b(a.B, static_cast<uint64_t>(a.G - (a.sh_rows > 0 ? 1 : 0)), tb, tb_tail))
    return cudaErrorInvalidValue;
  if (a.sh_rows > 0) {
    if (!make_b(a.sh_B, 1, tb2, tb2_tail)) return cudaErrorInvalidValue;
  } else {
    tb2 = tb;
    tb2_tail = tb_tail;
  }
  CUtensorMap ta_tail = ta, ta_lo_tail = ta_lo;
  if (kp.swap_tail) {  // swapped tails load their rows in 32-row boxes
    const uint64_t dims[2] = {static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M)};
    const uint64_t strides[1] = {static_cast<uint64_t>(a.K) * 2};
    const uint32_t box[2] = {BK, 32};
    if (!encode_tmap(&ta_tail, a.A, 2, dims, strides, box)) return cudaErrorInvalidValue;
    if (a.A_lo && !encode_tmap(&ta_lo_tail, a.A_lo, 2, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  const int tile_m = pair ? 2 * BM : BM;
  const long long max_tiles = cap_grid((static_cast<long long>((a.M + tile_m - 1) / tile_m) + a.G) *
                                           static_cast<long long>(kp.n_tiles) * kp.ksplit, a, pair);
  CUtensorMap tout = ta;
  make_out_map(a, kp, /*out_bf16=*/a.b_fp8 != 0, tout);
  // (pair is never set for fp8 weights: their kernels exist on 1-CTA tiles only)
#define MOE_LAUNCH(E_, S_, F_)                                                               \
  ((pair && !(F_)) ? launch_epi<E_, S_, F_, !(F_)>(ta, ta_lo, tb, tb_tail, ta_tail, ta_lo_tail, \
                                                  tb2, tb2_tail, tout, kp, max_tiles, s)      \
                   : launch_epi<E_, S_, F_, false>(ta, ta_lo, tb, tb_tail, ta_tail, ta_lo_tail, \
                                                   tb2, tb2_tail, tout, kp, max_tiles, s))
  if (a.epilogue == kEpiGateUpAct) {
    if (a.A_lo) return cudaErrorInvalidValue;
    if (a.a_gather && a.a_gather_cp && !a.b_fp8 && !a.a_fp16 && a.K % 8 == 0)  // cp.async row gather
      return launch_epi<kEpiGateUpAct, false, false, false, false, true>(
          ta, ta_lo, tb, tb_tail, ta_tail, ta_lo_tail, tb2, tb2_tail, tout, kp, max_tiles, s);
    return a.b_fp8 ? MOE_LAUNCH(kEpiGateUpAct, false, true) : MOE_LAUNCH(kEpiGateUpAct, false, false);
  }
  if (a.epilogue == kEpiStoreF32) {
    if (a.b_fp8) return MOE_LAUNCH(kEpiStoreF32, false, true);
    return a.A_lo ? MOE_LAUNCH(kEpiStoreF32, true, false) : MOE_LAUNCH(kEpiStoreF32, false, false);
  }
  if (a.epilogue == kEpiCombineF32) {  // bf16 h pairs only
    if (a.b_fp8 || !a.A_lo) return cudaErrorNotSupported;
    return MOE_LAUNCH(kEpiCombineF32, true, false);
  }
#undef MOE_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace moe
