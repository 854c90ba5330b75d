// Internal interfaces between the C ABI (moe_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "moe.h"

namespace moe {

// Control block at the start of every workspace.
struct ControlBlock {
  int32_t err;       // device error word (MOE_DEV_* flags)
  int32_t reserved[63];
};
static_assert(sizeof(ControlBlock) == 256, "control block is 256 bytes");
// reserved[kTileCounterSlot .. + 3]: the tile counters of the routed gate/up
// and down GEMMs and of the shared expert's two GEMMs (dynamic tile order),
// zeroed by the call that launches them before its first kernel
constexpr int kTileCounterSlot = 7;

// ------------------------------------------------- programmatic dependent launch
// Every kernel of the library starts with pdl_wait() (griddepcontrol.wait:
// returns once the grids this one depends on have completed and their memory
// is visible; a no-op when the launch carries no programmatic dependency)
// before it reads or writes global memory, and then calls
// pdl_launch_dependents(), which lets the next kernel of the stream be
// scheduled while this one runs.  Because every kernel waits unconditionally,
// the completion of kernel n implies that of every earlier kernel, so a
// kernel may read results from any earlier launch.
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

extern int g_pdl;  // moe_set_option(MOE_OPT_PDL, .)

// Launch with the programmatic-stream-serialization attribute when g_pdl is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = g_pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// TMA tensor map (gemm_sm103.cu) of a tensor with `rank` dimensions, innermost
// first: dims, rank - 1 byte strides of the outer dimensions (multiples of 16),
// box sizes; 128-byte swizzle by default.  Returns false when the driver's
// encoder is unavailable or refuses the shape.
bool encode_tmap(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                 CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B);

// Host-side validation shared by every entry point (moe_api.cu): the
// configuration's shape and dtype limits, and whether its (act_dtype,
// w_dtype, act) combination is built.
bool cfg_valid(const moe_config_t* c);
bool combo_supported(const moe_config_t* c);

inline size_t act_bytes(int dt) { return dt == MOE_F32 ? 4 : 2; }
inline size_t w_bytes(int dt) { return dt == MOE_F32 ? 4 : (dt == MOE_BF16 ? 2 : 1); }

// ---------------------------------------------------------------- routing.cu
// Expanded rows per init_routing segment: 512, raised for large R so that
// there are at most 128 segments (each scatter block reads all segments'
// histograms).
inline int route_segment_rows(long long R) {
  long long seg = 512;
  while ((R + seg - 1) / seg > 128) seg *= 2;
  return static_cast<int>(seg);
}
inline int route_segments(long long R) {
  const int seg = route_segment_rows(R);
  return static_cast<int>((R + seg - 1) / seg);
}

// Batches of at most kSmallRouteRows expanded rows use the one-launch
// init_routing + gather kernel (every CTA sorts all rows in shared memory).
constexpr int kSmallRouteRows = 8192;
inline bool small_route(long long R, int E) { return R > 0 && R <= kSmallRouteRows && E <= 512; }
cudaError_t launch_route_permute_small(const int32_t* ids, int R, int E, int k, int T,
                                       int32_t* counts, int32_t* offsets, int32_t* sorted_rows,
                                       int32_t* dest, const void* x, size_t row_bytes,
                                       void* x_perm, const float* tok_scale, float* row_scale,
                                       int32_t* err, cudaStream_t s, int extra_rows = 0);

// Router logits = sum of nsplit fp32 partial planes [nsplit, T, E] (+ bias),
// written to `logits` when nsplit > 1 or bias != nullptr; then top-k softmax.
cudaError_t launch_topk_softmax(const float* partials, int nsplit, const float* bias, float* logits,
                                int T, int E, int k, int renorm, int32_t* ids, float* w,
                                int32_t* err, cudaStream_t s);

// Router projection fused with the top-k softmax (router_sm103.cu), bf16 x
// and W_g: logits (+ bias) written, then ids / w.  router_topk_ok says which
// shapes it takes (64 <= E <= 512, E and D multiples of 8, k <= 32);
// router_topk_split gives its cluster shape: ck slices of D times nh expert
// halves (a function of the shape alone).
bool router_topk_ok(int T, int E, int D, int k);
// Whether the fused kernel is the faster choice for the shape (>= 64 CTAs).
bool router_topk_preferred(int T, int E, int D);
void router_topk_split(int T, int E, int D, int& ck, int& nh);
// Its CTAs, in launch order, and the expanded rows of each one's tokens
// (128 / (ck nh) tokens times k): CTA b's rows are [b chunk_rows, (b + 1)
// chunk_rows).  With chunk_hist (16-byte aligned, nchunks x E int32) the
// kernel also writes each CTA's expert histogram of those rows there.
void router_topk_chunks(int T, int E, int D, int k, int& nchunks, int& chunk_rows);
cudaError_t launch_router_topk(const void* x, const void* Wg, const float* bias, int T, int D,
                               int E, int k, int renorm, float* logits, int32_t* ids, float* w,
                               int32_t* err, cudaStream_t s, int32_t* chunk_hist = nullptr);
// init_routing from those histograms: a CTA per few chunks, no cluster (E <= 512,
// E % 4 == 0, chunk_rows <= 8192).  Same results as the other init_routing
// kernels when the histograms count the ids.
cudaError_t launch_route_sort_chunks(const int32_t* ids, int R, int E, int nchunks, int chunk_rows,
                                     const int32_t* chunk_hist, int32_t* counts, int32_t* offsets,
                                     int32_t* sorted_rows, int32_t* dest, int32_t* err,
                                     cudaStream_t s);

// Split-K factor of the router projection (a pure function of the shape, so
// the workspace size does not depend on the device).
int router_k_split(int T, int E, int D);
// Small batches (decode): the router projection on the CUDA cores, written as
// nsplit fp32 planes [nsplit, T, E] over consecutive slices of D (bf16 x and
// W_g, E even).  router_small_ok says whether a shape takes this path.
bool router_small_ok(int T, int E, int D, int nsplit);
cudaError_t launch_router_small(const void* x, const void* Wg, int T, int D, int E, int nsplit,
                                float* planes, cudaStream_t s);
// `mark`, when not null, is called on the stream right before each of the
// three launches (trace hook of moe_layer).
cudaError_t launch_init_routing(const int32_t* ids, int R, int E, int32_t* counts, int32_t* offsets,
                                int32_t* sorted_rows, int32_t* dest, int32_t* seg_scratch,
                                int32_t* err, cudaStream_t s, void (*mark)(cudaStream_t) = nullptr);
// Expanded rows up to which moe_permute / moe_layer sort with the cluster kernel.
constexpr long long kClusterSortRows = 65536;
// The same stable counting sort as launch_init_routing in one launch: a
// cluster of 8 CTAs that exchange their expert histograms through distributed
// shared memory (no scratch).  E <= 512.
cudaError_t launch_route_sort_cluster(const int32_t* ids, int R, int E, int32_t* counts,
                                      int32_t* offsets, int32_t* sorted_rows, int32_t* dest,
                                      int32_t* err, cudaStream_t s);
// tok_scale / row_scale (optional): row_scale[p] = tok_scale[sorted_rows[p] / k].
// extra_rows = T (all three permutation launchers): x_perm rows R + t are
// also written, copies of token t (the shared expert's rows as the last group
// of the routed GEMMs); x_perm then holds R + T rows.
cudaError_t launch_permute_gather(const void* x, const int32_t* sorted_rows, int R, int k, int T,
                                  size_t row_bytes, void* x_perm, int32_t* err, cudaStream_t s,
                                  const float* tok_scale = nullptr, float* row_scale = nullptr,
                                  int extra_rows = 0);
// The same permutation from the token side (x read once): x_perm[dest[t*k+j]]
// = x[t]; rows at positions >= *nvalid (only after invalid ids) are zeroed.
cudaError_t launch_permute_scatter(const void* x, const int32_t* dest, const int32_t* nvalid,
                                   int R, int k, int T, size_t row_bytes, void* x_perm,
                                   int32_t* err, cudaStream_t s, const float* tok_scale = nullptr,
                                   float* row_scale = nullptr, int extra_rows = 0);
// bf16 (or fp32 when src_f32) rows -> fp16 rows times an exact power of two
// (max |row| < 2^14); inv_scale[r] = the inverse power of two.
cudaError_t launch_rows_to_fp16(const void* x, int rows, int D, void* x16, float* inv_scale,
                                cudaStream_t s, bool src_f32 = false);
// bf16 (or fp32 when src_f32) rows -> two-term e4m3 rows [rows, 2D] (hi
// bytes, then lo bytes) times an exact power of two putting the row's largest
// |element| in [128, 256); inv_scale[r] = the inverse power of two.
cudaError_t launch_rows_to_e4m3x2(const void* x, int rows, int D, void* q, float* inv_scale,
                                  cudaStream_t s, bool src_f32 = false);
// bf16 (or fp32) rows -> one-term e4m3 rows [rows, D] with a dynamic per-row
// scale (W8A8): scale[r] = max|row| / 448, q = e4m3(x / scale[r]).
cudaError_t launch_rows_to_e4m3(const void* x, int rows, int D, void* q, float* scale,
                                cudaStream_t s, bool src_f32 = false);
// W_nk[g][n][c] = W[g][c][n], one-byte elements (K, N multiples of 16).
cudaError_t launch_transpose_bytes(const void* W, long long G, int K, int N, void* W_nk,
                                   cudaStream_t s);
// Fused combine: out[t] = bf16(acc[t] + s[t]) for the [T, D] fp32 sums acc; s
// fp32, bf16 (s_bf16) or null; D a multiple of 4.
cudaError_t launch_combine_round(const float* acc, const void* s_rows, bool s_bf16, int T, int D,
                                 void* out, cudaStream_t s);
// y_perm and s_rows are fp32 (bf16 when y_bf16); out is act_dtype.
cudaError_t launch_finalize(int act_dtype, const void* y_perm, const int32_t* dest, const float* w,
                            const void* s_rows, void* out, int T, int k, int D, int R,
                            int32_t* err, cudaStream_t s, bool y_bf16 = false);

// ---------------------------------------------------------------- simt_fp32.cu
// fp32 path (exact-fp32 configurations): plain CUDA-core kernels.
cudaError_t launch_simt_router(const float* x, const float* Wg, const float* bias, float* logits,
                               int T, int D, int E, cudaStream_t s);
// Gate/up projection + activation over groups (offsets == nullptr: one group of M rows).
cudaError_t launch_simt_gate_up(const float* A, const int32_t* offsets, int G, int M, int K,
                                const float* W13, int I, int act, float* h, int32_t* err,
                                cudaStream_t s);
cudaError_t launch_simt_down(const float* h, const int32_t* offsets, int G, int M, int I,
                             const float* W2, int N, float* y, int32_t* err, cudaStream_t s);

// ---------------------------------------------------------------- gemm_sm103.cu
enum GemmEpilogue : int {
  kEpiGateUpAct = 0,  // W13 pass: acc = [gate | up] -> act(gate) * up as a bf16 (hi, lo) pair
  kEpiStoreF32 = 2,   // down pass / router: acc (* scale) (+ bias) -> fp32
  // down pass with the combine fused in: row r's result (times its scales)
  // times its routing weight comb_w[q] (q = comb_rows[r], the expanded row
  // t * comb_k + j) is added with fp32 atomics into out[t] ([T, N] fp32,
  // zeroed beforehand); no per-row output
  kEpiCombineF32 = 3,
};

struct GroupedGemmArgs {
  int epilogue;                  // GemmEpilogue
  const void* A;                 // [M, K] bf16, K contiguous
  const void* A_lo;              // [M, K] bf16 low part of a split operand, or nullptr
  int M;                         // rows of A (and of the output)
  int K;
  const int32_t* group_offsets;  // [G+1] device, or nullptr for one group of M rows
  int G;
  const void* B;                 // [G, K, 2*N] (gate/up) or [G, K, N]; bf16 or e4m3
  int b_fp8;                     // 1: B is e4m3 (converted to bf16 on chip)
  int N;                         // output columns (I for gate/up)
  const float* b_scale;          // [G, 2N] or [G, N] per-column scales (fp8), or nullptr
  const float* bias;             // [N] fp32 (router), or nullptr
  const float* a_row_scale;      // per-A-row factor on the accumulator ([M], or [a_rows] when
                                 // gathering), or nullptr
  const int32_t* a_gather;       // [M] row gather: output row r reads A row a_gather[r] / gather_k
  int gather_k;
  int a_rows;                    // rows of A when gathering
  int a_gather_cp;               // 1: gather by cp.async warps (bf16 gate/up pass), not TMA gather4
  int a_fp16;                    // 1: A is fp16 (fp8 layers), B e4m3 expanded to fp16
  int a_e4m3x2;                  // 1: A rows are two-term e4m3 [M, 2K] (hi | lo) and B is
                                 //    e4m3 stored [G, N, K] (gate/up: [G, 2N, K]):
                                 //    the 8-bit tensor-core kind, no expansion
  int a_e4m3;                    // 1: A rows are one-term e4m3 [M, K] with a per-row scale
                                 //    in a_row_scale (W8A8), B as for a_e4m3x2
  int h_fp32;                    // gate/up pass: store h as fp32 (no lo plane)
  int ksplit;                    // >1: K split into planes out[s] = partial sums (fp32 store only)
  int pair_ok;                   // 1: 2-CTA (M=256) tiles may be used
  int decode_ok;                 // 1: the swap-AB decode kernel may be used
  void* out;                     // [M, N] fp32 (bf16 when the weights are fp8), or bf16 h_hi
                                 // (gate/up pass)
  void* out_lo;                  // [M, N] bf16 h_lo (gate/up pass)
  int act;                       // moe_act_t (gate/up epilogue)
  int32_t* err;
  // kEpiCombineF32: the expanded row of each output row (sorted_rows), the
  // routing weights [T * comb_k], and k
  const int32_t* comb_rows;
  const float* comb_w;
  int comb_k;
  // > 0: the last group (G - 1) is the shared expert, rows [M - sh_rows, M) of
  // A (and of the output), weights sh_B (one matrix, laid out as B's) with
  // per-column scales sh_b_scale (fp8)
  int sh_rows;
  const void* sh_B;
  const float* sh_b_scale;
  // dynamic tile order (moe_set_option(MOE_OPT_DYNAMIC_TILES, 1)): a counter
  // that is zero when the launch starts; nullptr = static round-robin order
  int32_t* tile_counter;
  // > 0: at most this many CTAs in the persistent grid (0: one per SM)
  int max_ctas;
};

cudaError_t launch_grouped_gemm(const GroupedGemmArgs& a, cudaStream_t s);

// Kernel-variant options (moe_set_option).
extern int g_pair_tiles;
extern int g_decode_kernel;
extern int g_tile_order;
extern int g_b_prefetch;  // moe_set_option(MOE_OPT_B_PREFETCH, .)

// Shared helper: SM count of the current device (cached).
int device_sm_count();

}  // namespace moe
