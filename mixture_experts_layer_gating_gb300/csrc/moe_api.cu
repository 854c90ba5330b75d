// C ABI of the MoE layer (include/moe.h): argument validation, workspace
// layout and the order of kernel launches on the caller's stream.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "moe_internal.h"

using namespace moe;

namespace {

constexpr size_t kAlign = 256;

int g_gather_a = 3;       // moe_set_option(MOE_OPT_GATHER_A, .)
int g_shared_stream = 1;  // moe_set_option(MOE_OPT_SHARED_STREAM, .)
int g_fused_combine = 0;  // moe_set_option(MOE_OPT_FUSED_COMBINE, .)
int g_shared_in_gemm = 0;  // moe_set_option(MOE_OPT_SHARED_IN_GEMM, .)
int g_fused_routing = 1;  // moe_set_option(MOE_OPT_FUSED_ROUTING, .)
int g_dynamic_tiles = 2;  // moe_set_option(MOE_OPT_DYNAMIC_TILES, .)
int g_shared_ctas = 0;    // moe_set_option(MOE_OPT_SHARED_CTAS, .)

// The shared expert depends on x alone, so moe_layer runs it on a second
// stream of the library's own (one per device, created on first use) that
// forks from the caller's stream after x is ready and joins it before the
// finalize kernel: its GEMMs then overlap the routing kernels and the routed
// GEMMs instead of following them.  Fork and join are event record + wait
// pairs, which stream capture turns into graph edges.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxDevices = 64;
SideStream g_side[kMaxDevices];
std::mutex g_side_mu;

// Fork: work enqueued on the returned stream starts after everything already
// on s.  nullptr when the stream cannot be had (the caller then stays serial).
cudaStream_t side_fork(cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream& d = g_side[dev];
  if (!d.stream) {
    if (cudaStreamCreateWithFlags(&d.stream, cudaStreamNonBlocking) != cudaSuccess) {
      d.stream = nullptr;
      return nullptr;
    }
    if (cudaEventCreateWithFlags(&d.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&d.join, cudaEventDisableTiming) != cudaSuccess)
      return nullptr;
  }
  if (cudaEventRecord(d.fork, s) != cudaSuccess) return nullptr;
  if (cudaStreamWaitEvent(d.stream, d.fork, 0) != cudaSuccess) return nullptr;
  return d.stream;
}

// Join: work enqueued on s after this starts after everything on `side`.
bool side_join(cudaStream_t side, cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream& d = g_side[dev];
  if (d.stream != side) return false;
  return cudaEventRecord(d.join, side) == cudaSuccess &&
         cudaStreamWaitEvent(s, d.join, 0) == cudaSuccess;
}

// Optional per-kernel trace events (moe_set_trace_events).
void* const* g_trace_events = nullptr;
int g_trace_n = 0;
int g_trace_next = -1;  // next event index during a traced moe_layer call, -1 = off

inline void trace_mark(cudaStream_t s) {
  if (g_trace_next >= 0 && g_trace_next < g_trace_n)
    cudaEventRecord(static_cast<cudaEvent_t>(g_trace_events[g_trace_next++]), s);
}

inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Layout {
  size_t off[12];
  size_t router_partials;  // split-K planes of the router projection (0 = none)
  // fp8-weight layers: x as fp16 rows with exact power-of-two scales, the
  // inverse scales per token and per permuted row (0 = none)
  size_t x16, tok_inv, row_inv;
  // fp8-weight layers: h (routed, shared) as fp16 rows with inverse scales
  size_t h16, h_inv, hs16, hs_inv;
  size_t seg_scratch;
  // expert histogram of each fused-router CTA's rows (0 = the shape has no
  // fused router)
  size_t chunk_hist;
  size_t total;
};

}  // namespace

namespace moe {

bool cfg_valid(const moe_config_t* c) {
  if (!c) return false;
  if (c->T < 0 || c->D < 8 || c->E < 1 || c->E > 512 || c->k < 1 || c->k > 16 || c->k > c->E ||
      c->I < 8 || c->I_shared < 0)
    return false;
  if (c->D % 8 || c->I % 8 || c->I_shared % 8) return false;
  if (c->act != MOE_ACT_SWIGLU && c->act != MOE_ACT_GEGLU_TANH) return false;
  if (c->act_dtype != MOE_F32 && c->act_dtype != MOE_BF16) return false;
  if (c->w_dtype != MOE_F32 && c->w_dtype != MOE_BF16 && c->w_dtype != MOE_FP8_E4M3 &&
      c->w_dtype != MOE_FP8_E4M3_NK && c->w_dtype != MOE_FP8_E4M3_NK_A8)
    return false;
  if ((c->w_dtype == MOE_FP8_E4M3 || c->w_dtype == MOE_FP8_E4M3_NK ||
       c->w_dtype == MOE_FP8_E4M3_NK_A8) &&
      (c->D % 16 || c->I % 16 || c->I_shared % 16))
    return false;
  const long long R = static_cast<long long>(c->T) * c->k;
  if (R > (1ll << 30)) return false;
  return true;
}

bool combo_supported(const moe_config_t* c) {
  if (c->act_dtype == MOE_F32) return c->w_dtype == MOE_F32;
  return c->w_dtype == MOE_BF16 || c->w_dtype == MOE_FP8_E4M3 || c->w_dtype == MOE_FP8_E4M3_NK ||
         c->w_dtype == MOE_FP8_E4M3_NK_A8;
}

}  // namespace moe

namespace {

// fp8 weights of any layout (per-column scales; A rows in an fp8 layer form
// with per-row scales)
inline bool is_fp8(const moe_config_t* c) {
  return c->w_dtype == MOE_FP8_E4M3 || c->w_dtype == MOE_FP8_E4M3_NK ||
         c->w_dtype == MOE_FP8_E4M3_NK_A8;
}
// fp8 weights stored K-contiguous: the 8-bit kind (two-term e4m3 rows, or
// one-term rows for W8A8)
inline bool is_nk(const moe_config_t* c) {
  return c->w_dtype == MOE_FP8_E4M3_NK || c->w_dtype == MOE_FP8_E4M3_NK_A8;
}
// W8A8: activations quantised per row to one e4m3 term with a dynamic scale
inline bool is_a8(const moe_config_t* c) { return c->w_dtype == MOE_FP8_E4M3_NK_A8; }

// bf16 / fp32 rows -> the A-row form of an fp8 layer: fp16 rows (expanded
// weights) or two-term e4m3 rows (K-contiguous weights), both D * 2 bytes per
// row, with inverse power-of-two scales; or, for W8A8, one-term e4m3 rows of
// D bytes with their dynamic scales.
cudaError_t rows_to_fp8_layer_form(const moe_config_t* c, const void* x, int rows, int D, void* q,
                                   float* inv_scale, cudaStream_t s, bool src_f32 = false) {
  if (is_a8(c)) return launch_rows_to_e4m3(x, rows, D, q, inv_scale, s, src_f32);
  return is_nk(c) ? launch_rows_to_e4m3x2(x, rows, D, q, inv_scale, s, src_f32)
                  : launch_rows_to_fp16(x, rows, D, q, inv_scale, s, src_f32);
}
// The shared expert can run as one more group of the routed GEMMs (it then
// has rows R .. R+T-1 of the permuted rows, h and the expert outputs): its
// intermediate size equals the experts', and the weights are bf16 or
// K-contiguous e4m3 (the 128-row / 2-CTA tile kernels).  The workspace of
// such a layer always has room for those T extra rows.
inline bool shared_group_capable(const moe_config_t* c) {
  return c->I_shared > 0 && c->I_shared == c->I && c->act_dtype == MOE_BF16 &&
         (c->w_dtype == MOE_BF16 || is_nk(c));
}
// Where the routed gate/up pass of moe_layer takes its rows (MOE_OPT_GATHER_A):
// 0 = the gather kernel's permuted copy, 1 = TMA tile::gather4 from x (or its
// row form), 2 = the GEMM's cp.async gather warps from x (bf16 layers).  The
// default (3) takes 2 for bf16 layers whose routed pass has at least 32 rows
// per expert on average (prefill: measured faster than the gather kernel plus
// 2-CTA tiles on the Qwen3-MoE and Gemma-4 prefill layers), else 0 -- and 0
// when the shared expert is asked to run inside the routed GEMMs.
inline int gather_mode(const moe_config_t* c) {
  if (c->act_dtype == MOE_F32) return 0;
  const bool bf16 = c->w_dtype == MOE_BF16;
  switch (g_gather_a) {
    case 0: return 0;
    case 1: return 1;
    case 2: return bf16 ? 2 : 1;
    default:
      if (g_shared_in_gemm && shared_group_capable(c)) return 0;
      return (bf16 && static_cast<long long>(c->T) * c->k >= 32ll * c->E) ? 2 : 0;
  }
}
inline bool shared_in_gemm_on(const moe_config_t* c) {
  return g_shared_in_gemm && shared_group_capable(c) && gather_mode(c) == 0;
}

// Bytes per row of D elements in the form moe_layer permutes: x itself, or
// for fp8 layers their A-row form (2 bytes per element, 1 for W8A8).
inline size_t layer_row_bytes(const moe_config_t* c) {
  return static_cast<size_t>(c->D) * (is_a8(c) ? 1 : act_bytes(c->act_dtype));
}

Layout make_layout(const moe_config_t* c) {
  Layout L{};
  const size_t T = c->T, E = c->E, R = static_cast<size_t>(c->T) * c->k, D = c->D, I = c->I,
               Is = c->I_shared;
  const size_t ab = act_bytes(c->act_dtype);
  // rows of the permuted rows, h and the expert outputs: R, plus T when the
  // shared expert may run as the last group of the routed GEMMs
  const size_t Rx = R + (shared_group_capable(c) ? T : 0);
  size_t cur = sizeof(ControlBlock);
  auto take = [&](size_t bytes) {
    const size_t o = cur;
    cur = align_up(cur + bytes);
    return o;
  };
  L.off[MOE_WS_LOGITS] = take(T * E * 4);
  {
    const int ks = router_k_split(c->T, c->E, c->D);
    L.router_partials = ks > 1 ? take(static_cast<size_t>(ks) * T * E * 4) : 0;
  }
  L.off[MOE_WS_TOPK_IDS] = take(R * 4);
  L.off[MOE_WS_TOPK_W] = take(R * 4);
  L.off[MOE_WS_COUNTS] = take(E * 4);
  L.off[MOE_WS_OFFSETS] = take((E + 1) * 4);
  L.off[MOE_WS_SORTED_ROWS] = take(R * 4);
  L.off[MOE_WS_DEST] = take(R * 4);
  L.seg_scratch = take(E * static_cast<size_t>(route_segments(static_cast<long long>(R))) * 4 + 4);
  if (router_topk_ok(c->T, c->E, c->D, c->k)) {
    int nchunks = 0, chunk_rows = 0;
    router_topk_chunks(c->T, c->E, c->D, c->k, nchunks, chunk_rows);
    L.chunk_hist = take(static_cast<size_t>(nchunks) * E * 4);
  }
  L.off[MOE_WS_X_PERM] = take(Rx * D * ab);
  L.off[MOE_WS_H] = take(Rx * I * 4);        // fp32, bf16 (hi, lo) planes, or bf16
  L.off[MOE_WS_Y_PERM] = take(Rx * D * 4);   // fp32 (bf16 rows for fp8 layers)
  L.off[MOE_WS_H_SHARED] = take(T * Is * 4);
  L.off[MOE_WS_S] = take(T * D * 4);
  if (is_fp8(c)) {
    L.x16 = take(T * D * 2);
    L.tok_inv = take(T * 4);
    L.row_inv = take(Rx * 4);
    L.h16 = take(Rx * I * 2);
    L.h_inv = take(Rx * 4);
    L.hs16 = take(T * Is * 2);
    L.hs_inv = take(T * 4);
  }
  L.total = cur;
  return L;
}

int check_ws(const moe_config_t* c, void* ws, size_t ws_bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign)) return MOE_ERR_WORKSPACE;
  if (ws_bytes < make_layout(c).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

inline int32_t* err_word(void* ws) { return &static_cast<ControlBlock*>(ws)->err; }
// The four tile counters of the control block (dynamic tile order), or null.
inline int32_t* tile_counters(void* ws) {
  return g_dynamic_tiles ? static_cast<ControlBlock*>(ws)->reserved + kTileCounterSlot : nullptr;
}
// Whether a gate/up pass of M rows in G groups takes the dynamic tile order
// (MOE_OPT_DYNAMIC_TILES 2: tiles of at least 64 k-blocks in a prefill-sized
// pass, at least 1024 rows and 32 per group; 1: every pass).
inline bool dynamic_gate_up(const moe_config_t* c, long long M, int G) {
  if (g_dynamic_tiles == 1) return true;
  if (!g_dynamic_tiles) return false;
  const int kblocks = c->D / ((is_nk(c) || is_a8(c)) ? 128 : 64);
  return kblocks >= 64 && M >= 1024 && M >= 32ll * G;
}
// Zeroes the counters on s before a call's first grouped GEMM when one of
// its passes takes the dynamic order (nothing otherwise).
inline cudaError_t zero_tile_counters(void* ws, const moe_config_t* c, cudaStream_t s) {
  int32_t* ctr = tile_counters(ws);
  const long long R = static_cast<long long>(c->T) * c->k;
  const bool any = g_dynamic_tiles == 1 || dynamic_gate_up(c, R, c->E) ||
                   dynamic_gate_up(c, R + c->T, c->E + 1) ||
                   (c->I_shared > 0 && dynamic_gate_up(c, c->T, 1));
  return (ctr && any) ? cudaMemsetAsync(ctr, 0, 4 * sizeof(int32_t), s) : cudaSuccess;
}
inline uint8_t* ws_at(void* ws, size_t off) { return static_cast<uint8_t*>(ws) + off; }

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// moe_layer runs the fused combine: the option is on and the layer's down
// pass has the kernel for it (bf16 weights, or e4m3 weights stored
// K-contiguous; bf16 activations; D a multiple of 4)
inline bool fused_combine_on(const moe_config_t* c) {
  return g_fused_combine && c->act_dtype == MOE_BF16 && (c->w_dtype == MOE_BF16 || is_nk(c)) &&
         c->D % 4 == 0;
}

int common_checks(const moe_config_t* cfg, void* ws, size_t ws_bytes) {
  if (!cfg_valid(cfg)) return MOE_ERR_INVALID_ARG;
  if (!combo_supported(cfg)) return MOE_ERR_UNSUPPORTED;
  return check_ws(cfg, ws, ws_bytes);
}

// The router projection and top-k as one kernel (MOE_OPT_FUSED_ROUTING): bf16
// activations, batches the CUDA-core projection does not take.
// MOE_OPT_FUSED_ROUTING 2 and 3 take it wherever the shape allows (testing).
bool fused_router_on(const moe_config_t* c, int nsplit) {
  return g_fused_routing && c->act_dtype == MOE_BF16 && !router_small_ok(c->T, c->E, c->D, nsplit) &&
         router_topk_ok(c->T, c->E, c->D, c->k) &&
         (g_fused_routing >= 2 || router_topk_preferred(c->T, c->E, c->D));
}

// moe_layer sorts the rows by the fused router's per-CTA histograms (one CTA
// per router CTA, launch_route_sort_chunks) instead of counting them again:
// the router is fused and the batch is above the one-launch size.
// MOE_OPT_FUSED_ROUTING 3 (testing): the fused router wherever the shape
// allows, as 2, with the other init_routing kernels.
bool chunk_sort_on(const moe_config_t* c) {
  return g_fused_routing != 3 && fused_router_on(c, router_k_split(c->T, c->E, c->D)) &&
         !small_route(static_cast<long long>(c->T) * c->k, c->E);
}

// ------------------------------------------------------------------ stages
// `partials`: workspace room for the router's split-K planes (may be null when
// the configuration does not split).
// `chunk_hist`: where the fused router also writes its per-CTA expert
// histograms (moe_layer with chunk_sort_on; null otherwise).
int do_route(const moe_config_t* c, const void* x, const void* Wg, const float* bias,
             float* logits, int32_t* ids, float* w, float* partials, int32_t* err,
             cudaStream_t s, int32_t* chunk_hist = nullptr) {
  cudaError_t e = cudaSuccess;
  const float* src = logits;
  int nsplit = 1;
  if (x) {
    trace_mark(s);
    if (c->act_dtype == MOE_F32) {
      e = launch_simt_router(static_cast<const float*>(x), static_cast<const float*>(Wg), bias,
                             logits, c->T, c->D, c->E, s);
      bias = nullptr;  // added by the projection
    } else {
      nsplit = partials ? router_k_split(c->T, c->E, c->D) : 1;
      float* dst = nsplit > 1 ? partials : logits;
      if (fused_router_on(c, nsplit)) {
        // projection and top-k in one launch
        return cuda_status(launch_router_topk(x, Wg, bias, c->T, c->D, c->E, c->k, c->renormalize,
                                              logits, ids, w, err, s, chunk_hist));
      }
      if (router_small_ok(c->T, c->E, c->D, nsplit)) {
        // a few tokens: a matrix-vector product per token on the CUDA cores,
        // into the same split planes
        e = launch_router_small(x, Wg, c->T, c->D, c->E, nsplit, dst, s);
      } else {
        GroupedGemmArgs a{};
        a.epilogue = kEpiStoreF32;
        a.A = x;
        a.M = c->T;
        a.K = c->D;
        a.group_offsets = nullptr;
        a.G = 1;
        a.B = Wg;
        a.N = c->E;
        a.bias = nullptr;  // added, after the split planes, by the top-k kernel
        a.ksplit = nsplit;
        a.out = dst;
        a.err = err;
        e = launch_grouped_gemm(a, s);
      }
      src = dst;
    }
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  } else {
    bias = nullptr;
  }
  trace_mark(s);
  return cuda_status(launch_topk_softmax(src, nsplit, bias, logits, c->T, c->E, c->k,
                                         c->renormalize, ids, w, err, s));
}

// The permutation of the rows of x after init_routing (batches above the
// one-launch size): x_perm[p] = x[sorted_rows[p] / k].
int do_permute_rows(const moe_config_t* c, const void* x, const int32_t* sorted_rows,
                    const int32_t* dest, const int32_t* offsets, void* x_perm, int32_t* err,
                    cudaStream_t s, size_t row_bytes, const float* tok_scale, float* row_scale,
                    int extra_rows) {
  const int R = c->T * c->k;
  trace_mark(s);
  // x well inside L2: gather rows in permuted order (each token row re-read
  // from L2 k times, the writes sequential); larger x: read each token row
  // once and write its k copies (Qwen3.5-style prefill, 67 MB of x: 162 ->
  // 117 us; Ling-style, 268 MB: 600 -> 388 us; Qwen3-style, 17 MB: 27.5 vs
  // 28.8 us in favour of the gather)
  cudaError_t e;
  if (static_cast<size_t>(c->T) * row_bytes > (size_t{32} << 20))
    e = launch_permute_scatter(x, dest, offsets + c->E, R, c->k, c->T, row_bytes, x_perm, err, s,
                               tok_scale, row_scale, extra_rows);
  else
    e = launch_permute_gather(x, sorted_rows, R, c->k, c->T, row_bytes, x_perm, err, s, tok_scale,
                              row_scale, extra_rows);
  return cuda_status(e);
}

// row_bytes: bytes of one row of x (act_dtype rows, or moe_layer's fp8 row form)
// extra_rows = T: x_perm rows R .. R+T-1 become copies of the tokens (the
// shared expert's rows as the last group of the routed GEMMs).
// chunk_hist: the fused router's per-CTA histograms of these ids (moe_layer
// with chunk_sort_on), or null.
int do_permute(const moe_config_t* c, const int32_t* ids, const void* x, int32_t* counts,
               int32_t* offsets, int32_t* sorted_rows, int32_t* dest, void* x_perm,
               int32_t* seg_scratch, int32_t* err, cudaStream_t s, size_t row_bytes,
               const float* tok_scale = nullptr, float* row_scale = nullptr, int extra_rows = 0,
               const int32_t* chunk_hist = nullptr) {
  const int R = c->T * c->k;
  if (small_route(R, c->E)) {  // one launch: sort + gather
    trace_mark(s);
    const bool gather = x && x_perm;
    return cuda_status(launch_route_permute_small(
        ids, R, c->E, c->k, c->T, counts, offsets, sorted_rows, dest, gather ? x : nullptr,
        row_bytes, gather ? x_perm : nullptr, tok_scale,
        row_scale, err, s, extra_rows));
  }
  cudaError_t e;
  // after the fused router: one CTA per router CTA, from its histograms;
  // otherwise histogram, scan and scatter as one 8-CTA cluster launch up to
  // 65536 expanded rows, and above, the two-kernel sort that spreads the
  // scattered writes over one CTA per segment (Ling-style prefill, 131072
  // rows: 38 us in the cluster against 25 us in two kernels)
  if (chunk_hist) {
    int nchunks = 0, chunk_rows = 0;
    router_topk_chunks(c->T, c->E, c->D, c->k, nchunks, chunk_rows);
    trace_mark(s);
    e = launch_route_sort_chunks(ids, R, c->E, nchunks, chunk_rows, chunk_hist, counts, offsets,
                                 sorted_rows, dest, err, s);
  } else if (g_fused_routing && R > 0 && R <= kClusterSortRows && c->E <= 512) {
    trace_mark(s);
    e = launch_route_sort_cluster(ids, R, c->E, counts, offsets, sorted_rows, dest, err, s);
  } else {
    e = launch_init_routing(ids, R, c->E, counts, offsets, sorted_rows, dest, seg_scratch, err, s,
                            g_trace_next >= 0 ? trace_mark : nullptr);
  }
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (x && x_perm)
    return do_permute_rows(c, x, sorted_rows, dest, offsets, x_perm, err, s, row_bytes, tok_scale,
                           row_scale, extra_rows);
  return MOE_OK;
}

// One gated FFN (gate/up + act, then down) over grouped rows.  For fp8
// weights A holds fp16 (or two-term e4m3) rows and a_row_scale their inverse
// power-of-two scales; h is written in fp32 (bf16 for K-contiguous weights)
// and converted to the same row form (h16, h_inv) for the down pass.
// When a_gather is given, the gate/up pass reads A row a_gather[r] / k of an
// [a_rows, D] A for output row r (a_row_scale then indexed by that A row).
// comb_rows / comb_w (fused combine, routed pass only): y is then the [T, D]
// fp32 accumulator the down pass adds each row times its routing weight into.
int do_ffn(const moe_config_t* c, const void* A, const float* a_row_scale, int M,
           const int32_t* offsets, int G, const void* W13, const float* s13, const void* W2,
           const float* s2, int I, void* h, void* y, void* h16, float* h_inv, int32_t* err,
           cudaStream_t s, const int32_t* a_gather = nullptr, int a_rows = 0,
           const int32_t* comb_rows = nullptr, const float* comb_w = nullptr, int sh_rows = 0,
           const void* W13s = nullptr, const float* s13s = nullptr, const void* W2s = nullptr,
           const float* s2s = nullptr, int32_t* counters = nullptr, int max_ctas = 0) {
  if (M <= 0) return MOE_OK;
  cudaError_t e;
  trace_mark(s);
  if (c->act_dtype == MOE_F32) {
    e = launch_simt_gate_up(static_cast<const float*>(A), offsets, G, M, c->D,
                            static_cast<const float*>(W13), I, c->act, static_cast<float*>(h), err,
                            s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    trace_mark(s);
    e = launch_simt_down(static_cast<const float*>(h), offsets, G, M, I,
                         static_cast<const float*>(W2), c->D, static_cast<float*>(y), err, s);
    return cuda_status(e);
  }
  // bf16 weights: h is two bf16 planes [M, I], h_hi then h_lo (h ~= h_hi + h_lo),
  // and the down pass multiplies both.  fp8 weights: h in fp32, then fp16 rows;
  // K-contiguous fp8 weights: h in bf16, then two-term e4m3 rows (exact for a
  // bf16 row but for its elements below 2^-9 of the row's largest).
  const bool fp8 = is_fp8(c);
  const bool nk = is_nk(c);
  void* h_lo = fp8 ? nullptr : static_cast<uint8_t*>(h) + static_cast<size_t>(M) * I * 2;
  GroupedGemmArgs a{};
  a.epilogue = kEpiGateUpAct;
  a.A = A;
  a.M = M;
  a.K = c->D;
  a.group_offsets = offsets;
  a.G = G;
  a.B = W13;
  a.b_fp8 = fp8;
  a.a_fp16 = fp8 && !nk;
  a.a_e4m3x2 = nk && !is_a8(c);
  a.a_e4m3 = is_a8(c);
  a.a_row_scale = a_row_scale;
  a.a_gather = a_gather;
  a.gather_k = c->k;
  a.a_rows = a_rows;
  a.a_gather_cp = gather_mode(c) == 2;
  a.N = I;
  a.b_scale = s13;
  a.out = h;
  a.out_lo = h_lo;
  a.h_fp32 = fp8 && !nk;
  a.act = c->act;
  a.pair_ok = 1;
  a.decode_ok = 1;
  a.err = err;
  a.sh_rows = sh_rows;  // > 0: the last group is the shared expert (its own weights)
  a.sh_B = W13s;
  a.sh_b_scale = s13s;
  // counters[0]: gate/up pass, counters[1]: down pass (MOE_OPT_DYNAMIC_TILES:
  // 1 = both; 2, the default = a prefill-sized gate/up pass whose tiles are at
  // least 64 k-blocks long -- there the balance pays for the queue, which
  // costs the short tiles of the down passes and decode-sized passes more
  // than it saves)
  a.tile_counter = (counters && dynamic_gate_up(c, M, G)) ? counters : nullptr;
  a.max_ctas = max_ctas;  // (b copies it)
  e = launch_grouped_gemm(a, s);
  if (e != cudaSuccess) return e == cudaErrorNotSupported ? MOE_ERR_UNSUPPORTED : MOE_ERR_CUDA;
  if (fp8) {
    trace_mark(s);
    if (rows_to_fp8_layer_form(c, h, M, I, h16, h_inv, s, /*src_f32=*/!nk) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  GroupedGemmArgs b = a;
  b.epilogue = kEpiStoreF32;
  b.A = fp8 ? h16 : h;
  b.A_lo = h_lo;
  b.K = I;
  b.B = W2;
  b.N = c->D;
  b.b_scale = s2;
  b.a_fp16 = fp8 && !nk;
  b.a_row_scale = fp8 ? h_inv : nullptr;
  b.a_gather = nullptr;
  b.h_fp32 = 0;
  b.out = y;  // fp8-weight layers: the store pass writes bf16 rows
  b.out_lo = nullptr;
  b.sh_B = W2s;
  b.sh_b_scale = s2s;
  b.tile_counter = (counters && g_dynamic_tiles == 1) ? counters + 1 : nullptr;
  if (comb_rows) {
    b.epilogue = kEpiCombineF32;
    b.comb_rows = comb_rows;
    b.comb_w = comb_w;
    b.comb_k = c->k;
  }
  trace_mark(s);
  e = launch_grouped_gemm(b, s);
  if (e != cudaSuccess) return e == cudaErrorNotSupported ? MOE_ERR_UNSUPPORTED : MOE_ERR_CUDA;
  return MOE_OK;
}

// x_perm / x: the routed and shared A rows (fp16 with inverse row scales
// xp_scale / x_scale for fp8 weights, else act_dtype and null scales).
// gather: when not null, x_perm is x itself ([T, D]) and the routed gate/up
// pass gathers row gather[p] / k for permuted row p (xp_scale indexed by token).
int do_grouped_ffn(const moe_config_t* c, const void* x_perm, const float* xp_scale,
                   const int32_t* offsets, const void* W13, const float* s13, const void* W2,
                   const float* s2, void* h, void* y_perm, const void* x, const float* x_scale,
                   const void* W13s, const float* s13s, const void* W2s, const float* s2s,
                   void* h_s, void* s_out, void* ws, int32_t* err, cudaStream_t s,
                   const int32_t* gather = nullptr, const int32_t* comb_rows = nullptr,
                   const float* comb_w = nullptr, bool shared_in_gemm = false) {
  const int R = c->T * c->k;
  const Layout L = make_layout(c);
  const bool fp8 = is_fp8(c);
  if (shared_in_gemm) {
    // the shared expert as group E of the routed GEMMs: rows R .. R+T-1 of
    // x_perm (written by the permutation), h and y_perm
    return do_ffn(c, x_perm, xp_scale, R + c->T, offsets, c->E + 1, W13, s13, W2, s2, c->I, h, y_perm,
                  fp8 ? ws_at(ws, L.h16) : nullptr,
                  fp8 ? reinterpret_cast<float*>(ws_at(ws, L.h_inv)) : nullptr, err, s, nullptr, 0,
                  comb_rows, comb_w, c->T, W13s, s13s, W2s, s2s, tile_counters(ws));
  }
  int32_t* ctr = tile_counters(ws);
  int st = do_ffn(c, x_perm, xp_scale, R, offsets, c->E, W13, s13, W2, s2, c->I, h, y_perm,
                  fp8 ? ws_at(ws, L.h16) : nullptr,
                  fp8 ? reinterpret_cast<float*>(ws_at(ws, L.h_inv)) : nullptr, err, s, gather,
                  gather ? c->T : 0, comb_rows, comb_w, 0, nullptr, nullptr, nullptr, nullptr, ctr);
  if (st != MOE_OK) return st;
  if (x && c->I_shared > 0)
    st = do_ffn(c, x, x_scale, c->T, nullptr, 1, W13s, s13s, W2s, s2s, c->I_shared, h_s, s_out,
                fp8 ? ws_at(ws, L.hs16) : nullptr,
                fp8 ? reinterpret_cast<float*>(ws_at(ws, L.hs_inv)) : nullptr, err, s, nullptr, 0,
                nullptr, nullptr, 0, nullptr, nullptr, nullptr, nullptr, ctr ? ctr + 2 : nullptr);
  return st;
}

bool fp8_scales_ok(const moe_config_t* c, const float* s13, const float* s2) {
  const bool fp8 = is_fp8(c);
  return fp8 ? (s13 && s2) : (!s13 && !s2);
}

}  // namespace

extern "C" {

size_t moe_workspace_size(const moe_config_t* cfg) {
  if (!cfg_valid(cfg)) return 0;
  return make_layout(cfg).total;
}

size_t moe_workspace_offset(const moe_config_t* cfg, int which) {
  if (!cfg_valid(cfg) || which < 0 || which > MOE_WS_ROW_INV) return static_cast<size_t>(-1);
  const Layout L = make_layout(cfg);
  if (which <= MOE_WS_S) return L.off[which];
  if (!is_fp8(cfg)) return static_cast<size_t>(-1);
  return which == MOE_WS_X16 ? L.x16 : which == MOE_WS_TOK_INV ? L.tok_inv : L.row_inv;
}

int moe_route(const moe_config_t* cfg, const void* x, const void* Wg, const float* logit_bias,
              float* logits, int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes,
              void* stream) {
  int st = common_checks(cfg, ws, ws_bytes);
  if (st != MOE_OK) return st;
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (x && (!Wg || !aligned16(x) || !aligned16(Wg))) return MOE_ERR_INVALID_ARG;
  if (!x && logit_bias) return MOE_ERR_INVALID_ARG;
  if (cfg->act_dtype == MOE_BF16 && x && (cfg->E % 8)) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  const Layout L = make_layout(cfg);
  float* partials = L.router_partials ? reinterpret_cast<float*>(ws_at(ws, L.router_partials)) : nullptr;
  return do_route(cfg, x, Wg, logit_bias, logits, topk_ids, topk_w, partials, err_word(ws),
                  static_cast<cudaStream_t>(stream));
}

int moe_permute(const moe_config_t* cfg, const int32_t* topk_ids, const void* x, int32_t* counts,
                int32_t* offsets, int32_t* sorted_rows, int32_t* dest, void* x_perm, void* ws,
                size_t ws_bytes, void* stream) {
  int st = common_checks(cfg, ws, ws_bytes);
  if (st != MOE_OK) return st;
  if (!topk_ids || !counts || !offsets || !sorted_rows || !dest) return MOE_ERR_INVALID_ARG;
  if (x && (!x_perm || !aligned16(x) || !aligned16(x_perm))) return MOE_ERR_INVALID_ARG;
  const Layout L = make_layout(cfg);
  return do_permute(cfg, topk_ids, x, counts, offsets, sorted_rows, dest, x_perm,
                    reinterpret_cast<int32_t*>(ws_at(ws, L.seg_scratch)), err_word(ws),
                    static_cast<cudaStream_t>(stream),
                    static_cast<size_t>(cfg->D) * act_bytes(cfg->act_dtype));
}

int moe_grouped_ffn(const moe_config_t* cfg, const void* x_perm, const int32_t* offsets,
                    const void* W13, const float* s13, const void* W2, const float* s2, void* h,
                    void* y_perm, const void* x, const void* W13s, const float* s13s,
                    const void* W2s, const float* s2s, void* h_s, void* s_out, void* ws,
                    size_t ws_bytes, void* stream) {
  int st = common_checks(cfg, ws, ws_bytes);
  if (st != MOE_OK) return st;
  if (!x_perm || !offsets || !W13 || !W2 || !h || !y_perm) return MOE_ERR_INVALID_ARG;
  for (const void* p : {x_perm, W13, W2, static_cast<const void*>(h), static_cast<const void*>(y_perm)})
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (!fp8_scales_ok(cfg, s13, s2)) return MOE_ERR_INVALID_ARG;
  const bool shared = x && cfg->I_shared > 0;
  if (shared) {
    if (!W13s || !W2s || !h_s || !s_out) return MOE_ERR_INVALID_ARG;
    for (const void* p : {x, W13s, W2s, static_cast<const void*>(h_s), static_cast<const void*>(s_out)})
      if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (!fp8_scales_ok(cfg, s13s, s2s)) return MOE_ERR_INVALID_ARG;
  }
  if (cfg->T == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (zero_tile_counters(ws, cfg, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (is_fp8(cfg)) {
    // fp8 weights: convert the bf16 rows to fp16 rows (or two-term e4m3 rows)
    // with exact power-of-two scales in the workspace first
    const Layout L = make_layout(cfg);
    const int R = cfg->T * cfg->k;
    void* xp16 = ws_at(ws, L.off[MOE_WS_X_PERM]);
    float* row_inv = reinterpret_cast<float*>(ws_at(ws, L.row_inv));
    if (rows_to_fp8_layer_form(cfg, x_perm, R, cfg->D, xp16, row_inv, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    void* x16 = nullptr;
    float* tok_inv = nullptr;
    if (shared) {
      x16 = ws_at(ws, L.x16);
      tok_inv = reinterpret_cast<float*>(ws_at(ws, L.tok_inv));
      if (rows_to_fp8_layer_form(cfg, x, cfg->T, cfg->D, x16, tok_inv, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    }
    return do_grouped_ffn(cfg, xp16, row_inv, offsets, W13, s13, W2, s2, h, y_perm, x16, tok_inv,
                          W13s, s13s, W2s, s2s, h_s, s_out, ws, err_word(ws), s);
  }
  return do_grouped_ffn(cfg, x_perm, nullptr, offsets, W13, s13, W2, s2, h, y_perm, x, nullptr,
                        W13s, s13s, W2s, s2s, h_s, s_out, ws, err_word(ws), s);
}

int moe_finalize(const moe_config_t* cfg, const void* y_perm, const int32_t* dest,
                 const float* topk_w, const void* s, void* out, void* ws, size_t ws_bytes,
                 void* stream) {
  int st = common_checks(cfg, ws, ws_bytes);
  if (st != MOE_OK) return st;
  if (!y_perm || !dest || !topk_w || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(out) || (s && !aligned16(s))) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  return cuda_status(launch_finalize(cfg->act_dtype, y_perm, dest, topk_w, s, out, cfg->T, cfg->k,
                                     cfg->D, cfg->T * cfg->k, err_word(ws),
                                     static_cast<cudaStream_t>(stream), is_fp8(cfg)));
}

int moe_layer(const moe_config_t* cfg, const void* x, const void* Wg, const float* logit_bias,
              const void* W13, const float* s13, const void* W2, const float* s2,
              const void* W13s, const float* s13s, const void* W2s, const float* s2s, void* out,
              void* ws, size_t ws_bytes, void* stream) {
  int st = common_checks(cfg, ws, ws_bytes);
  if (st != MOE_OK) return st;
  if (!x || !Wg || !W13 || !W2 || !out) return MOE_ERR_INVALID_ARG;
  for (const void* p : {x, Wg, W13, W2, static_cast<const void*>(out)})
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (!fp8_scales_ok(cfg, s13, s2)) return MOE_ERR_INVALID_ARG;
  const bool shared = cfg->I_shared > 0;
  if (shared) {
    if (!W13s || !W2s || !aligned16(W13s) || !aligned16(W2s)) return MOE_ERR_INVALID_ARG;
    if (!fp8_scales_ok(cfg, s13s, s2s)) return MOE_ERR_INVALID_ARG;
  }
  if (cfg->act_dtype == MOE_BF16 && (cfg->E % 8)) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout L = make_layout(cfg);
  int32_t* err = err_word(ws);
  float* logits = reinterpret_cast<float*>(ws_at(ws, L.off[MOE_WS_LOGITS]));
  int32_t* ids = reinterpret_cast<int32_t*>(ws_at(ws, L.off[MOE_WS_TOPK_IDS]));
  float* w = reinterpret_cast<float*>(ws_at(ws, L.off[MOE_WS_TOPK_W]));
  int32_t* counts = reinterpret_cast<int32_t*>(ws_at(ws, L.off[MOE_WS_COUNTS]));
  int32_t* offsets = reinterpret_cast<int32_t*>(ws_at(ws, L.off[MOE_WS_OFFSETS]));
  int32_t* sorted_rows = reinterpret_cast<int32_t*>(ws_at(ws, L.off[MOE_WS_SORTED_ROWS]));
  int32_t* dest = reinterpret_cast<int32_t*>(ws_at(ws, L.off[MOE_WS_DEST]));
  int32_t* seg = reinterpret_cast<int32_t*>(ws_at(ws, L.seg_scratch));
  void* x_perm = ws_at(ws, L.off[MOE_WS_X_PERM]);
  void* h = ws_at(ws, L.off[MOE_WS_H]);
  void* y_perm = ws_at(ws, L.off[MOE_WS_Y_PERM]);
  void* h_s = ws_at(ws, L.off[MOE_WS_H_SHARED]);
  void* s_out = ws_at(ws, L.off[MOE_WS_S]);

  const bool traced = g_trace_events && g_trace_n >= moe_layer_launch_count(cfg) + 1;
  g_trace_next = traced ? 0 : -1;
  const bool fp8 = is_fp8(cfg);
  // Fused combine (MOE_OPT_FUSED_COMBINE): the routed down pass adds each row
  // times its routing weight into [T, D] fp32 sums (the y_perm region), zeroed
  // here first, and the last kernel rounds sums + shared row; no y_perm rows.
  const bool fused = fused_combine_on(cfg);
  if (fused && cudaMemsetAsync(y_perm, 0, static_cast<size_t>(cfg->T) * cfg->D * 4, s) != cudaSuccess)
    return (g_trace_next = -1, MOE_ERR_CUDA);
  if (zero_tile_counters(ws, cfg, s) != cudaSuccess) return (g_trace_next = -1, MOE_ERR_CUDA);
  const void* x_rows = x;  // what the gather and the shared expert read
  float* tok_inv = nullptr;
  float* row_inv = nullptr;
  if (fp8) {
    // fp8 weights: x once to fp16 rows (or two-term e4m3 rows) with exact
    // power-of-two scales; the gather carries the inverse scale per row
    void* x16 = ws_at(ws, L.x16);
    tok_inv = reinterpret_cast<float*>(ws_at(ws, L.tok_inv));
    row_inv = reinterpret_cast<float*>(ws_at(ws, L.row_inv));
    trace_mark(s);
    if (rows_to_fp8_layer_form(cfg, x, cfg->T, cfg->D, x16, tok_inv, s) != cudaSuccess)
      return (g_trace_next = -1, MOE_ERR_CUDA);
    x_rows = x16;
  }
  // The shared expert as the last group of the routed GEMMs
  // (MOE_OPT_SHARED_IN_GEMM), or on the side stream (not while tracing: the
  // trace events time kernels one after another on the caller's stream).
  const bool in_gemm = shared && shared_in_gemm_on(cfg);
  cudaStream_t side = nullptr;
  // MOE_OPT_SHARED_STREAM 1: the side stream forks here, once x is ready;
  // 2: after init_routing, so that the shared expert's GEMMs (which hold most
  // of every SM's shared memory) start once the routing kernels (which need
  // some too) are done, and run beside the permutation kernel (which needs none)
  const bool want_side = shared && g_shared_stream && !traced && !in_gemm;
  auto fork_shared = [&]() -> int {
    side = side_fork(s);
    if (!side) return MOE_OK;  // no side stream: the shared expert runs on s below
    int32_t* ctr = tile_counters(ws);
    const int r = do_ffn(cfg, x_rows, tok_inv, cfg->T, nullptr, 1, W13s, s13s, W2s, s2s,
                         cfg->I_shared, h_s, s_out, fp8 ? ws_at(ws, L.hs16) : nullptr,
                         fp8 ? reinterpret_cast<float*>(ws_at(ws, L.hs_inv)) : nullptr, err, side,
                         nullptr, 0, nullptr, nullptr, 0, nullptr, nullptr, nullptr, nullptr,
                         ctr ? ctr + 2 : nullptr, g_shared_ctas);
    if (r != MOE_OK) {
      side_join(side, s);
      side = nullptr;
    }
    return r;
  };
  if (want_side && g_shared_stream == 1) {
    st = fork_shared();
    if (st != MOE_OK) return (g_trace_next = -1, st);
  }
  // after the fork every early return first joins the side stream back
  auto fail = [&](int code) {
    if (side) side_join(side, s);
    g_trace_next = -1;
    return code;
  };
  float* partials = L.router_partials ? reinterpret_cast<float*>(ws_at(ws, L.router_partials)) : nullptr;
  int32_t* chunk_hist =
      chunk_sort_on(cfg) ? reinterpret_cast<int32_t*>(ws_at(ws, L.chunk_hist)) : nullptr;
  st = do_route(cfg, x, Wg, logit_bias, logits, ids, w, partials, err, s, chunk_hist);
  if (st != MOE_OK) return fail(st);
  // The routed gate/up pass reads its rows from a permuted copy of x (the
  // gather kernel streams at HBM speed), or gathers them from x itself
  // (gather_mode): bf16 prefill layers by default with the GEMM's cp.async
  // gather warps (x stays in L2; no permuted copy is written or read), on
  // request with TMA tile::gather4 loads (slower on GB300: 32 four-row
  // requests per 16 KB A tile).
  const bool gather = gather_mode(cfg) != 0;
  const bool late_fork = want_side && g_shared_stream == 2;
  if (late_fork && !gather && !small_route(static_cast<long long>(cfg->T) * cfg->k, cfg->E)) {
    // init_routing, the fork, then the permutation beside the shared GEMMs
    st = do_permute(cfg, ids, nullptr, counts, offsets, sorted_rows, dest, nullptr, seg, err, s,
                    layer_row_bytes(cfg), nullptr, nullptr, 0, chunk_hist);
    if (st != MOE_OK) return fail(st);
    st = fork_shared();
    if (st != MOE_OK) return fail(st);
    st = do_permute_rows(cfg, x_rows, sorted_rows, dest, offsets, x_perm, err, s, layer_row_bytes(cfg),
                         tok_inv, row_inv, 0);
  } else {
    st = do_permute(cfg, ids, gather ? nullptr : x_rows, counts, offsets, sorted_rows, dest,
                    gather ? nullptr : x_perm, seg, err, s, layer_row_bytes(cfg), tok_inv, row_inv,
                    in_gemm ? cfg->T : 0, chunk_hist);
    if (st == MOE_OK && late_fork) st = fork_shared();
  }
  if (st != MOE_OK) return fail(st);
  st = do_grouped_ffn(cfg, gather ? x_rows : x_perm, gather ? tok_inv : row_inv, offsets, W13, s13,
                      W2, s2, h, y_perm, (shared && !side) ? x_rows : nullptr, tok_inv, W13s, s13s,
                      W2s, s2s, h_s, s_out, ws, err, s, gather ? sorted_rows : nullptr,
                      fused ? sorted_rows : nullptr, fused ? w : nullptr, in_gemm);
  if (st != MOE_OK) return fail(st);
  if (side && !side_join(side, s)) return (g_trace_next = -1, MOE_ERR_CUDA);
  trace_mark(s);
  // the shared expert's output rows: s_out, or rows R .. R+T-1 of y_perm when it
  // ran inside the routed GEMMs (the fused combine has added those already)
  const void* s_rows =
      !shared ? nullptr
              : in_gemm ? static_cast<const void*>(static_cast<const uint8_t*>(y_perm) +
                                                   static_cast<size_t>(cfg->T) * cfg->k * cfg->D *
                                                       (fp8 ? 2 : 4))
                        : s_out;
  if (fused)
    st = cuda_status(launch_combine_round(static_cast<const float*>(y_perm), in_gemm ? nullptr : s_rows,
                                          fp8, cfg->T, cfg->D, out, s));
  else
    st = cuda_status(launch_finalize(cfg->act_dtype, y_perm, dest, w, s_rows, out, cfg->T, cfg->k,
                                     cfg->D, cfg->T * cfg->k, err, s, fp8));
  trace_mark(s);
  g_trace_next = -1;
  return st;
}

int moe_pack_weights_nk(const void* W, int64_t G, int32_t K, int32_t N, void* W_nk, void* stream) {
  if (!W || !W_nk || !aligned16(W) || !aligned16(W_nk)) return MOE_ERR_INVALID_ARG;
  if (G < 1 || G > (1ll << 16) - 1 || K < 16 || N < 16 || K % 16 || N % 16) return MOE_ERR_INVALID_ARG;
  const uintptr_t a = reinterpret_cast<uintptr_t>(W), b = reinterpret_cast<uintptr_t>(W_nk);
  const uintptr_t bytes = static_cast<uintptr_t>(G) * static_cast<uintptr_t>(K) * static_cast<uintptr_t>(N);
  if (a < b + bytes && b < a + bytes) return MOE_ERR_INVALID_ARG;  // overlap
  return cuda_status(launch_transpose_bytes(W, G, K, N, W_nk, static_cast<cudaStream_t>(stream)));
}

int moe_read_device_status(void* ws, void* stream, int32_t* flags) {
  if (!ws) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, err_word(ws), sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(err_word(ws), 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (flags) *flags = v;
  return v ? MOE_ERR_DEVICE_CHECK : MOE_OK;
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null pointer, shape, alignment or range)";
    case MOE_ERR_UNSUPPORTED: return "unsupported dtype / activation combination";
    case MOE_ERR_CUDA: return "CUDA runtime or driver error";
    case MOE_ERR_DEVICE_CHECK: return "device data check failed (see the device error flags)";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

int moe_set_option(int option, int value) {
  switch (option) {
    case MOE_OPT_PAIR_TILES: {
      const int old = g_pair_tiles;
      g_pair_tiles = value < 0 ? 0 : (value > 3 ? 3 : value);
      return old;
    }
    case MOE_OPT_DECODE_KERNEL: {
      const int old = g_decode_kernel;
      g_decode_kernel = value < 0 ? 0 : (value > 3 ? 3 : value);
      return old;
    }
    case MOE_OPT_GATHER_A: {
      const int old = g_gather_a;
      g_gather_a = value <= 0 ? 0 : value >= 3 ? 3 : value;
      return old;
    }
    case MOE_OPT_SHARED_STREAM: {
      const int old = g_shared_stream;
      g_shared_stream = value <= 0 ? 0 : value >= 2 ? 2 : 1;
      return old;
    }
    case MOE_OPT_PDL: {
      const int old = g_pdl;
      g_pdl = value ? 1 : 0;
      return old;
    }
    case MOE_OPT_SHARED_IN_GEMM: {
      const int old = g_shared_in_gemm;
      g_shared_in_gemm = value ? 1 : 0;
      return old;
    }
    case MOE_OPT_TILE_ORDER: {
      const int old = g_tile_order;
      g_tile_order = value ? 1 : 0;
      return old;
    }
    case MOE_OPT_SHARED_CTAS: {
      const int old = g_shared_ctas;
      g_shared_ctas = value < 0 ? 0 : value;
      return old;
    }
    case MOE_OPT_DYNAMIC_TILES: {
      const int old = g_dynamic_tiles;
      g_dynamic_tiles = value <= 0 ? 0 : value >= 2 ? 2 : 1;
      return old;
    }
    case MOE_OPT_B_PREFETCH: {
      const int old = g_b_prefetch;
      g_b_prefetch = value < 0 ? 0 : value > 16 ? 16 : value;
      return old;
    }
    case MOE_OPT_FUSED_ROUTING: {
      const int old = g_fused_routing;
      g_fused_routing = value <= 0 ? 0 : value >= 3 ? 3 : value;
      return old;
    }
    case MOE_OPT_FUSED_COMBINE: {
      const int old = g_fused_combine;
      g_fused_combine = value ? 1 : 0;
      return old;
    }
    default: return MOE_ERR_INVALID_ARG;
  }
}

int moe_set_trace_events(void* const* events, int n_events) {
  g_trace_events = (events && n_events > 0) ? events : nullptr;
  g_trace_n = g_trace_events ? n_events : 0;
  return MOE_OK;
}

int moe_layer_launch_count(const moe_config_t* cfg) {
  if (!cfg_valid(cfg) || cfg->T == 0) return 0;
  int n = 0;
  // router projection and top-k softmax (one launch when fused)
  const int nsplit = router_k_split(cfg->T, cfg->E, cfg->D);
  n += fused_router_on(cfg, nsplit) ? 1 : 2;
  // the shared expert inside the routed GEMMs: no launches of its own
  const bool sep_shared = cfg->I_shared > 0 && !shared_in_gemm_on(cfg);
  if (is_fp8(cfg)) {
    n += 1;                     // x to fp16 (or e4m3) rows
    n += sep_shared ? 2 : 1;    // h to fp16 (or e4m3) rows, routed (and shared)
  }
  if (small_route(static_cast<long long>(cfg->T) * cfg->k, cfg->E)) {
    n += 1;  // init_routing + permutation gather in one kernel
  } else {
    // histogram, scan + stable scatter: one launch after the fused router
    // (from its histograms), or as one cluster up to kClusterSortRows rows
    n += (chunk_sort_on(cfg) ||
          (g_fused_routing && static_cast<long long>(cfg->T) * cfg->k <= kClusterSortRows))
             ? 1
             : 2;
    if (gather_mode(cfg) == 0) n += 1;  // permutation gather
  }
  n += 2;  // routed gate/up, down
  if (sep_shared) n += 2;  // shared gate/up, down
  n += 1;  // finalize
  return n;
}

}  // extern "C"
