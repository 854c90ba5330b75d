/*
 * moe.h -- C ABI of the GB300 (sm_103a) sparse Mixture-of-Experts FFN layer.
 *
 * The layer, as the source pages state it:
 *   logits = x W_g                                   (router projection)
 *   (ids, w) = top-k of softmax(logits), renormalised (gating_top_k_softmax)
 *   rows grouped by expert                            (init_routing)
 *   h_e = act(x W13_e[:, :I]) * (x W13_e[:, I:])      (grouped matmul + swiglu)
 *   y_e = h_e W2_e                                    (grouped matmul)
 *   out = sum_j w_j y_{ids_j} + SharedExpert(x)       (finalize_routing)
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensors are device pointers, row-major and contiguous, owned by the
 *   caller.  The library allocates no device memory; scratch space comes from
 *   the caller's workspace `ws` of at least moe_workspace_size(cfg) bytes
 *   (256-byte aligned).  The first 256 bytes of `ws` are a control block that
 *   holds the device error word (and, with MOE_OPT_DYNAMIC_TILES, the GEMMs'
 *   tile counters).
 * - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *   asynchronous on that stream and returns after enqueueing its kernels.
 *   The compute calls enqueue only kernels and event records / waits (no
 *   host synchronisation, no allocation), so they can be captured into a
 *   CUDA graph; the first call on a device does one-time set-up (kernel
 *   attributes, moe_layer's side stream), so make it before capturing.
 * - Return value: MOE_OK or a negative moe_status_t.  Argument errors are
 *   detected on the host before anything is enqueued.  Data errors found on
 *   the device (an expert id outside [0, E), non-monotone offsets, a permuted
 *   position outside [0, T*k), non-finite router logits) never fault: the
 *   offending element is skipped or clamped and a code is recorded in the
 *   device error word, which moe_read_device_status() reads.
 * - Pointers must be 16-byte aligned and every row pitch a multiple of 16
 *   bytes, which makes D, I and I_shared multiples of 8 (16 for fp8 weights).
 * - Dtypes: act_dtype applies to x, W_g, the permuted rows and out.  w_dtype
 *   applies to W13, W2 and the shared expert's weights.  Supported pairs:
 *   (F32, F32), (BF16, BF16), (BF16, FP8_E4M3), (BF16, FP8_E4M3_NK),
 *   (BF16, FP8_E4M3_NK_A8).
 *   Router logits and gate weights are always fp32; the expert outputs
 *   y_perm and the shared-expert output are fp32, or bf16 for fp8-weight
 *   layers (one rounding each, inside the 6e-2 RMS bar of those layers).
 *   The intermediate h takes 4 bytes per element: fp32 for fp32 layers and
 *   for FP8_E4M3 weights; for bf16 weights two bf16 planes [M, I] -- h_hi =
 *   bf16(h) followed by h_lo = bf16(h - h_hi) -- which the down projection
 *   consumes as two bf16 tensor-core products, so that h keeps about 16
 *   significant bits.  FP8_E4M3 weights (W8A16, in the pages' [.., K, N]
 *   layout) run on the fp16 tensor-core kind: e4m3 expands exactly to fp16,
 *   and the A rows (x, then h) are fp16 rows times exact powers of two, so
 *   each product equals the bf16-activation product up to fp32 summation
 *   order (x exactly; h rounded once to 11 significant bits relative to its
 *   row).
 * - FP8_E4M3_NK: the same e4m3 values and per-column scales, with each
 *   expert's matrix stored transposed (W13 [E, 2I, D], W2 [E, D, I], W13s
 *   [2 I_shared, D], W2s [D, I_shared]: the reduction dimension contiguous),
 *   as moe_pack_weights_nk writes it once from the [.., K, N] layout.  These
 *   layers run on the 8-bit tensor-core kind (kind::f8f6f4) with no weight
 *   expansion: every A row (x, then h) is scaled by an exact power of two so
 *   that its largest element lies in [128, 256) and carried as two e4m3
 *   terms, hi = e4m3(v) and lo = e4m3(v - hi), multiplied by the weights in
 *   two products into one fp32 accumulator.  A bf16 x is represented exactly
 *   except for elements below 2^-9 of their row's largest, which keep an
 *   absolute error under 2^-17 of it.  h is stored in bf16 (2 bytes per
 *   element; 8 significant bits) and reaches the down projection the same
 *   way, so both products see exactly the bf16 rows but for those small
 *   elements.
 * - FP8_E4M3_NK_A8 (W8A8, opt-in): the weights of FP8_E4M3_NK, and the
 *   activations quantised per row to one e4m3 term with a dynamic scale, as
 *   "用SGLang-JAX在TPU上优化Ling-2.6-1T" §5 ("激活量化", "逐通道
 *   direct_scaled_dot") describes: s = max|row| / 448 and q = e4m3(v / s)
 *   (fp32 divisions, nearest even, saturating); x per token before the
 *   permutation, h per row after it is stored in bf16; one 8-bit product per
 *   multiply-add, (sum q_a q_w) * s_a * s_w[n] after the reduction.  The
 *   router still projects the bf16 x.  This changes the result (e4m3 keeps
 *   4 significant bits of each activation); the bf16-activation layouts
 *   above are the configured arithmetic.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_F32 = 0,
  MOE_BF16 = 1,
  MOE_FP8_E4M3 = 2,   /* weights [.., K, N] as the pages write them */
  MOE_FP8_E4M3_NK = 3, /* the same weights transposed per matrix (moe_pack_weights_nk) */
  MOE_FP8_E4M3_NK_A8 = 4 /* FP8_E4M3_NK weights, activations quantised per row (W8A8) */
} moe_dtype_t;

/* SwiGLU: SiLU(gate) * up.  GEGLU: tanh-approximated GELU(gate) * up. */
typedef enum { MOE_ACT_SWIGLU = 0, MOE_ACT_GEGLU_TANH = 1 } moe_act_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,  /* null pointer, bad shape, misalignment, k > E, E > 512 */
  MOE_ERR_UNSUPPORTED = -2,  /* dtype / activation combination not built */
  MOE_ERR_CUDA = -3,         /* a CUDA runtime or driver call failed */
  MOE_ERR_DEVICE_CHECK = -4, /* the device error word is set (see moe_read_device_status) */
  MOE_ERR_WORKSPACE = -5     /* workspace missing, misaligned or too small */
} moe_status_t;

/* Codes stored in the device error word (bit flags, OR-ed together). */
#define MOE_DEV_BAD_EXPERT_ID 0x1   /* an id outside [0, E) reached routing */
#define MOE_DEV_BAD_OFFSETS 0x2     /* offsets not monotone or beyond T*k */
#define MOE_DEV_BAD_DEST 0x4        /* a permuted position outside [0, T*k) */
#define MOE_DEV_NONFINITE_LOGIT 0x8 /* NaN / Inf router logit (treated as -Inf) */
#define MOE_DEV_WAIT_TIMEOUT 0x10   /* a bounded pipeline wait gave up */

typedef struct {
  int32_t T;           /* tokens */
  int32_t D;           /* hidden size */
  int32_t E;           /* routed experts, 1..512 */
  int32_t k;           /* experts per token, 1..min(E, 16) */
  int32_t I;           /* routed expert intermediate size */
  int32_t I_shared;    /* shared expert / dense MLP intermediate, 0 = none */
  int32_t act;         /* moe_act_t */
  int32_t act_dtype;   /* moe_dtype_t: MOE_F32 or MOE_BF16 */
  int32_t w_dtype;     /* moe_dtype_t: MOE_F32, MOE_BF16 or MOE_FP8_E4M3 */
  int32_t renormalize; /* 1: gate weights renormalised over the k chosen experts */
} moe_config_t;

/* Bytes of workspace that every call below accepts for this configuration
 * (moe_layer needs all of it; the stage calls use the control block and
 * their own scratch).  Returns 0 for an invalid configuration. */
size_t moe_workspace_size(const moe_config_t* cfg);

/* Router projection and gating_top_k_softmax.
 * Pages: "千问 3.5 MoE 在 TPU 上的系统优化实战" (routed MoE paragraph: the
 * router projects each token and picks the top 10 experts by softmax);
 * "CANN/cann-recipes-infer：Qwen3-MoE优化", section "GMM使能和Routing优化"
 * (npu_moe_gating_top_k_softmax fuses top-k and softmax) and section
 * "融合RMSNorm + Cast" (the gate is computed in fp32).
 *   x          [T, D] act_dtype, or NULL: then `logits` is an input.
 *   Wg         [D, E] act_dtype (ignored when x is NULL).
 *   logit_bias [E] fp32 or NULL, added to x W_g (must be NULL when x is NULL).
 *   logits     [T, E] fp32: x W_g + bias with fp32 accumulation (output), or
 *              the input logits when x is NULL.
 *   topk_ids   [T, k] int32 out: experts by descending logit, the lower index
 *              first among equal logits.
 *   topk_w     [T, k] fp32 out: softmax over the k chosen logits when
 *              cfg->renormalize, else the full-softmax probabilities. */
int moe_route(const moe_config_t* cfg, const void* x, const void* Wg, const float* logit_bias,
              float* logits, int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes,
              void* stream);

/* init_routing + compute_expert_tokens + the permutation gather.
 * Pages: "CANN/cann-recipes-infer：Qwen3-MoE优化", section "GMM使能和Routing优化"
 * (npu_moe_init_routing orders rows by expert; npu_moe_compute_expert_tokens
 * counts tokens per expert); "千问 3.5 MoE 在 TPU 上的系统优化实战", SparseCore
 * paragraph (gather rows by routing index into one contiguous unpadded buffer).
 * Expanded row r = t*k + j is token t's j-th choice.
 *   topk_ids    [T, k] int32 in.
 *   x           [T, D] act_dtype in (may be NULL: no gather, x_perm unused).
 *   counts      [E] int32 out: rows per expert.
 *   offsets     [E+1] int32 out: exclusive scan of counts; offsets[E] = T*k.
 *   sorted_rows [T*k] int32 out: expanded row at each permuted position,
 *               grouped by expert, ascending r inside an expert (stable).
 *   dest        [T*k] int32 out: permuted position of each expanded row
 *               (inverse of sorted_rows; -1 for a row with an invalid id).
 *   x_perm      [T*k, D] act_dtype out: x_perm[p] = x[sorted_rows[p] / k]. */
int moe_permute(const moe_config_t* cfg, const int32_t* topk_ids, const void* x, int32_t* counts,
                int32_t* offsets, int32_t* sorted_rows, int32_t* dest, void* x_perm, void* ws,
                size_t ws_bytes, void* stream);

/* moe_permute for callers that cannot allocate device memory.  The source
 * pages have no counterpart: this is an interface for hosts that hand an
 * operator only its input and output buffers and forbid device allocation
 * while a request runs (a serving runtime that plans all device memory at
 * start-up, a plugin interface without a workspace argument), so they cannot
 * provide the workspace moe_permute takes.
 *   Same arguments, argument checks and results as moe_permute, without
 *   ws / ws_bytes (the configuration is validated exactly as there).  Its
 *   scratch (one expert histogram per routing segment: E <= 512 experts times
 *   at most 128 segments) is a fixed 256 KiB array in the library's device
 *   memory, held on every GPU that loads the library until the process exits.
 *   Limit: T*k <= 2^30 expanded rows, the same as every other call; larger
 *   sizes return MOE_ERR_INVALID_ARG before anything is enqueued.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  Nothing is allocated or freed, by this call
 *   or by any library routine it uses.
 *   Every call shares the one array, and it keeps the last call's contents:
 *   calls that overlap on the GPU (different streams, or different host
 *   threads, without ordering between them) race on it.
 *   There is no error word to read: a row with an id outside [0, E) gets
 *   dest = -1, is left out of sorted_rows, and offsets[E] < T*k. */
int moe_permute_noalloc(const moe_config_t* cfg, const int32_t* topk_ids, const void* x,
                        int32_t* counts, int32_t* offsets, int32_t* sorted_rows, int32_t* dest,
                        void* x_perm, void* stream);

/* Grouped matmul over expert segments, with the gate/up activation epilogue,
 * plus the shared expert (or dense MLP) over all tokens.
 * Pages: "CANN/cann-recipes-infer：Qwen3-MoE优化", sections "MoE TP优化 /
 * 计算分解" (w13 = [gate | up], swiglu = SiLU(first half) * second half) and
 * "GMM使能和Routing优化" (npu_grouped_matmul); "Gemma-4 模型优化报告" §2
 * (GEGLU experts; dense MLP added to the MoE output); "用SGLang-JAX在TPU上优化
 * Ling-2.6-1T" §5 "逐通道 direct_scaled_dot" (per-output-channel fp8 scale
 * applied after the K reduction).
 *   x_perm  [T*k, D] act_dtype: expert-ordered rows.
 *   offsets [E+1] int32: segment bounds (from moe_permute).
 *   W13     [E, D, 2I] w_dtype: columns [0, I) gate, [I, 2I) up
 *           (FP8_E4M3_NK: [E, 2I, D], rows [0, I) gate, [I, 2I) up).
 *   s13     [E, 2I] fp32 per-column scales (fp8 only, else NULL).
 *   W2      [E, I, D] w_dtype (FP8_E4M3_NK: [E, D, I]);
 *   s2      [E, D] fp32 (fp8 only, else NULL).
 *   h       out: act(gate) * up, [T*k, I] fp32 (fp32 layers and FP8_E4M3
 *           weights), [T*k, I] bf16 (FP8_E4M3_NK weights), or the bf16 pair
 *           [2, T*k, I] (hi plane, then lo plane) for bf16 weights.
 *   y_perm  [T*k, D] out: h W2 per segment (times s2 for fp8); fp32, or
 *           bf16 for fp8-weight layers (their 6e-2 bar leaves room, and the
 *           combine then reads half the bytes).
 *   x, W13s [D, 2*I_shared], s13s [2*I_shared], W2s [I_shared, D], s2s [D]:
 *           the shared expert (FP8_E4M3_NK: W13s [2*I_shared, D], W2s
 *           [D, I_shared]); x NULL (or I_shared == 0) skips it.
 *   h_s     shared intermediate, same layout as h with T rows.
 *   s_out   [T, D] out: shared expert output, fp32 (bf16 for fp8 weights). */
int moe_grouped_ffn(const moe_config_t* cfg, const void* x_perm, const int32_t* offsets,
                    const void* W13, const float* s13, const void* W2, const float* s2, void* h,
                    void* y_perm, const void* x, const void* W13s, const float* s13s,
                    const void* W2s, const float* s2s, void* h_s, void* s_out, void* ws,
                    size_t ws_bytes, void* stream);

/* finalize_routing fused with the shared-expert add.
 * Pages: "CANN/cann-recipes-infer：Qwen3-MoE优化", section "GMM使能和Routing优化"
 * (npu_moe_finalize_routing restores token order and takes the weighted sum);
 * "千问 3.5 MoE 在 TPU 上的系统优化实战": y = Router(x) + SharedExpert(x).
 *   out[t] = round( sum_{j<k} w[t, j] * y_perm[dest[t*k + j]] + s[t] ),
 *   accumulated in fp32 with j ascending, the shared row added last, one
 *   rounding to act_dtype.
 *   y_perm [T*k, D] fp32 (bf16 for fp8-weight layers), dest [T*k] int32,
 *   topk_w [T, k] fp32, s [T, D] of y_perm's type or NULL, out [T, D]
 *   act_dtype. */
int moe_finalize(const moe_config_t* cfg, const void* y_perm, const int32_t* dest,
                 const float* topk_w, const void* s, void* out, void* ws, size_t ws_bytes,
                 void* stream);

/* The whole layer: moe_route, moe_permute, moe_grouped_ffn, moe_finalize on
 * one stream, with every intermediate carved from `ws`.  Arguments as above;
 * the shared-expert weights may be NULL when cfg->I_shared == 0. */
int moe_layer(const moe_config_t* cfg, const void* x, const void* Wg, const float* logit_bias,
              const void* W13, const float* s13, const void* W2, const float* s2,
              const void* W13s, const float* s13s, const void* W2s, const float* s2s, void* out,
              void* ws, size_t ws_bytes, void* stream);

/* Device byte offsets inside `ws` where moe_layer keeps its intermediates,
 * for inspection (logits, ids, weights, counts, offsets, sorted_rows, dest,
 * x_perm, h, y_perm, h_s, s).  `which` is one of the MOE_WS_* indices;
 * returns (size_t)-1 for an unknown index, an invalid configuration, or an
 * fp8-only region of a layer without fp8 weights. */
#define MOE_WS_LOGITS 0
#define MOE_WS_TOPK_IDS 1
#define MOE_WS_TOPK_W 2
#define MOE_WS_COUNTS 3
#define MOE_WS_OFFSETS 4
#define MOE_WS_SORTED_ROWS 5
#define MOE_WS_DEST 6
#define MOE_WS_X_PERM 7
#define MOE_WS_H 8
#define MOE_WS_Y_PERM 9
#define MOE_WS_H_SHARED 10
#define MOE_WS_S 11
/* fp8-weight layers only: x times exact powers of two [T, D] -- as fp16
 * rows (FP8_E4M3) or as two-term e4m3 rows [T, 2D], hi in bytes [0, D) and
 * lo in [D, 2D) (FP8_E4M3_NK) -- their inverse scales per token [T] and per
 * permuted row [T*k] (fp32); for these layers MOE_WS_X_PERM holds rows of
 * the same form. */
#define MOE_WS_X16 12
#define MOE_WS_TOK_INV 13
#define MOE_WS_ROW_INV 14
size_t moe_workspace_offset(const moe_config_t* cfg, int which);

/* Synchronises `stream`, reads and clears the device error word of `ws`.
 * Returns MOE_OK, MOE_ERR_DEVICE_CHECK (flags written to *flags when not
 * NULL) or MOE_ERR_CUDA. */
int moe_read_device_status(void* ws, void* stream, int32_t* flags);

/* Transposes one-byte (e4m3) weight matrices into the layout of
 * MOE_FP8_E4M3_NK layers; run once when the weights are loaded.
 * Pages: "用SGLang-JAX在TPU上优化Ling-2.6-1T" §5 "逐通道 direct_scaled_dot"
 * (fp8 tokens and fp8 weights fed straight to the matrix unit, f32 partial
 * sums, per-token and per-channel scales after the reduction).  The pages
 * write each projection input dimension first; this library's 8-bit
 * tensor-core path reads both operands with the reduction dimension
 * contiguous, hence this one-time copy.
 *   W     [G, K, N] device, one byte per element (the pages' layout: W13 with
 *         G = E, K = D, N = 2I; W2 with K = I, N = D; G = 1 for the shared
 *         expert's matrices).
 *   W_nk  [G, N, K] device out: W_nk[g][n][c] = W[g][c][n].  Must not
 *         overlap W.
 *   1 <= G <= 65535; K and N positive multiples of 16; both pointers
 *   16-byte aligned and the two buffers disjoint, else MOE_ERR_INVALID_ARG
 *   before anything is enqueued.
 *   Asynchronous on `stream`; needs no workspace. */
int moe_pack_weights_nk(const void* W, int64_t G, int32_t K, int32_t N, void* W_nk, void* stream);

/* Human-readable text of a moe_status_t. */
const char* moe_status_string(int status);

/* Kernel launches one moe_layer call enqueues for this configuration. */
int moe_layer_launch_count(const moe_config_t* cfg);

/* Kernel-variant options (process-wide; set them from the thread that
 * launches, between calls).  Returns the previous value, or
 * MOE_ERR_INVALID_ARG for an unknown option.
 *   MOE_OPT_PAIR_TILES: how grouped GEMMs with a full 256-column B tile
 *   use 2-CTA clusters (tcgen05 cta_group::2, M = 256 rows per tile, each CTA
 *   loading half of B; a group's last tile with at most 64 (gate/up) or 128
 *   (down) rows runs swapped, with the weights as the M = 256 operand and the
 *   rows as N): 3 (default) = when there are at least 150 rows per group on
 *   average; 1 = always; 2 = always, without swapped tails; 0 = never (one
 *   CTA per 128-row tile).  FP8_E4M3 GEMMs always use one CTA per tile;
 *   FP8_E4M3_NK GEMMs follow the same policy (their swapped tails stack the
 *   hi and lo e4m3 rows along N).  Results are the same up to fp32
 *   summation order. */
#define MOE_OPT_PAIR_TILES 1
/*   MOE_OPT_GATHER_A: where moe_layer's routed gate/up GEMM takes its A
 *   rows.  0 = a permuted copy of x written by the gather kernel, read by
 *   tiled TMA loads; 1 = no copy: the GEMM reads the rows of x (for fp8
 *   weights, x's fp16 or two-term e4m3 rows) with TMA tile::gather4 loads, on
 *   one-CTA tiles (measured 2.5-2.8x slower on GB300); 2 = no copy, for bf16
 *   layers: four extra warps of the GEMM copy each tile row's 128 bytes per
 *   k-block from x by 16-byte cp.async, eight lanes per row (fp8 layers take
 *   1); 3 (default) = 2 for bf16 layers with at least 32 routed rows per
 *   expert on average (prefill: Qwen3-MoE-style layer 526 -> 490 us,
 *   Gemma-4-style 491 -> 469 us on GB300), 0 otherwise and when
 *   MOE_OPT_SHARED_IN_GEMM is set for a layer that can take it.  Same
 *   results. */
#define MOE_OPT_GATHER_A 2
/*   MOE_OPT_DECODE_KERNEL: 1 (default) = the swap-AB decode kernel (weights
 *   as the 128-row MMA operand, 16 or 64 rows per tile, each active expert's
 *   weights streamed once) for decode-size passes where it measured faster: a
 *   single group (shared expert) of at most 64 rows, at most one row per group
 *   on average, up to 4 rows per group with at most 256 groups (bf16), or fp8
 *   weights at up to 16 rows per group; 0 = always the 128-row-tile kernel;
 *   2 / 3 = the decode kernel with 64 / 16 rows per tile for every routed or
 *   shared FFN pass (testing).  Same results up to fp32
 *   summation order. */
#define MOE_OPT_DECODE_KERNEL 3
/*   MOE_OPT_PDL: 1 (default) = kernels are launched with programmatic
 *   dependent launch (each kernel may be scheduled while its predecessor in
 *   the stream runs and waits on the device, with griddepcontrol.wait, for
 *   the predecessor's completion before it touches memory); 0 = plain stream
 *   order.  Same results. */
#define MOE_OPT_PDL 4
/*   MOE_OPT_SHARED_STREAM: 1 (default) = moe_layer runs the shared expert
 *   on a second stream owned by the library (one per device, created on the
 *   first call that needs it) that forks from the caller's stream once x is
 *   ready and joins it before the finalize kernel, so that the shared GEMMs
 *   overlap routing and the routed GEMMs; 2 = the same stream, forked after
 *   init_routing instead (the shared GEMMs then start beside the permutation
 *   kernel, which needs no shared memory, rather than ahead of the routing
 *   kernels, which do); 0 = everything on the caller's stream.  Same results.
 *   Fork and join are event record / wait pairs made under a lock, so calls
 *   from several host threads stay correct (their shared experts then
 *   serialise on the one side stream). */
#define MOE_OPT_SHARED_STREAM 5
/*   MOE_OPT_FUSED_COMBINE: 1 = moe_layer fuses the combine into the routed
 *   down projection (NEXT-1's second half: "千问 3.5 MoE 在 TPU 上的系统优化实战",
 *   SparseCore paragraph -- un-permute and reduce without the intermediate
 *   expert rows): the down pass multiplies each row by its routing weight and
 *   adds it, with fp32 atomics, into [T, D] fp32 sums (the y_perm region of the
 *   workspace, zeroed first), and the last kernel adds the shared row and
 *   rounds once; no y_perm rows are written or read.  The k rows of a token
 *   are then summed in whatever order they arrive, so the output may differ
 *   from the default's fixed j-ascending order in the last bit (run to run as
 *   well).  Layers with bf16 weights or K-contiguous e4m3 weights; others
 *   (and 0, the default) keep finalize's fixed order. */
#define MOE_OPT_FUSED_COMBINE 6
/*   MOE_OPT_TILE_ORDER: 1 = the grouped GEMMs schedule the experts heaviest
 *   first (most rows; the lower index first among equal counts), the
 *   longest-processing-time order of "企业官网建设流程全解析" §4 (sort the
 *   experts' work heaviest first so that the largest ones do not trail);
 *   every CTA sorts the expert counts itself (a bitonic sort in one warp)
 *   while it builds its tile schedule; 0 (default) = expert order.  Same
 *   results. */
#define MOE_OPT_TILE_ORDER 7
/*   MOE_OPT_SHARED_IN_GEMM: 1 = moe_layer runs the shared expert as one more
 *   group of the routed grouped GEMMs (NEXT-3: "用SGLang-JAX在TPU上优化
 *   Ling-2.6-1T" §5 "核内共享专家", the shared expert moved into the routed
 *   kernel): its token rows are appended to the permuted rows (rows R .. R+T-1
 *   of x_perm, h and y_perm), its tiles follow the routed tiles in the same
 *   persistent launches, and the layer makes no launches of its own for it.
 *   Layers whose I_shared equals I with bf16 or K-contiguous e4m3 weights
 *   (the workspace of such a layer always holds those T extra rows); other
 *   layers, and 0 (default), run the shared expert in its own launches (on
 *   the side stream, MOE_OPT_SHARED_STREAM).  Same results. */
#define MOE_OPT_SHARED_IN_GEMM 9
/*   MOE_OPT_FUSED_ROUTING: 1 (default) = the routing chain in fewer
 *   launches ("CANN/cann-recipes-infer：Qwen3-MoE优化", section "GMM使能和
 *   Routing优化": fused gate + gating_top_k_softmax, fused init_routing):
 *   (a) for more than 64 tokens of bf16 activations (64 <= E <= 512), the
 *   router projection and the top-k softmax are one kernel: a cluster of up
 *   to 4 CTAs per 128 tokens splits the fp32 sum over D into consecutive
 *   slices on the tensor core and hands the partial rows through distributed
 *   shared memory to the CTA that adds them in slice order and takes the
 *   top-k; inside moe_layer each of its CTAs also counts its tokens' ids per
 *   expert, and init_routing (above the one-launch size) is one kernel with
 *   a CTA per router CTA that sorts that CTA's rows from those histograms;
 *   (b) otherwise, for 8193 to 65536 expanded rows, the histogram, scan and
 *   stable scatter of init_routing are one cluster of 8 CTAs that exchange
 *   their expert histograms through distributed shared memory.
 *   (a) applies where its grid has at least 64 CTAs (prefill; decode batches
 *   take the split-K projection); 2 = (a) wherever the shape allows it, 3 =
 *   the same without the histogram sort (testing).  0 = a grouped-GEMM launch
 *   writing split-K planes, then the top-k kernel; a histogram kernel, then a
 *   scan + scatter kernel.  The logits may differ in the last bits between
 *   the two (another split of the fp32 sum over D); ids and weights follow
 *   from each one's own logits by the same rule, and the permutation is the
 *   same. */
#define MOE_OPT_FUSED_ROUTING 10
/*   MOE_OPT_B_PREFETCH: n > 0 = the grouped GEMMs' TMA producer also
 *   prefetches its weight box n k-blocks ahead into L2 (near the end of a
 *   tile, the first k-blocks of its next tile), so that more weight bytes are
 *   in flight from HBM than the shared-memory ring holds; for the weights
 *   read in one box per stage (bf16 as 64-column blocks, K-contiguous e4m3).
 *   0 (default) = off; at most 16.  Same results. */
#define MOE_OPT_B_PREFETCH 11
/*   MOE_OPT_DYNAMIC_TILES: the persistent grouped GEMMs (128-row and 2-CTA
 *   tiles) can hand out their tiles dynamically: each CTA's producer (the
 *   leader's, in a pair) takes tiles from a counter in the workspace's
 *   control block with an atomic add and passes them to the CTA's (pair's)
 *   other roles through a small queue in shared memory, one tile ahead, so
 *   that CTAs whose tiles run faster take more of them; the calls that launch
 *   those GEMMs zero the counters first (one memset).  2 (default) = for the
 *   prefill-sized gate/up passes (at least 1024 rows and 32 per group) whose
 *   tiles are at least 64 k-blocks long (D >= 4096 for bf16 weights, D >=
 *   8192 for K-contiguous e4m3 weights; Ling-style prefill layer 11.35-11.39
 *   -> 11.04-11.07 ms on GB300); 1 = every pass (the short
 *   down-pass tiles measured 3-8 % slower); 0 = tile t to CTA (pair) t modulo
 *   the grid.  Same results. */
#define MOE_OPT_DYNAMIC_TILES 12
/*   MOE_OPT_SHARED_CTAS: n > 0 = the shared expert's GEMMs on the library's
 *   side stream use at most n CTAs (their persistent grid), leaving the other
 *   SMs to the routed path's kernels that run beside them; 0 (default) = one
 *   CTA per SM.  Same results. */
#define MOE_OPT_SHARED_CTAS 13
int moe_set_option(int option, int value);

/* Per-kernel timing hook (process-wide, off by default).  `events` holds
 * n_events cudaEvent_t handles created by the caller; while set, each
 * moe_layer call records events[i] on its stream right before its i-th kernel
 * launch and events[L] after the last one (L = moe_layer_launch_count), so
 * consecutive events bracket exactly one kernel.  Calls with fewer than L+1
 * events record nothing.  Pass NULL / 0 to switch it off.  Not thread-safe:
 * set it from the thread that calls moe_layer.  Returns MOE_OK. */
int moe_set_trace_events(void* const* events, int n_events);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
