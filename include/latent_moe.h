/*
 * latent_moe.h -- C ABI of the latent mixture-of-experts block on one GB300 (sm_103a).
 *
 * The block (from "SGLang and Miles Add Day-0 Support for Muse Spark Open", section
 * "MoE with Pooler, Unpooler and Per-Expert Normalization"; widths from "vLLM 对 Muse
 * Spark Open 的 Day 0 支持" (vLLM Day-0 support), section "潜空间 MoE"; router precision
 * from the same page's "Nvidia" section):
 *
 *   h_t   = RMSNorm_{g_in}(x_t)                         full-width norm        [T,d]
 *   l_t   = W_r h_t  (TF32 operands, FP32 accumulate)   router logits          [T,E]
 *   (e_t, w_t) = top-k of softmax(l_t), renormalised     packed ids/weights     [T,k]
 *   u_t   = RMSNorm_{g_pool}(W_pool h_t)                pooler + pooled norm   [T,p]
 *   y_tj  = W2_e (silu(Wg_e u_t) * Wu_e u_t), e = e_tj  routed SwiGLU experts
 *   c_t   = sum_j w_tj RMSNorm_{g_exp[e_tj]}(y_tj)      per-expert norm BEFORE the
 *                                                       FP32 route-weighted sum
 *   out_t = W_unpool c_t                                unpooler               [T,d]
 *
 * RMSNorm_g(v) = v / sqrt(mean(v^2) + eps) * g.  Slots j are ordered by logit, largest
 * first, ties to the lower expert id; the weighted sum runs in slot order in FP32.
 *
 * Conventions for every entry point:
 *  - All tensors are row-major and dense.  Pointers named "device" must point to
 *    device memory of the current CUDA device; the library reads or writes them only
 *    from kernels on `stream`.  Host pointers (configs, weight tables) are read during
 *    the call only.
 *  - The library allocates no memory and keeps no state beyond a per-device cache of
 *    attributes and kernel settings.  Every buffer belongs to the caller.
 *  - Calls are asynchronous on `stream` and never synchronise or read device memory
 *    from the host (except moe_read_status), so they can be captured in a CUDA graph.
 *  - Errors found on the host (null pointers, unsupported sizes, a workspace that is
 *    too small) are returned before anything is launched.  Errors found on the device
 *    (a bounded wait that ran out) are recorded in the workspace's status word and
 *    reported by moe_read_status; CUDA launch errors are returned as MOE_ERR_CUDA.
 *  - Results are deterministic: identical inputs give bit-identical outputs.
 *  - Outputs must not alias inputs.
 */
#ifndef LATENT_MOE_H
#define LATENT_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's stream and event handles (same layout as cudaStream_t /
 * cudaEvent_t), declared here so the header needs no CUDA include. */
typedef struct CUstream_st* moe_stream_t;
typedef struct CUevent_st* moe_event_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, k > E, bad dtype combination          */
  MOE_ERR_UNSUPPORTED = 2,   /* sizes outside what the kernels handle (see below)   */
  MOE_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or too small          */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed                */
  MOE_ERR_TIMEOUT = 5,       /* device: a pipeline wait ran past its time limit     */
  MOE_ERR_DEVICE_CHECK = 6   /* device: an index or value-range check failed        */
} moe_status_t;

typedef enum {
  MOE_F32 = 0,     /* float32; GEMM operands rounded to TF32 (ties away) */
  MOE_BF16 = 1,    /* bfloat16 */
  MOE_NVFP4 = 2    /* E2M1 codes + UE4M3 scale per 16 + FP32 tensor scale */
} moe_dtype_t;

/* Layer configuration.
 *   T      tokens in this call (>= 0; T = 0 is a no-op)
 *   d      model width           (multiple of 128, <= 32768)
 *   p      pooled (expert) width (multiple of 128, <= 8192)
 *   E      routed experts        (1..256)
 *   top_k  experts per token     (1..8, <= E)
 *   I      SwiGLU intermediate   (multiple of 128, <= 32768)
 *   eps    RMSNorm epsilon (added to mean(v^2) inside the square root)
 *   act    MOE_BF16 or MOE_F32: dtype of x, w_pool, w_unpool and the stored
 *          activations between the GEMMs
 *   expert MOE_BF16 or MOE_F32 (equal to act), or MOE_NVFP4 with act = MOE_BF16
 *          (then p and I must be multiples of 256)
 *   out    MOE_BF16 or MOE_F32: dtype of the layer output
 *   flags  0 or MOE_FLAG_TEST_TIMEOUT, MOE_FLAG_WEIGHT_TILES, one of MOE_FLAG_NVFP4_PAIR
 *          and MOE_FLAG_NVFP4_ONE_CTA (other bits must be zero) */
/* Test hook for the error path: the gate/up GEMM (and, in moe_forward_boundary, the
 * unpooler with the boundary's row workers) never issues its first operand load, so its
 * MMA wait runs out after 20 ms and every wait depending on it after as long; the call's
 * kernels then end early and moe_read_status reports MOE_ERR_TIMEOUT.  Outputs are
 * undefined.  Tests only. */
#define MOE_FLAG_TEST_TIMEOUT 0x80000000u
/* Run the BF16 / FP32 expert GEMMs with weight rows on the MMA's M side and each
 * expert's tokens on N (tiles shrink to the tokens present, in steps of 16) instead of
 * the default 128-token tiles on M.  Same results.  It removes the partly empty last
 * tile of each expert, but on a GB300 the expert GEMMs are bound by operand delivery
 * into shared memory, not by MMA work, and the default is faster at prefill sizes. */
#define MOE_FLAG_WEIGHT_TILES 0x40000000u
/* NVFP4 experts, kernel choice.  The expert GEMMs run either on one CTA per 128 x 256
 * output tile or on CTA pairs over 256 x 256 tiles (each CTA of a pair stages half of
 * the weight tile, so fewer bytes per MAC reach its shared memory).  Results are the
 * same, bit for bit.  By default the gate/up GEMM runs on single CTAs and the down GEMM
 * on pairs when T * top_k >= 256 * E (a full 256-row pair tile per expert on average),
 * else on single CTAs: measured on a GB300 at T = 16384, d = 8192, p = I = 4096, E = 256,
 * k = 8, the pairs take the down GEMM from 1.26 to 1.07 ms while the gate/up GEMM, whose
 * SwiGLU + requantisation epilogue is longer, is faster on single CTAs (2.16 against
 * 2.28 ms).  MOE_FLAG_NVFP4_PAIR puts both GEMMs on pairs, MOE_FLAG_NVFP4_ONE_CTA both on
 * single CTAs; setting both is an error. */
#define MOE_FLAG_NVFP4_PAIR 0x20000000u
#define MOE_FLAG_NVFP4_ONE_CTA 0x10000000u
typedef struct {
  int32_t T, d, p, E, top_k, I;
  float eps;
  int32_t act, expert, out;
  uint32_t flags;
} moe_config_t;

/* Weights as moe_forward consumes them (all device pointers, read only).  "Packed"
 * tensors are written by moe_pack_weights:
 *   g_in      [d]        FP32 gain of the full-width norm
 *   w_router  [E,d]      packed: FP32 router rows rounded to TF32
 *   w_pool    [p,d]      packed: FP16 (BF16 configs) or TF32-rounded FP32
 *   g_pool    [p]        FP32 gain of the pooled-input norm
 *   w13       packed gate/up rows of every expert: FP16 or TF32-rounded FP32
 *   w2        [E,p,I]    packed down projections: FP16 or TF32-rounded FP32
 *   g_exp     [E,p]      FP32 per-expert output-norm gains
 *   w_unpool  [d,p]      packed: FP16 or TF32-rounded FP32
 * BF16 configurations run every GEMM on FP16 operands and store every activation between
 * the GEMMs (h, u, s, y, c) in FP16: FP16 keeps 3 more significand bits than BF16 at the
 * same size and tensor-core rate, which keeps the rounding flips that FP32 accumulation
 * noise causes at storage points 8x rarer and 8x smaller.  h, u and c are RMS-normalised,
 * hence bounded by sqrt(width) * max|gain|; s and y are not bounded by construction.  The
 * BF16 -> FP16 weight copies are exact for |w| >= 2^-17.  A value of h, u or c that would
 * not fit FP16 (gains of extreme size, replayed weights with a large absolute sum), or an
 * s or y that overflowed it (and so made c non-finite), is reported through
 * moe_read_status (MOE_ERR_DEVICE_CHECK).                                            */
typedef struct {
  const float* g_in;
  const float* w_router;
  const void* w_pool;
  const float* g_pool;
  const void* w13;
  const void* w2;
  const float* g_exp;
  const void* w_unpool;
  /* NVFP4 experts only (NULL otherwise), all written by moe_quantize_nvfp4 except gs_act2:
   *   w13 / w2 then hold E2M1 codes (two per byte, even K element in the low nibble):
   *     w13 [E, 2I, p/2] with gate/up rows interleaved in blocks of 64,
   *     w2  [E, p, I/2];
   *   sf13, sf2  UE4M3 block scales (one per 16 elements along K) in the chunked layout:
   *     512-byte chunks indexed (row / 128, k / 64), chunk-row-major; inside a chunk the
   *     scale of (row, 16-block g) is at byte (row % 32) * 16 + ((row % 128) / 32) * 4
   *     + g % 4 -- the 4 x 32 arrangement the block-scaled MMA reads from tensor memory;
   *   gs13, gs2  [E] FP32 global scales (amax / (6 * 448) of each expert's W13 / W2);
   *   gs_act2    [E] FP32 static global scale of the requantised SwiGLU output (caller
   *              supplied, calibrated: the pages give no rule for it). */
  const uint8_t* sf13;
  const uint8_t* sf2;
  const float* gs13;
  const float* gs2;
  const float* gs_act2;
} moe_weights_t;

/* Canonical (unpacked) weights, as a checkpoint stores them (device pointers):
 *   w_router [E,d] FP32; w_pool [p,d]; w_gate, w_up [E,I,p]; w_down [E,p,I];
 *   w_unpool [d,p] (act / expert dtype as in the config).                     */
typedef struct {
  const float* w_router;
  const void* w_pool;
  const void* w_gate;
  const void* w_up;
  const void* w_down;
  const void* w_unpool;
} moe_canonical_weights_t;

/* Bytes of device workspace moe_route / moe_forward need for this config
 * (0 when the config is invalid).  The workspace holds the intermediates
 * (normalised rows, pooled rows, permuted expert inputs, SwiGLU and expert outputs,
 * the dispatch maps) and the status word.  It must be 256-byte aligned. */
size_t moe_workspace_size(const moe_config_t* cfg);

/* Clears the workspace's status word.  Call once after allocating a workspace
 * (before its first use); moe_read_status clears it again after each read. */
moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream);

/* Bytes of the packed buffers moe_pack_weights / moe_quantize_nvfp4 write.  which:
 * 0 = w_router (TF32 copy), 1 = w13, 2 = w2, 3 = w_pool, 4 = w_unpool, and for NVFP4
 * configs 5 = sf13, 6 = sf2, 7 = gs13, 8 = gs2.  Returns 0 for a buffer this config does
 * not use (the scale buffers of a BF16 or FP32 config). */
size_t moe_packed_bytes(const moe_config_t* cfg, int which);

/* Prepares weights for moe_forward ("SGLang and Miles Add Day-0 Support for Muse Spark
 * Open", section "Reading TensorRT-LLM's weights", describes the same need: the expert
 * GEMM reads gate and up rows of one tile together; this library uses its own layout).
 *  - w_router_out [E,d] FP32: w_router rounded to TF32 (ties away), the router's
 *    operand precision ("vLLM 对 Muse Spark Open 的 Day 0 支持", section "Nvidia":
 *    a TF32 router GEMM fed by the norm's FP32 output).
 *  - w13_out: gate and up rows interleaved in blocks of G rows (G = 128), so one
 *    256-row tile of the gate/up GEMM holds gate rows i..i+G and the matching up rows;
 *    converted to FP16 (BF16 configs) or rounded to TF32 (FP32 configs).
 *  - w_pool_out, w_unpool_out: FP16 copies (BF16 configs) or TF32-rounded copies.
 *  - w2_out: FP16 copy (BF16 configs) or TF32-rounded copy (FP32 configs).
 *  - NVFP4 configs: w13_out and w2_out must be NULL (moe_quantize_nvfp4 writes them);
 *    src->w_gate / w_up / w_down are not read.
 * Output buffers are caller-allocated with moe_packed_bytes; none may alias a source. */
moe_status_t moe_pack_weights(const moe_config_t* cfg, const moe_canonical_weights_t* src,
                              float* w_router_out, void* w13_out, void* w2_out,
                              void* w_pool_out, void* w_unpool_out, moe_stream_t stream);

/* NVFP4 expert weights from BF16 gate [E,I,p], up [E,I,p], down [E,p,I] (device):
 * per expert one FP32 global scale g = amax / (6 * 448) for gate+up together and one
 * for down; per 16 elements along K a UE4M3 scale sf = rne(bmax / (6 g)) (saturating at
 * 448); codes e2m1 = rne(x * (1 / sf) * (1 / g)) (saturating at 6) ("SGLang and Miles
 * Add Day-0 Support for Muse Spark Open", section "NVFP4 as a third MMA kind").  Output
 * layouts are those of moe_weights_t's NVFP4 fields; sizes from moe_packed_bytes. */
moe_status_t moe_quantize_nvfp4(const moe_config_t* cfg, const void* w_gate, const void* w_up,
                                const void* w_down, uint8_t* w13_out, uint8_t* sf13_out,
                                float* gs13_out, uint8_t* w2_out, uint8_t* sf2_out,
                                float* gs2_out, moe_stream_t stream);

/* Router only: full-width RMSNorm, TF32 router GEMM and top-k.
 *   x    [T,d] act dtype (device)
 *   ids  [T,k] int32 (device, written): chosen expert ids, slot order = logit order
 *   w    [T,k] FP32  (device, written): softmax over the chosen logits (sums to 1)
 * Routing replay passes these back to moe_forward. */
moe_status_t moe_route(const moe_config_t* cfg, const moe_weights_t* W, const void* x,
                       int32_t* ids, float* w, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* moe_route for callers that cannot allocate device memory at all -- code running where
 * no allocator is reachable, such as an engine that reserves all of its memory at start-up,
 * a plugin host that forbids device allocations, or a replayed CUDA graph that must not
 * grow its memory pool.  It takes no workspace: its scratch (status word, h32 and the
 * router's split-K partial logits) lives in a fixed 12 MiB + 256 B array inside the
 * library, which every GPU that loads the library holds until the process exits.  The
 * pages describe nothing like it; it is an addition of this library.
 *   Same arguments and results as moe_route, minus the workspace.
 *   Limit: T * d <= 2^21 (e.g. T <= 256 at d = 8192); larger calls return
 *   MOE_ERR_WORKSPACE before anything is launched.  Small T splits the router's
 *   reduction over up to 32 slices (as moe_route does), as many as 4 MiB of partial
 *   logits allow, so a decode batch does not stream the router weights through one CTA.
 *   The first call on a device looks up the array's device address (once per device,
 *   with that device current); make that first call before any stream capture.
 *   No cudaMalloc, cudaFree or allocating library routine is called.
 *   All calls share the one array, which keeps the previous call's contents (each call
 *   clears the status word it needs at zero): calls that overlap on the GPU -- on
 *   different streams, or from different threads -- race, so serialise them.
 *   Device-side failures of these calls are recorded in the array's status word:
 *   moe_read_noalloc_status reads it. */
moe_status_t moe_route_noalloc(const moe_config_t* cfg, const moe_weights_t* W, const void* x,
                               int32_t* ids, float* w, moe_stream_t stream);

/* The device-side status of the moe_route_noalloc calls on the current device since the
 * last read, like moe_read_status: synchronises `stream`, returns MOE_OK, MOE_ERR_TIMEOUT
 * or MOE_ERR_DEVICE_CHECK, writes the detail code to *detail (may be NULL) and clears
 * the status.  Allocates nothing. */
moe_status_t moe_read_noalloc_status(moe_stream_t stream, int32_t* detail);

/* The whole block for T tokens.
 *   x    [T,d] act dtype (device)
 *   ids, w  NULL: route internally.  Otherwise [T,k] int32 ids (each in [0,E)) and
 *           FP32 weights used instead of the router's (routing replay).
 *   out  [T,d] out dtype (device, written) */
moe_status_t moe_forward(const moe_config_t* cfg, const moe_weights_t* W, const void* x,
                         const int32_t* ids, const float* w, void* out, void* ws,
                         size_t ws_bytes, moe_stream_t stream);

/* What follows the block in the decoder, in one pass per row ("vLLM 对 Muse Spark Open 的
 * Day 0 支持", section "三明治归一化": each block sits between two norms,
 * x + post_norm(F(norm(x))); "SGLang and Miles Add Day-0 Support for Muse Spark Open",
 * section "Kernel Optimizations": post-FFN norm, gated residual add and pre-attention
 * norm fused, each row kept in registers across both RMS reductions):
 *   x_out  = x + gate * RMSNorm_{g_post}(y)       stored in the act dtype
 *   h_next = RMSNorm_{g_next}(x_out as stored)    stored in the act dtype
 * Uses cfg->T, d, eps, act (x, x_out, h_next) and out (y); the other fields must still
 * form a valid config.
 *   x       [T,d] act dtype (device): the residual stream entering the block
 *   y       [T,d] out dtype (device): the block's output, e.g. moe_forward's `out`
 *   g_post  [d] FP32 (device): gain of the post-norm;  g_next [d] FP32: of the next
 *           block's pre-norm
 *   gate    [d] FP32 (device) or NULL: per-channel gate of the residual add (NULL: 1).
 *           The pages do not give the gate's form; a per-channel vector is this
 *           library's reading.
 *   x_out   [T,d] act dtype (device, written); may be x itself (updated in place)
 *   h_next  [T,d] act dtype (device, written); may not overlap x, y or x_out
 * Every pointer 16-byte aligned.  Sums of squares are FP32, added in a fixed order; when
 * T is small several CTAs (a cluster) share each row through distributed shared memory.
 * Returns MOE_ERR_INVALID_ARG for null, misaligned or overlapping buffers. */
moe_status_t moe_boundary(const moe_config_t* cfg, const void* x, const void* y,
                          const float* g_post, const float* gate, const float* g_next,
                          void* x_out, void* h_next, moe_stream_t stream);

/* The block followed by its boundary, with the boundary's row pass inside the unpooler
 * GEMM's kernel ("SGLang and Miles Add Day-0 Support for Muse Spark Open", section "Kernel
 * Optimizations": the post-FFN norm, the gated residual add and the next block's pre-norm
 * fused into one kernel).  Same results as moe_forward(x, ids, w -> y) followed by
 * moe_boundary(x, y -> x_out, h_next) up to the order of FP32 additions in the two sums
 * of squares:
 *   y      [T,d] out dtype (device, written): the block output, as moe_forward's `out`;
 *          its rows are reread from L2 by the row pass, not from HBM
 *   x_out, h_next, g_post, gate, g_next: as for moe_boundary (x_out may be x)
 *   x, ids, w, ws, ws_bytes: as for moe_forward
 * The unpooler's epilogue stores the output tiles and their per-128-column sums of
 * squares and counts, per 32-row block, the column tiles stored; warps that are idle
 * during the GEMM's main loop run the row pass on each 2-row item once its block is
 * complete (a bounded wait: code 7 of moe_read_status if a block never completes).  The
 * kernel is launched with no more CTA pairs than the device can hold at once.  Shapes
 * whose unpooler runs split-K or on 128-column tiles (small T, d not a multiple of 256)
 * run moe_boundary's pass after the block instead.  Returns MOE_ERR_INVALID_ARG for null,
 * misaligned or overlapping buffers (y may overlap none of x, x_out, h_next). */
moe_status_t moe_forward_boundary(const moe_config_t* cfg, const moe_weights_t* W,
                                  const void* x, const int32_t* ids, const float* w,
                                  const float* g_post, const float* gate, const float* g_next,
                                  void* y, void* x_out, void* h_next, void* ws, size_t ws_bytes,
                                  moe_stream_t stream);

/* moe_forward with CUDA events recorded on `stream` at each stage boundary:
 * events[0] before the first kernel and events[i] after stage i-1 (i = 1..n_events-1,
 * at most moe_num_stages()+1 events).  For measurement only; same results. */
moe_status_t moe_forward_profiled(const moe_config_t* cfg, const moe_weights_t* W,
                                  const void* x, const int32_t* ids, const float* w,
                                  void* out, void* ws, size_t ws_bytes,
                                  moe_stream_t stream, moe_event_t* events, int n_events);

/* Number and names of the stages moe_forward_profiled brackets. */
int moe_num_stages(void);
const char* moe_stage_name(int stage);

/* Number of kernels moe_forward launches for this config (for launch accounting). */
int moe_forward_launches(const moe_config_t* cfg, int route_internally);

/* Byte offsets, inside the workspace of this config, of the intermediates a test may
 * inspect after a call (the buffers stay valid until the next call on the workspace):
 *   0 h32 [T,d] FP32 (TF32-rounded)   1 h16 [T,d] FP16     2 ids [T,k] int32
 *   3 w [T,k] FP32                    4 pooled [T,p] FP32   5 row_off [E+1] int32
 * Dispatched rows: row_off[e] is expert e's first row, row_cnt[e] its rows.  NVFP4
 * experts, and BF16 / FP32 experts when T*k >= 256*E, start every expert on a 128-row
 * boundary (R = 128 * (ceil(T*k/128) + E) rows in all), the rows after an expert's last
 * one being padding (zeros in A_perm and s for BF16 / FP32 experts); otherwise the rows
 * are packed (T*k of them).
 *   6 src [R] int32 (dispatched row -> t*k+j; padding rows hold no entry)
 *   7 inv [T*k] int32 (t*k+j -> dispatched row)
 *   8 A_perm [R,p] (FP16 / FP32)   9 s [R,I] (FP16 / FP32)
 *  10 y [R,p] (FP16 / FP32: FP32 for FP32 experts only)
 *  11 c [T,p] (FP16 / FP32)
 * NVFP4 configs: 8 A_perm [R, p/2] E2M1 codes, 9 s [R, I/2] codes, 10 y [R, p] FP16,
 * 12 sf_u, 13 sf_s chunked UE4M3 scales of A_perm / s, 14 alpha [R] FP32 per-row scales.
 * All configs: 15 row_cnt [E+1] int32 rows per expert;
 * moe_forward_boundary: 16 [T, d/128] FP32 sums of squares of the block output per 128
 * columns, 17 [8 * ceil(T/256) + 1] int32 column tiles stored per 32-row block, then the
 * row workers' item counter (all zero when the boundary ran as a separate pass).
 * Writes min(n, 18) offsets and returns how many it wrote (0 for an invalid config). */
int moe_workspace_offsets(const moe_config_t* cfg, size_t* offsets, int n);

/* Synchronises `stream`, returns the device-side status of every call since the last
 * read (MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_CHECK) and clears it.  detail (may
 * be NULL) receives a code naming the wait or check that failed first:
 *   1-7   a pipeline wait ran out (MOE_ERR_TIMEOUT): 1 producer slot, 2 MMA operands,
 *         3 MMA accumulator, 4 epilogue accumulator, 5 teardown drain, 6 combine rows,
 *         7 the fused boundary's row workers (moe_forward_boundary);
 *   16    a replayed expert id outside [0, E) (its slot is skipped);
 *   17    a row index check;
 *   18    the full-width norm: a non-finite input row, or an h value beyond the FP16
 *         range (BF16 configurations store h in FP16 for the pooler);
 *   19    the pooled-input norm: a non-finite row, or a u value beyond the FP16 range;
 *   20    the combine: a non-finite c, or (BF16 configurations) a c value beyond the
 *         FP16 range, e.g. from replayed weights whose absolute sum is large;
 *   21    NVFP4 experts: a requantised SwiGLU block whose scale saturated because its
 *         static global scale (gs_act2) is too small for it, or a non-finite s.
 *   Codes 18-21 report MOE_ERR_DEVICE_CHECK; the call's outputs are then undefined. */
moe_status_t moe_read_status(void* ws, size_t ws_bytes, moe_stream_t stream,
                             int32_t* detail);

/* Static description of a status code. */
const char* moe_status_string(moe_status_t s);

#ifdef __cplusplus
}
#endif
#endif /* LATENT_MOE_H */
