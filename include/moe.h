/*
 * block_scaled_fp8_moe -- routed-expert MoE layer for GB300 (sm_103a), C ABI.
 *
 * The layer (one call of moe_forward):
 *   router   : logits = x Wr^T (fp32, fixed order), sigmoid, + bias, top-k, weights normalised
 *   quant    : x -> MXFP8 (E4M3 codes, one UE8M0 scale per 32 along H)
 *   W13      : per live slot, gate/up projection with FP4 (E2M1) weights, SwiGLU, requant to MXFP8
 *   W2       : down projection per slot, scaled by the slot's routing weight
 *   combine  : out[t] = bf16( ((y_0 + y_1) + ...) ), slots in rank order
 *
 * Sources, cited by page and section:
 *  - "New Deepseek 4.1 flash recipe" (NVIDIA developer forum thread):
 *      post 2 "What changed / Speculative decoding": dead verification rows skip the MoE expert
 *        weight reads;
 *      post 4 "Quality and correctness": exact top-k ties break by lowest position;
 *      post 6 "Why TileLang": every kernel reduces in a fixed order, so a row's result does not
 *        depend on its batch; "How it works" items 1-3: block-scaled MMA for MXFP8 and FP8 x FP4,
 *        routed experts with FP8 activations x FP4 weights, 16/32/64-row decode tiles, panel
 *        rasterisation of weights larger than L2, MoE top-k gate and SwiGLU/quantisation casts.
 *  - TP4 serving profile README, settings table, "Experts" row: deterministic MoE reduction with a
 *    per-slot buffer and a fixed-order sum instead of atomics.
 *
 * Conventions shared by every entry point
 *  - All pointers are DEVICE pointers unless stated; the caller owns every buffer. The library
 *    allocates no device memory and keeps no per-call state.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). Calls are
 *    asynchronous and stream ordered; nothing synchronises the host except
 *    moe_check_device_status.
 *  - Return value: MOE_OK or an moe_status code. Argument and shape checks happen on the host
 *    before any launch; on failure nothing is launched. Launch failures return MOE_ERR_CUDA.
 *  - Device-side waits are bounded (about one second); an expired wait records an error code in
 *    the first 4 bytes of the workspace (the status word), the kernel unwinds, and
 *    moe_check_device_status then returns MOE_ERR_TIMEOUT. Inputs that only the device can check
 *    (an invalid anchor, a dead row that holds slots in the plan it was given) are recorded in the
 *    same word and reported as MOE_ERR_DEVICE_INPUT. Zero those 4 bytes once before first use (or
 *    call moe_check_device_status, which clears them).
 *  - bf16 tensors travel as uint16_t bit patterns.
 *  - Alignment (checked, MOE_ERR_INVALID_ARG otherwise): x, w_router, xq, hq, out, swiglu_debug
 *    16 bytes; xs, hs, topk_idx, topk_w 4 bytes; packed codes 32 bytes, packed scales 16 bytes.
 *  - Supported shapes: H % 128 == 0, I % 64 == 0, 1 <= k <= 32, k <= E <= 1024, T >= 0,
 *    H <= 16384, I <= 16384. T == 0 is a valid no-op. Anything else -> MOE_ERR_UNSUPPORTED_SHAPE.
 *
 * Data layouts (row-major, innermost dimension contiguous)
 *  x            bf16 [T, H]
 *  w_router     bf16 [E, H]
 *  bias         fp32 [E]                  added to the sigmoid score for selection only
 *  dead         u8   [T] or NULL          non-zero = dead verification row
 *  xq / xs      u8   [T, H] E4M3 codes / u8 [T, H/32] UE8M0 (byte b means 2^(b-127))
 *  hq / hs      u8   [S_max, I] / u8 [S_max, HS_PITCH] in plan order, S_max = T*k,
 *               HS_PITCH = roundup(I, 128) / 32 (bytes past I/32 are padding)
 *  MXFP4 canonical weights (input of moe_pack_*):
 *   w13 codes   u8 [E, 2I, H/2]  rows 0..I-1 gate, I..2I-1 up; element 2m in the LOW nibble
 *   w13 scales  u8 [E, 2I, H/32]
 *   w2 codes    u8 [E, H, I/2],  w2 scales u8 [E, H, I/32]
 *  Packed weights (what the GEMMs read; produced once by moe_pack_w13 / moe_pack_w2):
 *   tiles of 128 weight rows x 128 K elements; codes 8192 B per tile (64 B per row), scales one
 *   512 B block per tile (row r, K-block b at byte (r % 32) * 16 + (r / 32) * 4 + b).
 *   W13 tile (e, m, kc): rows 0..63 = gate rows 64m..64m+63, rows 64..127 = the matching up rows.
 *   W2 tile (e, n, kc): rows 128n..128n+127. K past the end of a row is zero-filled.
 *  Plan (written by moe_route_topk, S = live slots):
 *   topk_idx    i32 [T, k]   experts in rank order (key descending, ties -> lower index)
 *   topk_w      f32 [T, k]   score_j / sum of the k scores (summed in rank order)
 *   expert_counts  i32 [E]   live slots per expert
 *   expert_offsets i32 [E+1] exclusive prefix sum of expert_counts
 *   slot_of_row i32 [T*k]    plan row p (< S) -> slot t*k + j; rows inside an expert by token
 *   row_of_slot i32 [T*k]    slot t*k + j -> plan row, -1 for dead rows
 */
#ifndef BLOCK_SCALED_FP8_MOE_H
#define BLOCK_SCALED_FP8_MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_shape {
  int32_t T;      /* rows (tokens) in this call                      */
  int32_t H;      /* hidden size                                      */
  int32_t E;      /* experts                                          */
  int32_t k;      /* experts per row                                  */
  int32_t I;      /* expert intermediate size                         */
  int32_t flags;  /* MOE_FLAG_* bits, read by moe_w13_swiglu_grouped  */
} moe_shape;

/* moe_shape.flags */
#define MOE_FLAG_SWIGLU_DEBUG 1   /* W13 writes the fp32 SwiGLU values to swiglu_debug              */
#define MOE_FLAG_X_PLAN_ORDER 2   /* xq / xs given to W13 hold plan rows ([T*k, H] / [T*k, H/32]:
                                     row p = the token of plan row p), as moe_quant_mxfp8_plan writes */

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,        /* null pointer where one is required, negative size   */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* shape outside the supported set above               */
  MOE_ERR_WORKSPACE = 3,          /* workspace pointer null/misaligned or too small       */
  MOE_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed                    */
  MOE_ERR_TIMEOUT = 5,            /* a bounded device-side wait expired                  */
  MOE_ERR_DEVICE_INPUT = 6        /* an input checked on the device was invalid (anchor,  */
                                  /* or a dead row holding slots in the plan)             */
} moe_status;

typedef struct moe_intermediates {
  /* Optional outputs of moe_forward; any member may be NULL (then it lives in the workspace). */
  int32_t* topk_idx;       /* [T, k]   */
  float* topk_w;           /* [T, k]   */
  int32_t* expert_counts;  /* [E]      */
  int32_t* expert_offsets; /* [E + 1]  */
  uint8_t* xq;             /* [T, H]   */
  uint8_t* xs;             /* [T, H/32]*/
  uint8_t* hq;             /* [T*k, I] plan order */
  uint8_t* hs;             /* [T*k, HS_PITCH]     */
  float* swiglu;           /* [T*k, I] fp32 pre-requant SwiGLU, plan order */
} moe_intermediates;

/* Human-readable name of a status code (static string, never NULL). */
MOE_API const char* moe_status_string(int status);

/* Bytes of device workspace moe_forward needs for `shape` (256-byte aligned pointer required).
 * The other entry points need at most this much; 0 on an unsupported shape. */
MOE_API size_t moe_workspace_bytes(const moe_shape* shape);

/* Bytes of packed codes / packed scales for W13 (gate+up) and W2 of all E experts. */
MOE_API size_t moe_packed_w13_bytes(const moe_shape* shape, size_t* scale_bytes);
MOE_API size_t moe_packed_w2_bytes(const moe_shape* shape, size_t* scale_bytes);

/* MXFP4 quantisation of fp32 weights, per 32 consecutive elements of a row:
 *   s = smallest integer with max|w| <= 6 * 2^s (clamped to [-127, 127]; all-zero block -> -127),
 *   code = E2M1 round-to-nearest-even of w * 2^-s. Scale byte = s + 127.
 * w fp32 [rows, cols] -> q u8 [rows, cols/2] (element 2m low nibble), s u8 [rows, cols/32].
 * cols % 32 == 0. A one-time weight-preparation step, not part of the layer's step. */
MOE_API int moe_quant_mxfp4(int32_t rows, int32_t cols, const float* w, uint8_t* q, uint8_t* s, void* stream);

/* Canonical MXFP4 weights -> packed tiles (layouts above). Outputs must not alias inputs. */
MOE_API int moe_pack_w13(const moe_shape* shape, const uint8_t* q, const uint8_t* s, uint8_t* q_packed,
                 uint8_t* s_packed, void* stream);
MOE_API int moe_pack_w2(const moe_shape* shape, const uint8_t* q, const uint8_t* s, uint8_t* q_packed,
                uint8_t* s_packed, void* stream);

/* Router: sigmoid gate with bias-selected top-k and the expert plan.
 * "New Deepseek 4.1 flash recipe", post 6 "How it works" item 3 (TileKernels MoE top-k gate);
 * post 4 "Exact indexer selections" (ties by lowest index); post 2 (dead verification rows).
 * logit[t,e]: h cut into chunks of 64; each chunk summed sequentially in fp32 from +0 with fused
 * multiply-add; chunk sums added left to right from +0. score = 1 / (1 + exp(-logit)) with a
 * library-independent exp built from fp32 +, -, *, / (Cody-Waite reduction, degree-7 Taylor
 * polynomial), key = score + bias[e]. Dead rows are routed (topk_idx/topk_w written) but take no
 * slot. All outputs are required (non-NULL). ws: workspace of moe_workspace_bytes(shape). */
MOE_API int moe_route_topk(const moe_shape* shape, const uint16_t* x, const uint16_t* w_router, const float* bias,
                   const uint8_t* dead, int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                   int32_t* expert_offsets, int32_t* slot_of_row, int32_t* row_of_slot, void* ws,
                   size_t ws_bytes, void* stream);

/* Dead verification rows from the caller's survival estimates ("New Deepseek 4.1 flash recipe",
 * post 2, "Speculative decoding": draft rows whose estimated chance of surviving verification is
 * below 0.2 skip the MoE expert weight reads). dead[t] = (p_survive[t] < threshold) ? 1 : 0,
 * compared in fp32; a row exactly at the threshold and a NaN estimate stay live. p_survive: fp32
 * [T] (4-byte aligned), dead: u8 [T], both device memory owned by the caller; the result feeds the
 * `dead` argument of the calls below. T == 0 is a no-op; T < 0, NULL pointers or a NaN threshold
 * -> MOE_ERR_INVALID_ARG. */
MOE_API int moe_dead_from_survival(int32_t T, const float* p_survive, float threshold, uint8_t* dead, void* stream);

/* MXFP8 quantisation of bf16 rows ("How it works" item 3, quantisation casts):
 *   s = smallest integer with max|x| <= 448 * 2^s (clamped to [-127, 127]; zero block -> -127),
 *   code = E4M3 round-to-nearest-even of x * 2^-s (never saturates). cols % 32 == 0. */
MOE_API int moe_quant_mxfp8(int32_t rows, int32_t cols, const uint16_t* x, uint8_t* q, uint8_t* s, void* stream);

/* The same quantisation written in plan order, the form the wide-tile W13 reads (and what
 * moe_forward runs for large batches): the codes and scale bytes of token t go to plan rows
 * row_of_slot[t*k + j] of xq_plan u8 [T*k, H] / xs_plan u8 [T*k, H/32] (slots with -1 are skipped;
 * rows past the live slots are left untouched), and also to xq / xs in token order when those are
 * non-NULL (both or neither). row_of_slot as written by moe_route_topk. x 16-byte aligned, xq_plan
 * and xq 8-byte aligned. */
MOE_API int moe_quant_mxfp8_plan(const moe_shape* shape, const uint16_t* x, const int32_t* row_of_slot,
                                 uint8_t* xq_plan, uint8_t* xs_plan, uint8_t* xq, uint8_t* xs, void* stream);

/* Gate/up grouped GEMM fused with SwiGLU and MXFP8 requantisation, for every live slot:
 *   g = Wg[e] x^, u = Wu[e] x^ (block-scaled FP8 x FP4 tensor-core MMA, fp32 accumulate),
 *   a = g * sigmoid(g) * u (fp32), then per 32 along I: the MXFP8 rule of moe_quant_mxfp8.
 * Writes hq/hs rows in plan order (row p = slot slot_of_row[p]); swiglu_debug (nullable, written
 * when shape->flags has MOE_FLAG_SWIGLU_DEBUG) gets a. xq / xs are token rows [T, H] / [T, H/32],
 * or plan rows [T*k, H] / [T*k, H/32] with MOE_FLAG_X_PLAN_ORDER. expert_offsets / slot_of_row as
 * produced by moe_route_topk. w13 / w13_s are PACKED weights. */
MOE_API int moe_w13_swiglu_grouped(const moe_shape* shape, const uint8_t* xq, const uint8_t* xs, const uint8_t* w13,
                           const uint8_t* w13_s, const int32_t* expert_offsets, const int32_t* slot_of_row,
                           uint8_t* hq, uint8_t* hs, float* swiglu_debug, void* ws, size_t ws_bytes,
                           void* stream);

/* Down grouped GEMM and fixed-order weighted combine (TP4 profile README, "Experts" row):
 *   per slot (t, j) with plan row p: y_j = topk_w[t, j] * (W2[e] h^[p]) in fp32 (the product
 *   W2[e] h^[p] sits in a per-slot buffer in the workspace, one fp32 multiply by the weight),
 *   out[t] = bf16_rne( ((y_0 + y_1) + ...) ), slots in rank order; dead rows get +0.0.
 * w2 / w2_s are PACKED weights. dead (u8 [T] or NULL) is the mask the plan was made with: a row
 * with dead[t] != 0 gets +0.0 whatever the plan says, and if the plan still gives it slots (a plan
 * made without that mask) the status word records it (moe_check_device_status ->
 * MOE_ERR_DEVICE_INPUT). With dead = NULL a row is dead when row_of_slot[t*k] == -1. This call is
 * moe_w2_grouped followed by moe_combine on the workspace's per-slot buffer. */
MOE_API int moe_w2_combine_grouped(const moe_shape* shape, const uint8_t* hq, const uint8_t* hs, const uint8_t* w2,
                           const uint8_t* w2_s, const float* topk_w, const int32_t* expert_offsets,
                           const int32_t* slot_of_row, const int32_t* row_of_slot, const uint8_t* dead,
                           uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/* The down-projection GEMM alone (the first half of moe_w2_combine_grouped), into a per-slot buffer
 * the caller owns, in plan order and before the routing weight: y fp32 [T*k, H], 16-byte aligned;
 * row p (p < live slots) = W2[e] h^[p], e the expert of plan row p; rows past the live slots are
 * not written. ws: a workspace of at least 256 bytes (its first 4 bytes are the status word;
 * moe_workspace_bytes is not needed). */
MOE_API int moe_w2_grouped(const moe_shape* shape, const uint8_t* hq, const uint8_t* hs, const uint8_t* w2,
                           const uint8_t* w2_s, const int32_t* expert_offsets, const int32_t* slot_of_row,
                           float* y, void* ws, size_t ws_bytes, void* stream);

/* The fixed-order combine alone (TP4 profile README, "Experts" row): with r_j = row_of_slot[t*k+j]
 * and y_j = topk_w[t, j] * y[r_j] (fp32, one rounding), out[t] = bf16_rne(((y_0 + y_1) + ...) +
 * y_{k-1}) in fp32, slots in rank order, for each row t with row_of_slot[t*k] >= 0 and (dead ==
 * NULL or dead[t] == 0); every other row gets +0.0. y fp32 [T*k, H] as moe_w2_grouped writes it
 * (16-byte aligned), topk_w f32 [T, k] and row_of_slot i32 [T*k] as the router writes them, dead
 * u8 [T] or NULL, out bf16 [T, H]. A dead row that holds slots is recorded as for
 * moe_w2_combine_grouped. ws: at least 256 bytes, as for moe_w2_grouped. */
MOE_API int moe_combine(const moe_shape* shape, const float* y, const float* topk_w, const int32_t* row_of_slot,
                        const uint8_t* dead, uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/* Both expert GEMMs on a plan: moe_w13_swiglu_grouped (hq / hs, and swiglu_debug when flags ask for
 * it) followed by moe_w2_grouped (y, plan order, before the routing weight), with the same
 * arguments and results as those two calls. For decode-sized batches (at most 32 plan rows per
 * expert on average) they run as ONE persistent launch: each CTA streams its down-projection weight
 * tiles as soon as it has finished its gate/up tiles, and gathers an expert's h rows once every
 * gate/up tile of that expert is stored (per-expert counters in the workspace, zeroed by this call
 * before the launch). ws: workspace of moe_workspace_bytes(shape). */
MOE_API int moe_experts_grouped(const moe_shape* shape, const uint8_t* xq, const uint8_t* xs, const uint8_t* w13,
                                const uint8_t* w13_s, const uint8_t* w2, const uint8_t* w2_s,
                                const int32_t* expert_offsets, const int32_t* slot_of_row, uint8_t* hq, uint8_t* hs,
                                float* swiglu_debug, float* y, void* ws, size_t ws_bytes, void* stream);

/* The whole layer: route -> quant -> W13+SwiGLU+requant -> W2 -> combine, on one stream, no host
 * synchronisation and no allocation (capturable in a CUDA graph for a fixed shape). For
 * decode-sized batches W13 and W2 run as one launch, as in moe_experts_grouped; for at most 12 rows
 * and 256 experts that launch also takes the top-k and builds the plan itself (every CTA from the
 * router's scores, the same choices and weights as moe_route_topk), so the layer is two launches.
 * `inter` (nullable) receives the intermediates the caller wants to keep. */
MOE_API int moe_forward(const moe_shape* shape, const uint16_t* x, const uint16_t* w_router, const float* bias,
                const uint8_t* dead, const uint8_t* w13, const uint8_t* w13_s, const uint8_t* w2,
                const uint8_t* w2_s, uint16_t* out, const moe_intermediates* inter, void* ws,
                size_t ws_bytes, void* stream);

/* Anchored verify rows (TP4 serving profile README, settings table row "Verify length": verify
 * rows that the confidence head does not expect to survive reuse the anchor row's experts inside
 * the router, so they read no extra expert weights).
 *   anchor  i32 [T] or NULL: -1 = the row routes itself; a in [0, T) = the row takes row a's
 *           experts (in a's rank order) and weights them with its own scores,
 *           w_j = score[t, e_j] / ((score[t, e_0] + score[t, e_1]) + ...). Row a must route itself.
 * An anchor outside [0, T) or pointing at an anchored row is ignored (that row routes itself) and
 * recorded in the workspace status word (moe_check_device_status then returns
 * MOE_ERR_DEVICE_INPUT). Otherwise identical to moe_route_topk / moe_forward, which are these
 * calls with anchor = NULL. anchor must be 4-byte aligned. */
MOE_API int moe_route_topk_anchored(const moe_shape* shape, const uint16_t* x, const uint16_t* w_router,
                                    const float* bias, const uint8_t* dead, const int32_t* anchor,
                                    int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                                    int32_t* expert_offsets, int32_t* slot_of_row, int32_t* row_of_slot, void* ws,
                                    size_t ws_bytes, void* stream);
MOE_API int moe_forward_anchored(const moe_shape* shape, const uint16_t* x, const uint16_t* w_router,
                                 const float* bias, const uint8_t* dead, const int32_t* anchor, const uint8_t* w13,
                                 const uint8_t* w13_s, const uint8_t* w2, const uint8_t* w2_s, uint16_t* out,
                                 const moe_intermediates* inter, void* ws, size_t ws_bytes, void* stream);

/* Shared expert (TP4 serving profile README: "Rank-0 decode profile" table, shared expert on a side
 * stream; settings row DSV41_SHARED_PAD_K, the shared expert runs on an MXFP8 kernel): one dense
 * SwiGLU expert every live row passes through beside the routed ones, with MXFP8 (E4M3 + UE8M0/32)
 * weights, the same SwiGLU and MXFP8 requantisation as a routed expert, weight 1; its row is added
 * after the routed slots: out[t] = bf16_rne((((y[t,0] + y[t,1]) + ...) + y[t,k-1]) + y_shared[t]).
 * Dead rows stay +0.0.
 * Shapes: the shared expert is described by moe_shape {T, H, E = 1, k = 1, I = I_shared}.
 *  canonical codes  u8 [2 I_s, H] E4M3 (rows 0..I_s-1 gate, I_s..2I_s-1 up), scales u8 [2 I_s, H/32];
 *                   u8 [H, I_s] / [H, I_s/32] for the down projection.
 *  packed           tiles of 128 rows x 128 K elements, 16384 B of codes per tile (128 B per row),
 *                   scale blocks as for the routed experts; gate/up interleave as W13 above. */
typedef struct {
  int32_t I;                                 /* shared intermediate size (I % 64 == 0)            */
  const uint8_t* w13;                        /* packed by moe_pack_shared_w13                     */
  const uint8_t* w13_s;
  const uint8_t* w2;                         /* packed by moe_pack_shared_w2                      */
  const uint8_t* w2_s;
  void* ws;                                  /* moe_shared_workspace_bytes(shape, I), 256-B aligned */
  size_t ws_bytes;
} moe_shared_expert;

MOE_API size_t moe_packed_shared_w13_bytes(const moe_shape* shared_shape, size_t* scale_bytes);
MOE_API size_t moe_packed_shared_w2_bytes(const moe_shape* shared_shape, size_t* scale_bytes);
MOE_API int moe_pack_shared_w13(const moe_shape* shared_shape, const uint8_t* q, const uint8_t* s,
                                uint8_t* q_packed, uint8_t* s_packed, void* stream);
MOE_API int moe_pack_shared_w2(const moe_shape* shared_shape, const uint8_t* q, const uint8_t* s,
                               uint8_t* q_packed, uint8_t* s_packed, void* stream);
/* Scratch of the shared expert for a layer of `shape` (T rows); 0 for an unsupported I_shared. */
MOE_API size_t moe_shared_workspace_bytes(const moe_shape* shape, int32_t I_shared);
/* moe_forward_anchored plus the shared expert. With side_stream non-NULL the shared expert's
 * GEMMs run there, forked from `stream` after the activation quantisation and joined before the
 * combine (events created and released inside the call); with NULL they run on `stream`. */
MOE_API int moe_forward_shared(const moe_shape* shape, const uint16_t* x, const uint16_t* w_router,
                               const float* bias, const uint8_t* dead, const int32_t* anchor, const uint8_t* w13,
                               const uint8_t* w13_s, const uint8_t* w2, const uint8_t* w2_s,
                               const moe_shared_expert* shared, uint16_t* out, const moe_intermediates* inter,
                               void* ws, size_t ws_bytes, void* stream, void* side_stream);

/* Test hook for the bounded waits: launches one thread that waits on a barrier nothing arrives at,
 * for limit_ns (<= 2 s). The wait expires, writes its code into the status word at the start of
 * `ws` and the kernel returns; moe_check_device_status then reports MOE_ERR_TIMEOUT. No fault, no
 * hang, the context stays usable. Not part of the layer. */
MOE_API int moe_selftest_timeout(void* ws, uint64_t limit_ns, void* stream);

/* Rate probe of the block-scaled tensor-core instruction the grouped GEMMs use (tcgen05.mma
 * kind::mxf8f6f4, E2M1 x E4M3 with UE8M0 scales per 32; "New Deepseek 4.1 flash recipe", post 6
 * "How it works" item 1): one CTA per SM issues `iters` back-to-back M = 128, N = 256, K = 32 MMAs
 * from operands resident in shared memory, with nothing else to do (mode 0: the denominator of the
 * prefill GEMMs' tensor utilisation). Mode bits move it toward what the GEMMs issue: bit 0, the
 * K-chunks (4 MMAs each) read 4 different operand buffers in turn; bit 1, each K-chunk is preceded
 * by its scale copies (tcgen05.cp of one A and two B scale atoms); bit 2, N = 224. The caller times
 * the call with CUDA events on `stream`; *flops receives the multiply-add work (2 * 128 * N * 32 *
 * iters * CTAs) and *ctas the grid. Not part of the layer. iters in [1, 2^24], mode in [0, 7];
 * ws: at least 256 bytes, its first 4 bytes the status word. */
MOE_API int moe_probe_mma_rate(int32_t iters, int32_t mode, int32_t* ctas, int64_t* flops, void* ws,
                               size_t ws_bytes, void* stream);

/* Allocation-free variant of moe_route_topk, for callers that cannot allocate device memory:
 * engines that reserved all of HBM for their own pool at start-up, or code running inside a host
 * framework's callback where allocation is not allowed. It takes no workspace; its scratch lives in
 * a 512 KiB array inside the library, present on every GPU that loads it until exit. The pages have
 * no counterpart to this entry point: it is an interface convenience, not part of the method.
 * Same arguments and results as moe_route_topk without ws/ws_bytes. Limits: T <= 256 and
 * T * E <= 65536, otherwise MOE_ERR_UNSUPPORTED_SHAPE and nothing is launched. The first call on a
 * device looks up the array's device address (once per device; make that first call before any
 * stream capture). All calls share the array: calls that can overlap on the GPU race and must be
 * serialised by the caller. Nothing in it needs clearing between calls. Allocates nothing. */
MOE_API int moe_route_topk_noalloc(const moe_shape* shape, const uint16_t* x, const uint16_t* w_router,
                                   const float* bias, const uint8_t* dead, int32_t* topk_idx, float* topk_w,
                                   int32_t* expert_counts, int32_t* expert_offsets, int32_t* slot_of_row,
                                   int32_t* row_of_slot, void* stream);

/* Test/debug helper: synchronises `stream`, reads and clears the device status word at the start
 * of `ws`, and returns MOE_OK, MOE_ERR_TIMEOUT (an expired device-side wait) or
 * MOE_ERR_DEVICE_INPUT (an input the device found invalid); MOE_ERR_CUDA if the stream itself
 * failed. */
MOE_API int moe_check_device_status(void* ws, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* BLOCK_SCALED_FP8_MOE_H */
