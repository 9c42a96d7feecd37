/*
 * moe_w4a8.h -- C ABI of the E2M1-K32 weight x FP8 activation variant of the
 * MoE expert computation (GB300, sm_103a).
 *
 * The variant is the one sglang-glm53-flash-sm120 pull request #13 ("SM120
 * FP8 prefill", description) adds for E2M1-K32 experts: E2M1 (FP4) weight
 * codes with one FP32 scale per 32 elements along K, applied in FP32, and
 * E4M3 activations with one FP32 scale per row.  Gate/up projection, SwiGLU,
 * requantisation of the intermediate, down projection and the top-k-weighted
 * reduction onto a caller-owned BF16 output are as in moe_fp8.h.
 *
 * Conventions are those of moe_fp8.h (device pointers owned by the caller,
 * asynchronous on `stream`, host-side argument errors returned before any
 * launch, device-side conditions OR-ed into *device_status, dense row-major
 * layouts, BF16 as uint16 bit patterns).
 *
 * Formats:
 *  - E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit; values 0,
 *    0.5, 1, 1.5, 2, 3, 4, 6 and their negatives; no NaN or infinity (the OCP
 *    Microscaling Formats FP4 element type).  Two codes per byte: element 2i
 *    in the low nibble of byte i, element 2i + 1 in the high nibble.
 *  - K32 weight scales: scale[row, kb] covers elements 32kb .. 32kb + 31 of
 *    that row; the quantiser sets it to amax / 6 (FP32) and the codes to
 *    E2M1(w / scale), rounded to nearest even and saturated at 6.
 *  - Row activation scales: one FP32 scale per row, amax / 448; codes
 *    E4M3(x / scale), rounded to nearest even and saturated at 448.
 *  A zero block or row gets scale 0 and zero codes.
 */
#ifndef MOE_W4A8_H
#define MOE_W4A8_H

#include <stddef.h>
#include <stdint.h>

#include "moe_fp8.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Per-row FP8 activation quantiser (the row quantizer the SM120 page names).
 *  x      [M, K] BF16 bits
 *  q      [M, K] E4M3 codes out
 *  scale  [M] FP32 out
 * K % 32 == 0, K >= 32; x and q 16-byte aligned.  M == 0 does nothing. */
moe_status moe_quantize_act_per_row(const uint16_t* x, int64_t M, int K, uint8_t* q, float* scale,
                                    moe_stream_t stream);

/* K32 E2M1 weight quantiser.
 *  w         [rows, K] BF16 bits (leading dimensions such as experts folded into rows)
 *  q_packed  [rows, K/2] packed E2M1 codes out
 *  scale     [rows, K/32] FP32 out
 * K % 32 == 0, K >= 32, rows >= 1; w and q_packed 16-byte aligned. */
moe_status moe_quantize_weight_k32(const uint16_t* w, int64_t rows, int K, uint8_t* q_packed, float* scale,
                                   moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Forward over a moe_plan plan (moe_fp8.h).
 *
 * For every route r = t * top_k + j the plan holds:
 *   g, u  = the gate and up rows of W13[e] against A[t]: per 32-wide K block
 *           the dot of the decoded codes times the block's weight scale,
 *           summed over the blocks in FP32, times a_scale[t];
 *   h     = silu(g) * u, requantised per route row (amax / 448, E4M3);
 *   y     = W2[e] against the requantised row, the same way, times its scale;
 *   c     = y * (topk_weights[t, j] * routed_scale).
 * out[t] = bf16_rn(f32(out[t]) + c_0 + c_1 + ...), the routes added in slot
 * order j in FP32.  Pad slots (ids >= M * top_k), blocks at and past P, and
 * blocks whose expert is -1 contribute nothing; any other expert id outside
 * [0, E) sets MOE_DEV_BAD_EXPERT and its block is skipped.
 *
 * The projections run on the tensor cores (tcgen05 kind::f8f6f4, E2M1 x E4M3
 * into tensor memory, each 32-wide K block promoted in FP32 with its weight
 * row's scale) when H and I are multiples of 128, block_m <= 64, w13 and w2
 * are 32-byte aligned and the scale arrays 16-byte aligned; otherwise, or
 * with path = MOE_W4A8_CUDA_CORES, on the CUDA cores.  Five launches either
 * way (a memset of the route flags, gate/up, requant, down, combine); the
 * workspace needs no initialisation.
 * ------------------------------------------------------------------------ */
typedef struct moe_w4a8_args {
  const uint8_t* a;                        /* [M, H] E4M3 activations                       */
  const float* a_scale;                    /* [M] FP32 row scales                           */
  const uint8_t* w13;                      /* [E, 2I, H/2] packed E2M1: gate rows, then up rows */
  const float* w13_scale;                  /* [E, 2I, H/32] FP32 K32 scales                 */
  const uint8_t* w2;                       /* [E, H, I/2] packed E2M1                       */
  const float* w2_scale;                   /* [E, H, I/32] FP32 K32 scales                  */
  const float* topk_weights;               /* [M, top_k] FP32 route weights                 */
  const int32_t* sorted_token_ids;         /* [sorted_cap] plan (moe_plan)                  */
  const int32_t* expert_ids;               /* [blocks_cap] plan                             */
  const int32_t* num_tokens_post_padded;   /* [1] device scalar P; never read on the host   */
  uint16_t* out;                           /* [M, H] BF16 bits, accumulated in place        */
  void* workspace;                         /* moe_w4a8_workspace_size bytes (scratch)       */
  int32_t* device_status;                  /* nullable [1]: MOE_DEV_* bits are OR-ed in     */
  uint8_t* debug_q_inter;                  /* nullable [sorted_cap, I]: intermediate codes by slot */
  float* debug_s_inter;                    /* nullable [sorted_cap]: their row scales       */
  int64_t M;                               /* tokens                                        */
  int64_t sorted_cap;                      /* length of sorted_token_ids                    */
  int64_t blocks_cap;                      /* length of expert_ids                          */
  size_t workspace_bytes;
  int32_t H;                               /* hidden size (K of the gate/up projection)     */
  int32_t I;                               /* intermediate size                             */
  int32_t E;                               /* experts                                       */
  int32_t top_k;
  int32_t block_m;
  float routed_scale;                      /* routed scaling factor (1.0 = none)            */
  int32_t path;                            /* MOE_W4A8_AUTO or MOE_W4A8_CUDA_CORES          */
} moe_w4a8_args;

/* path values: MOE_W4A8_AUTO (0) takes the tensor cores where the sizes and
 * alignments allow; MOE_W4A8_CUDA_CORES (1) always runs the projections on
 * the CUDA cores.  Both compute the same result up to FP32 summation order.
 * Any other value returns MOE_ERR_SHAPE. */
#define MOE_W4A8_AUTO 0
#define MOE_W4A8_CUDA_CORES 1

/* Workspace bytes of the forward (host-only; 0 for invalid sizes): route
 * flags [M * top_k], SwiGLU rows [M * top_k, I] FP32, their codes and row
 * scales, and the route contributions [M * top_k, H] FP32. */
size_t moe_w4a8_workspace_size(int64_t M, int H, int I, int top_k);

/* Run the forward.  Constraints: H % 32 == 0, I % 32 == 0, both >= 32;
 * 1 <= top_k <= 64; 8 <= block_m <= 64, block_m % 8 == 0; block_m * H and
 * block_m * I at most 131072; sorted_cap >= blocks_cap * block_m,
 * blocks_cap >= 1; a, w13, w2, out, the workspace and debug_q_inter 16-byte
 * aligned; all pointers on the current device, which must be sm_103. */
moe_status moe_w4a8_forward(const moe_w4a8_args* args, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_W4A8_H */
