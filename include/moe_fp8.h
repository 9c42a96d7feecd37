/*
 * moe_fp8.h -- C ABI of the block-scaled FP8 MoE expert library for GB300
 * (sm_103a).
 *
 * The library computes the routed MoE expert layer with FP8 (E4M3) operands
 * and FP32 block scales, as described by FlashInfer pull request #4287
 * ("feat(cake_alpha_moe): add optimized Blackwell W8A8 expert up/down
 * compute": commit summary; PR description, "Public contract and review
 * fixes") and SGLang pull request #43556 ("Requantize block-FP8 MoE weights
 * to UE8M0 for DeepGEMM": "Motivation", "Modifications").
 *
 * Conventions shared by every entry point:
 *  - Pointers are DEVICE pointers on the current CUDA device unless the
 *    argument says otherwise; the caller owns every buffer.  The library
 *    allocates no device memory and keeps no per-call global state, with
 *    one exception: the allocation-free forward at the end of this header
 *    draws its scratch from a fixed static device array (32 MiB per GPU
 *    that loads the library) that all of its calls share.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Argument errors are detected on the host and returned
 *    before anything is launched; a failed launch returns MOE_ERR_CUDA.
 *  - Conditions that only the device can see (a bounded wait that ran out, an
 *    out-of-range expert id in a plan) are OR-ed into *device_status where an
 *    entry point takes one (see MOE_DEV_* bits); nothing traps.
 *  - Layouts are dense row-major.  E4M3 codes are uint8 bytes; BF16 values are
 *    passed as their uint16 bit patterns.
 */
#ifndef MOE_FP8_H
#define MOE_FP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_NULL = 1,     /* a required pointer is NULL                         */
  MOE_ERR_SHAPE = 2,    /* a size violates the documented constraints         */
  MOE_ERR_ALIGN = 3,    /* a pointer is not 16-byte aligned                   */
  MOE_ERR_CAPACITY = 4, /* plan or workspace buffers too small                */
  MOE_ERR_DTYPE = 5,    /* unsupported id width                               */
  MOE_ERR_DEVICE = 6,   /* pointer not on the current device / not sm_103     */
  MOE_ERR_CUDA = 7,     /* a CUDA runtime/driver call failed                  */
  MOE_ERR_TIMEOUT = 8   /* a synchronous call saw a device wait run out (only
                           moe_selftest_wait_timeout blocks on the device and
                           returns it; asynchronous calls report device
                           timeouts as MOE_DEV_TIMEOUT in *device_status)    */
} moe_status;

/* Bits OR-ed into *device_status by the kernels. */
#define MOE_DEV_TIMEOUT 0x1         /* a bounded pipeline wait ran out (after 1 s, or
                                       2^25 polls); the CTA stopped.  The
                                       results of that call are invalid and its
                                       workspace may hold stale sums: zero it
                                       again (moe_workspace_init) before reuse */
#define MOE_DEV_BAD_EXPERT 0x2      /* a plan block named an expert outside [0, E) other than -1 */
#define MOE_DEV_BAD_SCALE 0x4       /* MOE_SCALES_UE8M0: an activation or weight block scale
                                       the gate/up GEMM read is not +0 or a normal power of
                                       two (the call's results are invalid)                */

/* Human-readable name of a status code (static string). */
const char* moe_status_string(int status);

/* ------------------------------------------------------------------------
 * Routing plan (the moe_align_block_size plan; PR #4287 commit summary and
 * "Public contract and review fixes").
 *
 * Route r = t * top_k + j sends token t to expert topk_ids[t, j].  The plan
 * lists, expert by expert in ascending order, the route indices r of each
 * expert in ascending order, padded with the sentinel R = M * top_k up to a
 * multiple of block_m.  expert_ids[b] is the expert of block b and
 * *num_tokens_post_padded = P, the padded length.  Ids outside [0, E)
 * (including -1, "masked") are dropped.  Slots at and past P (and blocks at
 * and past P / block_m) are NOT written: the caller may leave garbage there.
 * ------------------------------------------------------------------------ */

/* Worst-case (tight) sizes of the plan buffers: sorted_cap =
 * roundup(R + min(E, R) * (block_m - 1), block_m), blocks_cap = sorted_cap /
 * block_m.  Host-only; writes through the two host pointers. */
moe_status moe_plan_capacity(int64_t M, int top_k, int E, int block_m,
                             int64_t* sorted_cap, int64_t* blocks_cap);

/* Device workspace bytes moe_plan needs for these sizes (host-only). */
size_t moe_plan_workspace_size(int64_t M, int top_k, int E);

/* Build the plan on the device.
 *  topk_ids              [M, top_k] int32 (id_bits 32) or int64 (id_bits 64)
 *  sorted_token_ids      [sorted_cap] int32 out
 *  expert_ids            [blocks_cap] int32 out
 *  num_tokens_post_padded [1] int32 out (device scalar)
 *  workspace             >= moe_plan_workspace_size bytes, any contents
 * Constraints: 1 <= E <= 2048; 8 <= block_m <= 1024, block_m % 8 == 0;
 * sorted_cap and blocks_cap at least the moe_plan_capacity values.
 * Deterministic: the same ids give the same bytes. */
moe_status moe_plan(const void* topk_ids, int id_bits, int64_t M, int top_k, int E,
                    int block_m, int32_t* sorted_token_ids, int64_t sorted_cap,
                    int32_t* expert_ids, int64_t blocks_cap,
                    int32_t* num_tokens_post_padded, void* workspace,
                    size_t workspace_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Offline weight preparation.
 * ------------------------------------------------------------------------ */

/* Gate/up eight-row interleave (PR #4287, "Public contract and review
 * fixes": the gate and up rows of W13 come interleaved in groups of eight).  w13 holds
 * [E, 2I, H] E4M3 codes in the logical layout (gate rows [0, I), up rows
 * [I, 2I)); w13_interleaved receives, per expert, rows 16q..16q+7 = gate rows
 * 8q..8q+7 and rows 16q+8..16q+15 = up rows I+8q..I+8q+7.  Out of place (the
 * two buffers must not overlap).  Scales are NOT interleaved: the forward
 * keeps reading w13_scale in the logical [E, 2I/128, H/128] layout.
 * Constraints: N = 2I, I % 128 == 0, H % 16 == 0, 16-byte aligned pointers. */
moe_status moe_prep_weights(const uint8_t* w13, uint8_t* w13_interleaved,
                            int E, int N, int H, moe_stream_t stream);

/* Power-of-two (UE8M0) block-scale requant, in place (SGLang PR #43556,
 * "Motivation": grouped FP8 GEMMs that take UE8M0 scales need scales that are
 * powers of two).  For every 128x128 block with FP32 scale s > 0:
 * s' = 2^ceil(log2 s) (rounded up) and every code w becomes
 * E4M3_rn_satfinite(f32(decode(w) * f32(s / s'))).  Blocks with s <= 0 or a
 * non-finite s are left unchanged, and so is a scale above 2^127 that is not a
 * power of two (no FP32 power of two lies above it).
 *  w          [E, rows, cols] E4M3 codes, rewritten in place
 *  scale      [E, rows/128, cols/128] FP32, rewritten in place
 *  ue8m0_exp  nullable [E, rows/128, cols/128] uint8 out: log2(s') + 127
 *             clamped to [0, 254]; 0 for blocks left unchanged.
 * Constraints: rows % 128 == 0, cols % 128 == 0. */
moe_status moe_requant_scales_ue8m0(uint8_t* w, float* scale, uint8_t* ue8m0_exp,
                                    int E, int rows, int cols, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Quantisers (the step before the path; PR #4287, "Public contract and
 * review fixes": activations carry one FP32 scale per token and 128 columns,
 * weights one FP32 scale per 128x128 block).  scale = f32(amax / 448);
 * code = E4M3_rn_satfinite(f32(x / scale)) with an IEEE FP32 division; a
 * group whose amax is 0 gets scale 0 and all-zero codes.
 * ------------------------------------------------------------------------ */

/* x [M, H] BF16 bits -> q [M, H] E4M3, scale [M, H/128] FP32.  H % 128 == 0. */
moe_status moe_quantize_act_1x128(const uint16_t* x, int64_t M, int H,
                                  uint8_t* q, float* scale, moe_stream_t stream);

/* The same with power-of-two (UE8M0) group scales, the form a hardware
 * block-scaled MMA consumes: each group's scale amax/448 is rounded up to the
 * smallest power of two not below it (as moe_requant_scales_ue8m0 rounds
 * weight block scales; a scale above 2^127 is kept), so codes stay within
 * +-448 and divide exactly.  Scales are still written as FP32. */
moe_status moe_quantize_act_1x128_ue8m0(const uint16_t* x, int64_t M, int H,
                                        uint8_t* q, float* scale, moe_stream_t stream);

/* w [E, rows, cols] BF16 bits -> q [E, rows, cols] E4M3,
 * scale [E, rows/128, cols/128] FP32.  rows, cols % 128 == 0. */
moe_status moe_quantize_weight_128x128(const uint16_t* w, int64_t E, int rows, int cols,
                                       uint8_t* q, float* scale, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Router (the step before the plan: PR #4287 description, "Related Issues",
 * companion router; the serving traces run the router kernel ahead of the
 * expert kernel).  The pages give no formula; this is the reading:
 *   ids[t, :]     = the top_k largest logits[t, :], equal logits by
 *                   ascending expert index, in that order (exact: only input
 *                   values are compared);
 *   weights[t, j] = exp(l_j - m) / D * routed_scale, m = max_e logits[t, e],
 *                   D = sum of exp(l_i - m) over the selection (renormalize
 *                   != 0) or over all E experts (renormalize == 0).
 * FP32 arithmetic (expf, IEEE division).  Logits must not be NaN (the
 * selection is then unspecified; nothing is written out of bounds).
 * ------------------------------------------------------------------------ */

#define MOE_LOGITS_F32 0
#define MOE_LOGITS_BF16 1

/* logits [M, E] (MOE_LOGITS_F32: float; MOE_LOGITS_BF16: BF16 bits),
 * row-major, device memory -> topk_ids [M, top_k] (int32 or int64 per
 * id_bits, ready for moe_plan) and topk_weights [M, top_k] FP32, both
 * caller-owned device memory, fully written for every token.
 * 1 <= E <= 2048, 1 <= top_k <= min(E, 32).  Errors: MOE_ERR_DTYPE (dtype,
 * id_bits), MOE_ERR_SHAPE, MOE_ERR_NULL, MOE_ERR_DEVICE; M == 0 is a no-op. */
moe_status moe_route_topk(const void* logits, int logit_dtype, int64_t M, int E, int top_k, float routed_scale,
                          int renormalize, void* topk_ids, int id_bits, float* topk_weights, moe_stream_t stream);

/* Router and plan in one launch, for small problems (decode): the ids and
 * weights moe_route_topk writes, then the plan moe_plan builds from those
 * ids, bit-identical to the two calls in sequence but without the second
 * launch or a round trip through global memory between them (one CTA: a
 * warp per token selects, then the single-CTA plan runs on the ids held in
 * shared memory).  Arguments are those of the two calls; no plan workspace
 * is needed.  Limits: M * top_k <= 1024 and E <= 1024, else MOE_ERR_SHAPE
 * (use the two calls); otherwise the checks and errors of both calls
 * (M == 0 writes an empty plan, P = 0).  Meant for a few tokens: the one
 * CTA routes 32 tokens at a time, so from a few dozen tokens on the two
 * calls, whose router spreads the tokens over many SMs, are faster. */
moe_status moe_route_plan(const void* logits, int logit_dtype, int64_t M, int E, int top_k, float routed_scale,
                          int renormalize, void* topk_ids, int id_bits, float* topk_weights, int block_m,
                          int32_t* sorted_token_ids, int64_t sorted_cap, int32_t* expert_ids, int64_t blocks_cap,
                          int32_t* num_tokens_post_padded, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * The fused forward (PR #4287 commit summary and "Public contract and review
 * fixes"; post-dot scale application, "Final W8 kernel performance (v46)").
 *
 * For every plan block b < P / block_m whose expert e = expert_ids[b] is in
 * [0, E), and every slot whose route id r = sorted_token_ids[slot] < R, with
 * token t = r / top_k:
 *   g|u[n] = sum_kb f32(dot128(a[t], w13[e, n])) * a_scale[t, kb] * w13_scale[e, n/128, kb]
 *   h[i]   = silu(gate[i]) * up[i]
 *   q, s   = per-128-column E4M3 requant of h (scale amax/448; zero -> 0)
 *   y[c]   = sum_ib f32(dot128(q, w2[e, c])) * s[ib] * w2_scale[e, c/128, ib]
 *   out[t, c] += y[c] * topk_weights[t, j] * routed_scale
 * Each route's contribution y * w is rounded to BF16 once; a token's
 * contributions are added in route order to f32(out) in FP32 and `out` is
 * rounded to BF16 once per call: out = bf16_rn(f32(out) + sum_j c_j).  (The
 * pages' kernel reduce-adds every contribution into BF16 `out`, one rounding
 * per add.)  Blocks past P exit untouched; pad slots (id >= R) and routes
 * the plan does not hold contribute nothing.
 * ------------------------------------------------------------------------ */
typedef struct moe_fwd_args {
  const uint8_t* a;                        /* [M, H] E4M3 activations                       */
  const float* a_scale;                    /* [M, H/128] FP32 per-token group scales        */
  const uint8_t* w13;                      /* [E, 2I, H] E4M3, interleaved by moe_prep_weights */
  const float* w13_scale;                  /* [E, 2I/128, H/128] FP32, LOGICAL row blocks   */
  const uint8_t* w2;                       /* [E, H, I] E4M3                                */
  const float* w2_scale;                   /* [E, H/128, I/128] FP32                        */
  const float* topk_weights;               /* [M, top_k] FP32 route weights                 */
  const int32_t* sorted_token_ids;         /* [sorted_cap] plan (moe_plan)                  */
  const int32_t* expert_ids;               /* [blocks_cap] plan                             */
  const int32_t* num_tokens_post_padded;   /* [1] device scalar P; never read on the host   */
  uint16_t* out;                           /* [M, H] BF16 bits, accumulated in place        */
  void* workspace;                         /* moe_forward_workspace_size bytes, zeroed once */
  int32_t* device_status;                  /* nullable [1]: MOE_DEV_* bits are OR-ed in     */
  uint8_t* debug_q_inter;                  /* nullable [sorted_cap, I]: intermediate codes  */
  float* debug_s_inter;                    /* nullable [sorted_cap, I/128]: their scales    */
  int64_t M;                               /* tokens                                        */
  int64_t sorted_cap;                      /* length of sorted_token_ids                    */
  int64_t blocks_cap;                      /* length of expert_ids                          */
  size_t workspace_bytes;
  int32_t H;                               /* hidden size (K of the gate/up GEMM)           */
  int32_t I;                               /* intermediate size (gate/up width N = 2I)      */
  int32_t E;                               /* experts                                       */
  int32_t top_k;
  int32_t block_m;
  float routed_scale;                      /* routed scaling factor (1.0 = none)            */
  void* const* profile_events;             /* nullable: 5 cudaEvent_t handles, recorded on
                                              `stream` before the staging kernel, after it,
                                              after the gate/up kernel, after the down kernel
                                              and after the combine kernel (per-kernel
                                              timing; events between the launches keep them
                                              from overlapping; no effect if NULL).  On the
                                              vector path the staging and combine intervals
                                              are empty: its two kernels are timed as the
                                              gate/up and down intervals                     */
  int32_t tile_mode;                       /* MOE_TILE_*: how the GEMM tiles map to CTAs    */
  int32_t scale_mode;                      /* MOE_SCALES_*: how the block scales are applied */
} moe_fwd_args;

/* tile_mode values.  Every mode computes the same result (up to FP32
 * summation order).
 *   MOE_TILE_AUTO   the library chooses: the vector path for sparse plans
 *                   (M * top_k <= 32 routes, where it is supported), else
 *                   one CTA per tile.
 *   MOE_TILE_SINGLE one CTA per 128-row tile (cta_group::1 MMAs).
 *   MOE_TILE_PAIR   two CTAs of a cluster per pair of plan blocks of one
 *                   expert (cta_group::2, M = 256): each CTA streams half of
 *                   the weight tile.  Used where the plan qualifies (activation
 *                   rows copied into plan order and at most 1024 plan blocks),
 *                   otherwise the forward falls back to MOE_TILE_SINGLE.
 *   MOE_TILE_VECTOR the vector path for decode-sized plans: the two
 *                   projections as matrix-vector products on the CUDA cores
 *                   (two launches, no staging or combine launch; each
 *                   route's contributions are added to f32(out) in FP32
 *                   without a BF16 rounding of their own).  Supported for
 *                   M * top_k <= 1024, M <= 64 and I <= 1024; otherwise this
 *                   mode returns MOE_ERR_SHAPE.  A plan that holds one route
 *                   in two slots is malformed; this path counts the route at
 *                   its first slot.
 * Any other value returns MOE_ERR_SHAPE. */
#define MOE_TILE_AUTO 0
#define MOE_TILE_SINGLE 1
#define MOE_TILE_PAIR 2
#define MOE_TILE_VECTOR 3

/* scale_mode values (SGLang PR #43556, "Motivation" and "Modifications":
 * block scales requantised to powers of two, the UE8M0 form that grouped
 * FP8 GEMMs with hardware block scaling consume).
 *   MOE_SCALES_FP32  (0, default) any FP32 block scales: every 128-wide K
 *                    slice's partial sum is promoted in FP32 by the
 *                    epilogue (acc += dot * a_scale * w_scale).
 *   MOE_SCALES_UE8M0 the caller guarantees that every activation scale
 *                    (a_scale) and W13 block scale is +0 or a normal power
 *                    of two, as moe_quantize_act_1x128_ue8m0 and
 *                    moe_requant_scales_ue8m0 produce.  The gate/up GEMM on
 *                    the tensor-core tiles then hands the scales to the
 *                    tensor core as UE8M0 scale factors
 *                    (tcgen05.mma kind::mxf8f6f4.block_scale) and each tile
 *                    accumulates over all of K in tensor memory, with no
 *                    per-slice promotion; a scale that is not a power of two
 *                    sets MOE_DEV_BAD_SCALE.  A zero scale becomes the
 *                    smallest UE8M0 scale, 2^-127: its block adds at most
 *                    about 2^-100 of the FP32 values it meets, and an expert
 *                    whose W13 scales are all zero still yields exactly zero
 *                    after SwiGLU (the products underflow).  The down GEMM,
 *                    whose intermediate scales are amax/448, and the vector
 *                    path keep the FP32 promotion.  Runs on single CTAs
 *                    (MOE_TILE_PAIR then falls back to MOE_TILE_SINGLE).
 * Any other value returns MOE_ERR_SHAPE. */
#define MOE_SCALES_FP32 0
#define MOE_SCALES_UE8M0 1

/* Workspace bytes the forward needs (host-only; 0 for invalid sizes).  The
 * workspace holds the BF16 route contributions [M * top_k, H], for problems
 * the vector path supports its FP32 SwiGLU output [M * top_k, I], the requantised
 * intermediate (sorted_cap x I codes and sorted_cap x I/128 scales) and, for
 * well-filled plans (M * top_k >= 8 * min(E, M * top_k)), the activation rows
 * and scales copied into plan order (sorted_cap x H bytes and
 * sorted_cap x H/128 scales). */
size_t moe_forward_workspace_size(int64_t M, int H, int I, int E, int top_k, int block_m,
                                  int64_t sorted_cap);

/* Zero a forward workspace (async).  A workspace must be zeroed once before
 * its first forward for a given set of sizes (M, H, I, E, top_k, block_m,
 * sorted_cap); every forward with those sizes leaves it ready for the next:
 * split-K tickets and partial sums go back to zero, and each route's flag
 * holds the stamp of the last forward whose plan held it, against a stamp
 * counter the gate/up kernel advances once per forward (so a replayed CUDA
 * graph stays correct).  A forward that set MOE_DEV_TIMEOUT may leave it
 * dirty: zero it again before the next forward.  The layout depends on the sizes, so before a
 * forward with other sizes zero the workspace again (or use another one).
 * The BF16 route contributions, the first M * top_k * H * 2 bytes, are
 * scratch written before they are read.  Two forwards that share a
 * workspace must not run concurrently. */
moe_status moe_workspace_init(void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* Run the forward.  Constraints: H % 128 == 0; I % 128 == 0 (so 2I % 256 ==
 * 0); 1 <= top_k <= 64; 8 <= block_m <= 128, block_m % 8 == 0; sorted_cap >= blocks_cap *
 * block_m; blocks_cap >= 1; a, w13, w2 and the workspace 16-byte aligned; all
 * pointers on the current device, which must be sm_103 (GB300: the library
 * is built for sm_103a only). */
moe_status moe_fp8_block_scale_forward(const moe_fwd_args* args, moe_stream_t stream);

/* Failure-detection self-test (the pages have no counterpart: it exercises
 * this library's bounded waits, the GB300 replacement for a hang).  Launches
 * one CTA on `stream` whose first warp waits, through the GEMM pipelines'
 * own bounded mbarrier wait, on a barrier that nothing arrives at and gives
 * up after limit_us microseconds; its second warp waits on another such
 * barrier with the pipelines' normal one-second limit and must stop as soon
 * as the first raises the CTA's abort flag.  The CTA then ORs
 * MOE_DEV_TIMEOUT into *device_status as a GEMM CTA whose wait ran out does,
 * and writes how long each warp waited, in nanoseconds, to elapsed_ns[0]
 * and elapsed_ns[1] (0 for a wait that completed).  Nothing traps or
 * faults: the context stays usable.
 *  device_status  [1] int32, device memory, caller-owned (OR-ed into)
 *  elapsed_ns     [2] uint64, device memory, caller-owned (written)
 * Blocks until the kernel has finished (not capturable in a CUDA graph),
 * then returns MOE_ERR_TIMEOUT if *device_status holds MOE_DEV_TIMEOUT (the
 * expected outcome), MOE_OK otherwise.  1 <= limit_us <= 1000000, else
 * MOE_ERR_SHAPE. */
moe_status moe_selftest_wait_timeout(uint32_t limit_us, int32_t* device_status, uint64_t* elapsed_ns,
                                     moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Bounds-checking build.  A library compiled with -DMOE_DEBUG_BOUNDS
 * (libmoe_fp8_debug.so from the package's build script) checks, before each
 * access, every global index its kernels derive from data or tiling (plan
 * entries, route, token, slot and expert ids, workspace offsets) and every
 * tensor-copy coordinate (in range, and the innermost one 16-byte aligned).
 * A failed check is counted in a device-side record, the access is skipped
 * (a tensor copy is moved to coordinate 0 so its barrier still completes)
 * and the kernel carries on; nothing traps.  Results are then unspecified,
 * but the context stays usable.  The normal build compiles the checks away.
 * ------------------------------------------------------------------------ */
/* 1 in the bounds-checking build, 0 otherwise. */
int moe_debug_bounds_enabled(void);
/* Waits for the device (cudaDeviceSynchronize), then writes to *failures the
 * number of failed checks since the library loaded or the last reset, and
 * to *first_file / *first_line (both nullable) the source file (a static
 * string, NULL when there was none) and line of the first failure in the
 * first file that has one.  reset != 0 zeroes the records afterwards.  In the
 * normal build *failures = 0.  MOE_ERR_NULL if failures is NULL, MOE_ERR_CUDA
 * if the synchronisation or a read fails. */
moe_status moe_debug_bounds_read(uint64_t* failures, const char** first_file, int32_t* first_line, int reset);
/* Self-test of the checks: one thread reads data[probe] into *out.  In the
 * bounds-checking build a probe outside [0, n) fails the kernel's check,
 * which counts it and writes -1 instead of reading; in the normal build such
 * a probe is refused on the host (MOE_ERR_SHAPE) and nothing is launched.
 *  data  [n] int32, device memory;  out  [1] int32, device memory (written)
 * n >= 1, else MOE_ERR_SHAPE; asynchronous on `stream`. */
moe_status moe_debug_bounds_selftest(const int32_t* data, int n, int probe, int32_t* out, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Allocation-free forward.  The pages have no counterpart to this entry
 * point; it exists for callers that cannot call cudaMalloc: engines that
 * hand all of device memory to their own pool at start-up and forbid any
 * later allocation, plug-ins that reach the GPU only through this C ABI and
 * own no allocator, and latency-critical loops where an allocation could
 * synchronise the device.
 *
 * Same arguments and results as moe_fp8_block_scale_forward, except that
 * args->workspace and args->workspace_bytes are ignored: the scratch is a
 * file-scope static device array of moe_noalloc_scratch_bytes() bytes
 * (32 MiB) that every GPU loading the library holds until the process exits.
 * Problems whose moe_forward_workspace_size exceeds it are rejected with
 * MOE_ERR_CAPACITY before anything is launched (decode-sized problems fit;
 * prefill-sized ones do not).  The caller still passes every input and the
 * output.  Each call zeroes the part of the array it uses (async, on
 * `stream`) before the forward.  All calls share the one array, so calls
 * whose work overlaps on the GPU (different streams, or different host
 * threads) race and corrupt each other's results: serialise them.  The first
 * call on a device looks up the array's device address for that device (a
 * host-side set-up step); make that first call before any stream capture.
 * Allocates nothing: no cudaMalloc/cudaFree and no allocating library call.
 * ------------------------------------------------------------------------ */
/* The address looked up on a device's first call is kept for the life of the
 * process: do not use this entry point on a device after cudaDeviceReset (or
 * anything else that destroys and recreates its primary context). */
size_t moe_noalloc_scratch_bytes(void);
moe_status moe_fp8_block_scale_forward_noalloc(const moe_fwd_args* args, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FP8_H */
