// Tensor-core projections of the E2M1-K32 weight x FP8 activation path
// (w4a8_tc.cu), launched by moe_w4a8_forward (w4a8.cu).
#pragma once

#include "common.cuh"

namespace moe {

struct W4GemmParams {
  const int32_t* sorted_ids;       // plan
  const int32_t* expert_ids;
  const int32_t* num_post_padded;
  const float* a_scale;            // gate/up: [M] activation row scales
  const float* s_inter;            // down: [R] intermediate row scales
  const float* topk_w;             // down: [R] route weights
  float* h;                        // gate/up out: [R, I] silu(g) * u by route id
  float* y;                        // down out: [R, H] y * s * w by route id
  int32_t* status;                 // nullable
  int64_t nblocks;                 // plan blocks the grid walks
  int64_t sorted_cap;              // entries of sorted_ids
  int64_t rows_total;              // rows of the gathered tensor (set by the launcher)
  int R, top_k, block_m, E, H, I;
  int up;                          // 1: gate/up projection, 0: down projection
  int ntw;                         // weight tiles per plan block: I / 64 (gate/up) or H / 128 (down)
  int w_rows;                      // weight rows per expert: 2I or H
  int nkb;                         // K / 128 (set by the launcher)
  int group;                       // plan blocks of one expert per tile, at most (set by the launcher)
  float routed_scale;
};

struct W4GemmTensors {
  const uint8_t* w;                // packed E2M1 weights [w_total_rows, k / 2]
  const float* w_scale;            // [w_total_rows, k / 32]
  uint64_t w_total_rows;           // E * (2I or H)
  const uint8_t* rows;             // E4M3 rows gathered by the plan: a [M, H] or q [R, I]
  uint64_t rows_total;             // M or R
  uint64_t k;                      // H or I
};

// The tensor-core projections need K extents that are multiples of 128 (the
// copy engine's 4-bit boxes), plan blocks of at most 64 rows, packed weights
// 32-byte aligned and scales 16-byte aligned.
bool w4a8_tc_supported(int H, int I, int block_m, const void* w13, const void* w2, const void* w13_scale,
                       const void* w2_scale);

moe_status launch_w4a8_tc_gemm(const W4GemmTensors& t, W4GemmParams p, int sms, cudaStream_t stream);

}  // namespace moe
