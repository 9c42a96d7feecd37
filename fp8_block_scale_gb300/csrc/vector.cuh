// The vector path of the forward (vector.cu): parameters and launcher.
#pragma once

#include "common.cuh"

namespace moe {

// Largest plans the vector path takes: routes and tokens (the down kernel
// keeps the route list and each token's running sums in shared memory).
constexpr int kVecMaxRoutes = 1024;
constexpr int kVecMaxTokens = 64;

struct VecUpParams {
  const uint8_t* a;                 // [M, H] E4M3
  const float* a_scale;             // [M, H/128]
  const uint8_t* w13;               // [E, 2I, H] interleaved E4M3
  const float* w13_scale;           // [E, 2I/128, H/128] logical row blocks
  const uint8_t* w2;                // [E, H, I]: the expert's rows are prefetched into L2
  const int32_t* sorted_ids;
  const int32_t* expert_ids;
  const int32_t* num_post_padded;
  float* h;                         // [R, I] silu(gate) * up by route id (workspace)
  int32_t* status;
  int64_t nblocks;                  // plan blocks that can hold work
  int R, top_k, block_m, E, H, I;
};

struct VecDownParams {
  const float* h;                   // [R, I] from the gate/up kernel
  const uint8_t* w2;                // [E, H, I] E4M3
  const float* w2_scale;            // [E, H/128, I/128]
  const float* topk_w;              // [M, top_k]
  const int32_t* sorted_ids;
  const int32_t* expert_ids;
  const int32_t* num_post_padded;
  uint16_t* out;                    // [M, H] BF16, accumulated
  uint8_t* dbg_q;                   // nullable [sorted_cap, I]
  float* dbg_s;                     // nullable [sorted_cap, I/128]
  int64_t nblocks;
  int R, top_k, block_m, E, H, I;
  float routed_scale;
};

// True if the vector path can run this problem.
bool vector_path_supported(int64_t M, int64_t R, int H, int I);

// Launches both kernels on `stream`; records ev[1..3] when ev is non-null
// (ev[1] right away: the path has no staging launch).
moe_status launch_vector_path(const VecUpParams& up, const VecDownParams& dn, cudaStream_t stream,
                              cudaEvent_t const* ev);

}  // namespace moe
