// The router's per-token selection (router.cu), shared with the fused
// router + plan launch (plan.cu).
//
// Reading (the pages give no formula; the oracle follows the same one):
//   ids     = the top_k largest logits of the token, equal logits by
//             ascending expert index, listed in that order;
//   weights = exp(l_j - m) / D, m = the token's largest logit,
//             D = sum over the selection (renormalize) or over all E experts,
//             times routed_scale.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kRouteMaxE = 2048;
constexpr int kRouteMaxTopK = 32;

__device__ __forceinline__ float load_logit(const void* logits, int dtype, int64_t i) {
  if (dtype == 0) return static_cast<const float*>(logits)[i];
  const uint32_t bits = static_cast<const uint16_t*>(logits)[i];
  return __uint_as_float(bits << 16);  // BF16 -> FP32 is exact
}

// One warp routes token t (every lane must call it).  Lane l holds the
// logits of experts l, l+32, ... in registers; each of the top_k rounds takes
// a lane-local best untaken (value, index) and a warp argmax over (value
// descending, index ascending), so the selection compares input values only
// and is exact.  On return lane j < top_k holds the j-th selection's expert
// id and route weight.
template <int kPer>  // logits per lane: E <= 32 * kPer
__device__ __forceinline__ void route_token(const void* logits, int dtype, int64_t t, int E, int top_k,
                                            float routed_scale, int renormalize, int& out_id, float& out_w) {
  const int lane = threadIdx.x % 32;
  float v[kPer];
  uint64_t taken = 0;  // bit i: expert lane + 32 i already selected, or past E
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? load_logit(logits, dtype, t * E + e) : 0.f;
    if (e >= E) taken |= uint64_t(1) << i;
  }
  constexpr int kNone = 0x7fffffff;
  float my_l = 0.f;  // lane j < top_k: logit and expert of the j-th selection
  int my_id = 0;
  for (int j = 0; j < top_k; ++j) {
    float bv = 0.f;
    int bi = kNone;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = lane + 32 * i;
      if (!((taken >> i) & 1u) && (bi == kNone || v[i] > bv || (v[i] == bv && e < bi))) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (oi != kNone && (bi == kNone || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == (bi & 31)) taken |= uint64_t(1) << (bi >> 5);
    if (lane == j) {
      my_l = bv;
      my_id = bi;
    }
  }
  const float m = __shfl_sync(0xffffffffu, my_l, 0);  // the largest logit
  const float num = lane < top_k ? expf(my_l - m) : 0.f;
  float part = num;
  if (!renormalize) {
    part = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (lane + 32 * i < E) part += expf(v[i] - m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  out_id = my_id;
  out_w = num / part * routed_scale;
}

}  // namespace moe
