// moe_route_topk: router logits -> top-k expert ids and route weights, the
// companion step before the routing plan (FlashInfer PR #4287 description,
// "Related Issues": companion router; the serving traces run
// kernel_alpha_moe_fused_router ahead of the expert kernel).  The pages give
// no formula; the reading implemented here (and in the oracle) is:
//   ids     = the top_k largest logits of the token, equal logits by
//             ascending expert index, listed in that order;
//   weights = exp(l_j - m) / D, m = the token's largest logit,
//             D = sum over the selection (renormalize) or over all E experts,
//             times routed_scale.
//
// One warp per token.  Lane l holds the logits of experts l, l+32, ... in
// registers; each of the top_k rounds takes a lane-local best untaken
// (value, index) and a warp argmax over (value descending, index ascending),
// so the selection compares input values only and is exact.
#include "common.cuh"
#include "router.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 8;

template <int kPer>  // logits per lane: E <= 32 * kPer
__global__ void __launch_bounds__(32 * kRouteWarps) route_topk_kernel(const void* logits, int dtype, int64_t M,
                                                                      int E, int top_k, float routed_scale,
                                                                      int renormalize, void* ids, int id_bits,
                                                                      float* weights) {
  // launched with programmatic stream serialization: wait for the
  // predecessor (it may still read the previous ids), then release the
  // dependents (the plan waits for this grid in turn)
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x % 32;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kRouteWarps + threadIdx.x / 32;
  if (t >= M) return;  // whole warp
  int id;
  float w;
  route_token<kPer>(logits, dtype, t, E, top_k, routed_scale, renormalize, id, w);
  if (lane < top_k) {
    const int64_t o = t * top_k + lane;
    weights[o] = w;
    if (id_bits == 64)
      static_cast<int64_t*>(ids)[o] = id;
    else
      static_cast<int32_t*>(ids)[o] = id;
  }
}

template <int kPer>
cudaError_t launch_route(const void* logits, int dtype, int64_t M, int E, int top_k, float routed_scale,
                         int renormalize, void* ids, int id_bits, float* weights, cudaStream_t stream) {
  const int64_t grid = ceil_div(M, static_cast<int64_t>(kRouteWarps));
  return launch_pdl(route_topk_kernel<kPer>, dim3(static_cast<unsigned>(grid)), dim3(32 * kRouteWarps), 0, stream, 1,
                    logits, dtype, M, E, top_k, routed_scale, renormalize, ids, id_bits, weights);
}

}  // namespace
}  // namespace moe

extern "C" {

moe_status moe_route_topk(const void* logits, int logit_dtype, int64_t M, int E, int top_k, float routed_scale,
                          int renormalize, void* topk_ids, int id_bits, float* topk_weights, moe_stream_t stream) {
  using namespace moe;
  if (logit_dtype != MOE_LOGITS_F32 && logit_dtype != MOE_LOGITS_BF16) return MOE_ERR_DTYPE;
  if (id_bits != 32 && id_bits != 64) return MOE_ERR_DTYPE;
  if (M < 0 || E < 1 || E > kRouteMaxE || top_k < 1 || top_k > kRouteMaxTopK || top_k > E) return MOE_ERR_SHAPE;
  if (M * static_cast<int64_t>(E) >= (int64_t(1) << 40)) return MOE_ERR_SHAPE;
  if (M == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_weights) return MOE_ERR_NULL;
  DeviceInfo dev;
  if (current_device(&dev) != MOE_OK) return MOE_ERR_CUDA;
  if (!on_device(logits, dev.device) || !on_device(topk_ids, dev.device) || !on_device(topk_weights, dev.device))
    return MOE_ERR_DEVICE;
  cudaError_t err;
  const int per = static_cast<int>(ceil_div(static_cast<int64_t>(E), int64_t(32)));
  if (per <= 1)
    err = launch_route<1>(logits, logit_dtype, M, E, top_k, routed_scale, renormalize, topk_ids, id_bits, topk_weights, stream);
  else if (per <= 2)
    err = launch_route<2>(logits, logit_dtype, M, E, top_k, routed_scale, renormalize, topk_ids, id_bits, topk_weights, stream);
  else if (per <= 4)
    err = launch_route<4>(logits, logit_dtype, M, E, top_k, routed_scale, renormalize, topk_ids, id_bits, topk_weights, stream);
  else if (per <= 8)
    err = launch_route<8>(logits, logit_dtype, M, E, top_k, routed_scale, renormalize, topk_ids, id_bits, topk_weights, stream);
  else if (per <= 16)
    err = launch_route<16>(logits, logit_dtype, M, E, top_k, routed_scale, renormalize, topk_ids, id_bits, topk_weights, stream);
  else if (per <= 32)
    err = launch_route<32>(logits, logit_dtype, M, E, top_k, routed_scale, renormalize, topk_ids, id_bits, topk_weights, stream);
  else
    err = launch_route<64>(logits, logit_dtype, M, E, top_k, routed_scale, renormalize, topk_ids, id_bits, topk_weights, stream);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"

MOE_BOUNDS_TU()
