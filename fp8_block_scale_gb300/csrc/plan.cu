// moe_plan: the moe_align_block_size routing plan on the device (FlashInfer
// PR #4287 commit summary: routes sorted per expert and padded to block_m;
// "Public contract and review fixes": sorted_token_ids holds
// expert_ids.numel() * block_m slots).
//
// Deterministic counting sort.  Up to kSmallRoutes routes (decode) it runs
// as one CTA in one launch (plan_small_kernel); above that in three:
//   1. rank:    each CTA takes a chunk of kChunk routes, computes every route's
//               stable rank among same-expert routes of its chunk (warp
//               match + per-warp histograms in shared memory) and the chunk's
//               per-expert counts.
//   2. scan:    one CTA: a warp per expert scans that expert's per-chunk
//               counts into bases, then the experts' padded lengths are
//               scanned; writes expert_ids, the pad sentinels and P.
//   3. scatter: sorted_token_ids[base(chunk, e) + rank] = r.
// No inter-CTA waits; the same ids always give the same bytes.
#include "common.cuh"
#include "router.cuh"

namespace moe {
namespace {

constexpr int kChunk = 512;  // routes per CTA in the rank/scatter launches (one per thread)
constexpr int kChunkWarps = kChunk / 32;
constexpr int kScanThreads = 1024;
constexpr int kMaxExperts = 2048;
constexpr int kSmallRoutes = kScanThreads;  // one route per thread of the single-CTA plan
constexpr int kSmallMaxExperts = 1024;      // its per-warp histograms: 32 x E ints of shared memory
constexpr int kScanBatch = 8;               // chunk counts in flight per lane and expert

struct PlanWs {
  int32_t* counts;  // [E, chunks]: per-chunk counts, then bases inside the expert
  int32_t* rank;    // [R] stable rank of each route inside its chunk (or -1)
  int32_t* seg;     // [E] segment start of each expert
  int nchunks;
  int64_t sorted_cap;  // entries of sorted_token_ids
  int64_t blocks_cap;  // entries of expert_ids
};

__device__ __forceinline__ int load_id(const void* ids, int id_bits, int64_t r, int E) {
  int64_t v = id_bits == 64 ? static_cast<const int64_t*>(ids)[r] : static_cast<const int32_t*>(ids)[r];
  return (v >= 0 && v < E) ? static_cast<int>(v) : -1;
}

// Every plan kernel is launched with programmatic stream serialization: it
// waits for its predecessor (which may have produced the ids, or may still
// read the previous plan) before touching memory, then lets its own
// dependents begin launching.
__device__ __forceinline__ void plan_enter() {
  pdl_wait();
  pdl_launch_dependents();
}

__global__ void __launch_bounds__(kChunk) plan_rank_kernel(const void* ids, int id_bits, int64_t R, int E, PlanWs ws) {
  extern __shared__ int32_t wh[];  // [kChunkWarps][E]
  plan_enter();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int i = threadIdx.x; i < kChunkWarps * E; i += blockDim.x) wh[i] = 0;
  __syncthreads();
  const int64_t r = static_cast<int64_t>(blockIdx.x) * kChunk + threadIdx.x;
  const int e = r < R ? load_id(ids, id_bits, r, E) : -1;
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const unsigned below = peers & ((1u << lane) - 1u);
  const int in_warp = __popc(below);
  if (e >= 0 && below == 0) wh[warp * E + e] = __popc(peers);
  __syncthreads();
  // exclusive scan over warps, per expert; chunk total goes to counts
  for (int x = threadIdx.x; x < E; x += blockDim.x) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < kChunkWarps; ++w) {
      const int v = wh[w * E + x];
      wh[w * E + x] = run;
      run += v;
    }
    ws.counts[static_cast<int64_t>(x) * ws.nchunks + blockIdx.x] = run;
  }
  __syncthreads();
  if (r < R) ws.rank[r] = e >= 0 ? wh[warp * E + e] + in_warp : -1;
}

// Block-wide exclusive scan of one int per thread (kScanThreads threads).
__device__ int block_exclusive_scan(int v, int* total, int* smem /* 32 ints */) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) smem[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = smem[lane];
    int winc = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, winc, o);
      if (lane >= o) winc += n;
    }
    smem[lane] = winc - w;  // exclusive prefix of warp sums
    if (lane == 31) smem[32] = winc;
  }
  __syncthreads();
  const int res = smem[warp] + inc - v;
  *total = smem[32];
  __syncthreads();
  return res;
}

// Pad sentinels (R) after each expert's routes and the expert of each of its
// blocks: a warp per expert, lanes over the slots.
__device__ void fill_pads(int E, int block_m, int64_t R, const int* totals, const int* seg, int32_t* sorted_ids,
                          int32_t* expert_ids, int64_t sorted_cap, int64_t blocks_cap) {
  const int lane = threadIdx.x % 32;
  for (int e = threadIdx.x / 32; e < E; e += blockDim.x / 32) {
    const int tot = totals[e];
    if (tot == 0) continue;  // no routes: no slots, no blocks
    const int st = seg[e];
    const int end = st + (tot + block_m - 1) / block_m * block_m;
    for (int q = st + tot + lane; q < end; q += 32)
      if (MOE_IN_BOUNDS(q >= 0 && q < sorted_cap)) sorted_ids[q] = static_cast<int32_t>(R);
    for (int b = st / block_m + lane; b < end / block_m; b += 32)
      if (MOE_IN_BOUNDS(b >= 0 && b < blocks_cap)) expert_ids[b] = e;
  }
}

__global__ void __launch_bounds__(kScanThreads) plan_scan_kernel(int64_t R, int E, int block_m, int nchunks, PlanWs ws,
                                                                  int32_t* sorted_ids, int32_t* expert_ids,
                                                                  int32_t* num_post_padded) {
  __shared__ int scan_smem[33];
  __shared__ int totals[kMaxExperts];
  __shared__ int seg[kMaxExperts];
  plan_enter();
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  // 1. one warp per expert: exclusive scan of its chunk counts (bases inside
  //    the expert) and the expert's total.  A warp takes two experts at a
  //    time and loads up to kScanBatch x 32 counts of each before scanning,
  //    so the loads overlap instead of paying one latency per 32 chunks.
  constexpr int kWarps = kScanThreads / 32;
  for (int e0 = warp; e0 < E; e0 += 2 * kWarps) {
    const int ee[2] = {e0, e0 + kWarps};
    int carry[2] = {0, 0};
    for (int c0 = 0; c0 < nchunks; c0 += 32 * kScanBatch) {
      int v[2][kScanBatch];
      // batches of this round that hold chunks (warp-uniform)
      const int nbat = min(kScanBatch, (nchunks - c0 + 31) / 32);
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int32_t* row = ws.counts + static_cast<int64_t>(ee[x] < E ? ee[x] : 0) * nchunks;
#pragma unroll
        for (int j = 0; j < kScanBatch; ++j) {
          const int c = c0 + 32 * j + lane;
          v[x][j] = (j < nbat && ee[x] < E && c < nchunks) ? row[c] : 0;
        }
      }
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (ee[x] >= E) continue;
        int32_t* row = ws.counts + static_cast<int64_t>(ee[x]) * nchunks;
#pragma unroll
        for (int j = 0; j < kScanBatch; ++j) {
          if (j >= nbat) break;
          const int c = c0 + 32 * j + lane;
          int inc = v[x][j];
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += n;
          }
          if (c < nchunks) row[c] = carry[x] + inc - v[x][j];
          carry[x] += __shfl_sync(0xffffffffu, inc, 31);
        }
      }
    }
#pragma unroll
    for (int x = 0; x < 2; ++x)
      if (lane == 0 && ee[x] < E) totals[ee[x]] = carry[x];
  }
  __syncthreads();
  // 2. pad every expert to block_m and scan the experts
  constexpr int kPer = kMaxExperts / kScanThreads;  // experts per thread (2)
  int total[kPer], padded[kPer];
  int mine = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = threadIdx.x * kPer + i;
    total[i] = e < E ? totals[e] : 0;
    padded[i] = (total[i] + block_m - 1) / block_m * block_m;
    mine += padded[i];
  }
  int P = 0;
  int start = block_exclusive_scan(mine, &P, scan_smem);
  // 3. segment starts; then a warp per expert writes its pad sentinels and
  //    block experts (one slot per lane); P
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = threadIdx.x * kPer + i;
    if (e < E) {
      ws.seg[e] = start;
      seg[e] = start;
    }
    start += padded[i];
  }
  __syncthreads();
  fill_pads(E, block_m, R, totals, seg, sorted_ids, expert_ids, ws.sorted_cap, ws.blocks_cap);
  if (threadIdx.x == 0) *num_post_padded = P;
}

__global__ void __launch_bounds__(kChunk) plan_scatter_kernel(const void* ids, int id_bits, int64_t R, int E, PlanWs ws,
                                                               int32_t* sorted_ids) {
  plan_enter();
  const int64_t r = static_cast<int64_t>(blockIdx.x) * kChunk + threadIdx.x;
  if (r >= R) return;
  const int rk = ws.rank[r];
  if (rk < 0) return;
  const int e = load_id(ids, id_bits, r, E);
  const int base = ws.seg[e] + ws.counts[static_cast<int64_t>(e) * ws.nchunks + blockIdx.x];
  if (MOE_IN_BOUNDS(base + rk >= 0 && base + rk < ws.sorted_cap)) sorted_ids[base + rk] = static_cast<int32_t>(r);
}

// The single-CTA plan: thread r < R holds its route's expert e (-1 for a
// route the plan drops).  wh is [32][E] ints of dynamic shared memory.
__device__ __forceinline__ void plan_small_body(int e, int64_t R, int E, int block_m, int32_t* sorted_ids,
                                                int32_t* expert_ids, int32_t* num_post_padded, int64_t sorted_cap,
                                                int64_t blocks_cap, int32_t* wh, int* scan_smem, int* totals,
                                                int* seg) {
  constexpr int kWarps = kScanThreads / 32;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int r = threadIdx.x;
  for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x) wh[i] = 0;
  __syncthreads();
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const unsigned below = peers & ((1u << lane) - 1u);
  const int in_warp = __popc(below);
  if (e >= 0 && below == 0) wh[warp * E + e] = __popc(peers);
  __syncthreads();
  for (int x = threadIdx.x; x < E; x += blockDim.x) {
    int run = 0;
#pragma unroll 8
    for (int w = 0; w < kWarps; ++w) {
      const int v = wh[w * E + x];
      wh[w * E + x] = run;
      run += v;
    }
    totals[x] = run;
  }
  __syncthreads();
  // padded expert lengths, scanned (the same steps as plan_scan_kernel)
  constexpr int kPer = kSmallMaxExperts / kScanThreads;  // 1
  int total[kPer], padded[kPer];
  int mine = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int x = threadIdx.x * kPer + i;
    total[i] = x < E ? totals[x] : 0;
    padded[i] = (total[i] + block_m - 1) / block_m * block_m;
    mine += padded[i];
  }
  int P = 0;
  int start = block_exclusive_scan(mine, &P, scan_smem);
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int x = threadIdx.x * kPer + i;
    if (x < E) seg[x] = start;
    start += padded[i];
  }
  if (threadIdx.x == 0) *num_post_padded = P;
  __syncthreads();
  fill_pads(E, block_m, R, totals, seg, sorted_ids, expert_ids, sorted_cap, blocks_cap);
  if (e >= 0) {
    const int q = seg[e] + wh[warp * E + e] + in_warp;
    if (MOE_IN_BOUNDS(q >= 0 && q < sorted_cap)) sorted_ids[q] = static_cast<int32_t>(r);
  }
}

// The whole plan in one CTA for R <= kSmallRoutes and E <= kSmallMaxExperts:
// one route per thread, ranked by a warp match plus per-warp expert
// histograms, then the padded expert scan and the scatter.  Same bytes as the
// three-launch path (a stable counting sort).
__global__ void __launch_bounds__(kScanThreads) plan_small_kernel(const void* ids, int id_bits, int64_t R, int E,
                                                                   int block_m, int32_t* sorted_ids,
                                                                   int32_t* expert_ids, int32_t* num_post_padded,
                                                                   int64_t sorted_cap, int64_t blocks_cap) {
  extern __shared__ int32_t wh[];  // [32][E]: per-warp counts, then their exclusive prefix over warps
  __shared__ int scan_smem[33];
  __shared__ int totals[kSmallMaxExperts];
  __shared__ int seg[kSmallMaxExperts];
  plan_enter();
  const int r = threadIdx.x;
  const int e = r < R ? load_id(ids, id_bits, r, E) : -1;
  plan_small_body(e, R, E, block_m, sorted_ids, expert_ids, num_post_padded, sorted_cap, blocks_cap, wh, scan_smem,
                  totals, seg);
}

// Router and plan in one CTA (R <= kSmallRoutes, E <= kSmallMaxExperts): a
// warp per token selects its top_k experts exactly as the router kernel does
// and writes the ids and weights, keeping the ids in shared memory; then the
// single-CTA plan runs on them.
template <int kPer>
__global__ void __launch_bounds__(kScanThreads) route_plan_kernel(const void* logits, int dtype, int64_t M, int E,
                                                                   int top_k, float routed_scale, int renormalize,
                                                                   void* ids, int id_bits, float* weights,
                                                                   int block_m, int32_t* sorted_ids,
                                                                   int32_t* expert_ids, int32_t* num_post_padded,
                                                                   int64_t sorted_cap, int64_t blocks_cap) {
  extern __shared__ int32_t wh[];  // [32][E]
  __shared__ int s_e[kSmallRoutes];
  __shared__ int scan_smem[33];
  __shared__ int totals[kSmallMaxExperts];
  __shared__ int seg[kSmallMaxExperts];
  plan_enter();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t R = M * top_k;
  for (int64_t t = warp; t < M; t += kScanThreads / 32) {
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
      if (MOE_IN_BOUNDS(o < kSmallRoutes)) s_e[o] = (id >= 0 && id < E) ? id : -1;
    }
  }
  __syncthreads();
  const int r = threadIdx.x;
  const int e = r < R ? s_e[r] : -1;
  plan_small_body(e, R, E, block_m, sorted_ids, expert_ids, num_post_padded, sorted_cap, blocks_cap, wh, scan_smem,
                  totals, seg);
}

size_t plan_ws_bytes(int64_t R, int E, int64_t* nchunks_out) {
  const int64_t nchunks = ceil_div(R > 0 ? R : 1, kChunk);
  if (nchunks_out) *nchunks_out = nchunks;
  return static_cast<size_t>(round_up(nchunks * E * 4, 256) + round_up(R * 4, 256) + round_up(E * 4, 256));
}

}  // namespace
}  // namespace moe

extern "C" {

size_t moe_plan_workspace_size(int64_t M, int top_k, int E) {
  if (M < 0 || top_k < 1 || E < 1) return 0;
  return moe::plan_ws_bytes(M * top_k, E, nullptr);
}

moe_status moe_plan(const void* topk_ids, int id_bits, int64_t M, int top_k, int E, int block_m,
                    int32_t* sorted_token_ids, int64_t sorted_cap, int32_t* expert_ids, int64_t blocks_cap,
                    int32_t* num_tokens_post_padded, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  using namespace moe;
  if (!sorted_token_ids || !expert_ids || !num_tokens_post_padded || !workspace) return MOE_ERR_NULL;
  if (id_bits != 32 && id_bits != 64) return MOE_ERR_DTYPE;
  if (M < 0 || top_k < 1 || E < 1 || E > kMaxExperts) return MOE_ERR_SHAPE;
  if (block_m < 8 || block_m > 1024 || block_m % 8 != 0) return MOE_ERR_SHAPE;
  const int64_t R = M * top_k;
  if (R >= (int64_t(1) << 31) - 1) return MOE_ERR_SHAPE;
  if (R > 0 && !topk_ids) return MOE_ERR_NULL;
  int64_t need_cap = 0, need_blocks = 0;
  moe_plan_capacity(M, top_k, E, block_m, &need_cap, &need_blocks);
  if (sorted_cap < need_cap || blocks_cap < need_blocks) return MOE_ERR_CAPACITY;
  int64_t nchunks = 0;
  if (workspace_bytes < plan_ws_bytes(R, E, &nchunks)) return MOE_ERR_CAPACITY;
  DeviceInfo dev;
  if (current_device(&dev) != MOE_OK) return MOE_ERR_CUDA;
  if ((R > 0 && !on_device(topk_ids, dev.device)) || !on_device(sorted_token_ids, dev.device) ||
      !on_device(expert_ids, dev.device) || !on_device(num_tokens_post_padded, dev.device) ||
      !on_device(workspace, dev.device))
    return MOE_ERR_DEVICE;

  uint8_t* w = static_cast<uint8_t*>(workspace);
  PlanWs ws;
  ws.counts = reinterpret_cast<int32_t*>(w);
  w += round_up(nchunks * E * 4, 256);
  ws.rank = reinterpret_cast<int32_t*>(w);
  w += round_up(R * 4, 256);
  ws.seg = reinterpret_cast<int32_t*>(w);
  ws.nchunks = static_cast<int>(R > 0 ? nchunks : 0);
  ws.sorted_cap = sorted_cap;
  ws.blocks_cap = blocks_cap;

  const size_t smem = static_cast<size_t>(kChunkWarps) * E * sizeof(int32_t);
  static bool attr_set[64] = {};
  if (!attr_set[dev.device]) {
    MOE_CUDA_TRY(cudaFuncSetAttribute(plan_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kChunkWarps * kMaxExperts * 4));
    MOE_CUDA_TRY(cudaFuncSetAttribute(plan_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (kScanThreads / 32) * kSmallMaxExperts * 4));
    attr_set[dev.device] = true;
  }
  if (R <= kSmallRoutes && E <= kSmallMaxExperts) {
    const size_t small_smem = static_cast<size_t>(kScanThreads / 32) * E * sizeof(int32_t);
    MOE_CUDA_TRY(launch_pdl(plan_small_kernel, dim3(1), dim3(kScanThreads), small_smem, stream, 1, topk_ids, id_bits,
                            R, E, block_m, sorted_token_ids, expert_ids, num_tokens_post_padded, sorted_cap,
                            blocks_cap));
    return MOE_OK;
  }
  if (R > 0) {
    MOE_CUDA_TRY(launch_pdl(plan_rank_kernel, dim3(static_cast<unsigned>(nchunks)), dim3(kChunk), smem, stream, 1,
                            topk_ids, id_bits, R, E, ws));
  } else {
    nchunks = 0;
  }
  MOE_CUDA_TRY(launch_pdl(plan_scan_kernel, dim3(1), dim3(kScanThreads), 0, stream, 1, R, E, block_m,
                          static_cast<int>(nchunks), ws, sorted_token_ids, expert_ids, num_tokens_post_padded));
  if (R > 0) {
    MOE_CUDA_TRY(launch_pdl(plan_scatter_kernel, dim3(static_cast<unsigned>(nchunks)), dim3(kChunk), 0, stream, 1,
                            topk_ids, id_bits, R, E, ws, sorted_token_ids));
  }
  return MOE_OK;
}

moe_status moe_route_plan(const void* logits, int logit_dtype, int64_t M, int E, int top_k, float routed_scale,
                          int renormalize, void* topk_ids, int id_bits, float* topk_weights, int block_m,
                          int32_t* sorted_token_ids, int64_t sorted_cap, int32_t* expert_ids, int64_t blocks_cap,
                          int32_t* num_tokens_post_padded, moe_stream_t stream) {
  using namespace moe;
  if (logit_dtype != MOE_LOGITS_F32 && logit_dtype != MOE_LOGITS_BF16) return MOE_ERR_DTYPE;
  if (id_bits != 32 && id_bits != 64) return MOE_ERR_DTYPE;
  if (M < 0 || E < 1 || E > kSmallMaxExperts || top_k < 1 || top_k > kRouteMaxTopK || top_k > E) return MOE_ERR_SHAPE;
  if (block_m < 8 || block_m > 1024 || block_m % 8 != 0) return MOE_ERR_SHAPE;
  if (M * static_cast<int64_t>(top_k) > kSmallRoutes) return MOE_ERR_SHAPE;
  if (!sorted_token_ids || !expert_ids || !num_tokens_post_padded) return MOE_ERR_NULL;
  if (M > 0 && (!logits || !topk_ids || !topk_weights)) return MOE_ERR_NULL;
  int64_t need_cap = 0, need_blocks = 0;
  moe_plan_capacity(M, top_k, E, block_m, &need_cap, &need_blocks);
  if (sorted_cap < need_cap || blocks_cap < need_blocks) return MOE_ERR_CAPACITY;
  DeviceInfo dev;
  if (current_device(&dev) != MOE_OK) return MOE_ERR_CUDA;
  if ((M > 0 && (!on_device(logits, dev.device) || !on_device(topk_ids, dev.device) ||
                 !on_device(topk_weights, dev.device))) ||
      !on_device(sorted_token_ids, dev.device) || !on_device(expert_ids, dev.device) ||
      !on_device(num_tokens_post_padded, dev.device))
    return MOE_ERR_DEVICE;
  static bool attr_set[64] = {};
  if (!attr_set[dev.device]) {
    const int smem = (kScanThreads / 32) * kSmallMaxExperts * 4;
    MOE_CUDA_TRY(cudaFuncSetAttribute(route_plan_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    MOE_CUDA_TRY(cudaFuncSetAttribute(route_plan_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    MOE_CUDA_TRY(cudaFuncSetAttribute(route_plan_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    MOE_CUDA_TRY(cudaFuncSetAttribute(route_plan_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    MOE_CUDA_TRY(cudaFuncSetAttribute(route_plan_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    MOE_CUDA_TRY(cudaFuncSetAttribute(route_plan_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    attr_set[dev.device] = true;
  }
  const size_t smem = static_cast<size_t>(kScanThreads / 32) * E * sizeof(int32_t);
  const int per = static_cast<int>(ceil_div(static_cast<int64_t>(E), int64_t(32)));
  cudaError_t err;
#define MOE_ROUTE_PLAN(K)                                                                                          \
  launch_pdl(route_plan_kernel<K>, dim3(1), dim3(kScanThreads), smem, stream, 1, logits, logit_dtype, M, E, top_k, \
             routed_scale, renormalize, topk_ids, id_bits, topk_weights, block_m, sorted_token_ids, expert_ids,   \
             num_tokens_post_padded, sorted_cap, blocks_cap)
  if (per <= 1)
    err = MOE_ROUTE_PLAN(1);
  else if (per <= 2)
    err = MOE_ROUTE_PLAN(2);
  else if (per <= 4)
    err = MOE_ROUTE_PLAN(4);
  else if (per <= 8)
    err = MOE_ROUTE_PLAN(8);
  else if (per <= 16)
    err = MOE_ROUTE_PLAN(16);
  else
    err = MOE_ROUTE_PLAN(32);
#undef MOE_ROUTE_PLAN
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"

MOE_BOUNDS_TU()
