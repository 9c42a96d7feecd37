// moe_fp8_block_scale_forward: the fused block-scaled FP8 MoE expert
// computation on GB300 (FlashInfer PR #4287: commit summary; "Public contract
// and review fixes"; post-dot scale application from "Final W8 kernel
// performance (v46)").
//
// Three launches on the caller's stream:
//   1. up   (gemm kernel, kUp = true): for every (plan block, 256-wide tile of
//      the interleaved gate/up weights): gathered activation rows x W13 tile on
//      tcgen05 tensor cores, one 128-wide K slice at a time into TMEM; the
//      epilogue warps promote each slice in FP32 with the activation and
//      weight block scales, then apply SwiGLU and requantise the 128
//      intermediate columns of the tile to E4M3 (scale amax/448) into the
//      workspace.
//   2. down (gemm kernel, kUp = false): intermediate rows x W2 tile, promoted
//      with the intermediate and W2 block scales, times the route weight and
//      routed scale, reduced into an FP32 [M, H] accumulator.
//   3. finalize: out = bf16_rn(f32(out) + acc); acc = 0.
//
// The GEMM kernel is persistent and warp specialised (320 threads):
//   warp 0      TMA producer: gathered activation rows (tile::gather4) or
//               intermediate rows, plus the 256-row weight tile, into a
//               4-stage ring of 48 KiB stages (128-byte swizzle);
//   warp 1      TMEM allocation and the single MMA-issuing thread
//               (kind::f8f6f4, M=128, N=256, K=32 per instruction, 4 per slice);
//   warps 2..9  epilogue: each owns 32 tile rows (its TMEM lane quarter) and
//               128 of the 256 columns; FP32 accumulators live in registers.
// TMEM holds two 256-column FP32 partial buffers so the tensor core computes
// slice k+1 while the epilogue promotes slice k.  Every wait is bounded; a
// wait that runs out raises MOE_DEV_TIMEOUT in *device_status and the CTA
// winds down (draining its copies and MMAs, freeing TMEM).
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kStages = 4;
constexpr int kTileM = 128;
constexpr int kTileN = 256;
constexpr int kTileK = 128;
constexpr int kABytes = kTileM * kTileK;  // 16 KiB
constexpr int kBBytes = kTileN * kTileK;  // 32 KiB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kNumEpiWarps = 8;
constexpr int kNumThreads = 64 + 32 * kNumEpiWarps;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdesc = idesc_e4m3_f32(kTileM, kTileN);

struct SmemCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint32_t tmem_base;
  int abort_flag;
  int pad[2];
  float xchg[2][2][kTileM];  // [tile parity][column half][row]: amax exchange
};

constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(kStages) * kStageBytes + sizeof(SmemCtl);

struct GemmParams {
  const int32_t* sorted_ids;
  const int32_t* expert_ids;
  const int32_t* num_post_padded;
  const float* a_scale;   // up: [M, nkb] per token; down: [sorted_cap, nkb] per plan slot
  const float* b_scale;   // up: w13_scale [E, 2I/128, nkb]; down: w2_scale [E, H/128, nkb]
  const float* topk_w;    // down: [M * top_k]
  float* acc_out;         // down: [M, H]
  uint8_t* q_inter;       // up: [sorted_cap, I]
  float* s_inter;         // up: [sorted_cap, I/128]
  uint8_t* dbg_q;         // up, nullable
  float* dbg_s;           // up, nullable
  int32_t* status;        // nullable
  int64_t nblocks;        // plan block slots the grid walks
  int R;
  int top_k;
  int block_m;
  int E;
  int nkb;                // K / 128
  int ntiles_n;           // 256-wide output tiles per expert
  int b_rows;             // weight rows per expert (2I or H)
  int b_row_blocks;       // b_rows / 128 rounded up
  int I;
  int H;
  float routed_scale;
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Bounded wait used while winding down: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  int dummy = 0;
  mbar_wait(bar, parity, &dummy);
}

__device__ __forceinline__ void report(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

// Tile -> (plan block, n tile, expert); false if the tile has no work.
__device__ __forceinline__ bool tile_coords(const GemmParams& p, int64_t tile, int64_t nvalid, int& b, int& t, int& e) {
  b = static_cast<int>(tile % p.nblocks);
  t = static_cast<int>(tile / p.nblocks);
  if (b >= nvalid) return false;
  e = p.expert_ids[b];
  return e >= 0 && e < p.E;
}

__device__ __forceinline__ float silu_f32(float g) { return __fdiv_rn(g, 1.0f + expf(-g)); }

template <bool kUp>
__global__ void __launch_bounds__(kNumThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem + kStages * kStageBytes);
  volatile int* abort_flag = &ctl->abort_flag;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctl->tfull[b]), 1);
      mbar_init(smem_u32(&ctl->tempty[b]), kNumEpiWarps);
    }
    ctl->abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  int64_t P = *p.num_post_padded;
  if (P < 0) P = 0;
  int64_t nvalid = P / p.block_m;
  if (nvalid > p.nblocks) nvalid = p.nblocks;
  const int64_t total = p.nblocks * p.ntiles_n;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t it = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      int b, t, e;
      if (!tile_coords(p, tile, nvalid, b, t, e)) continue;
      int tok[4] = {0, 0, 0, 0};
      if (kUp) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 4 * lane + i;
          int id = -1;
          if (r < p.block_m) id = p.sorted_ids[static_cast<int64_t>(b) * p.block_m + r];
          tok[i] = (id >= 0 && id < p.R) ? id / p.top_k : 0;
        }
      }
      const int brow = e * p.b_rows + t * kTileN;
      for (int kb = 0; kb < p.nkb; ++kb) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        if (!warp_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t full = smem_u32(&ctl->full[s]);
        if (lane == 0) mbar_arrive_expect_tx(full, kStageBytes);
        __syncwarp();
        const uint32_t a_dst = smem_u32(sA + s * kABytes);
        if (kUp) {
          tma_gather4(a_dst + 512u * lane, &tmA, full, kb * kTileK, tok[0], tok[1], tok[2], tok[3]);
        } else if (lane == 0) {
          tma_load_2d(a_dst, &tmA, full, kb * kTileK, b * p.block_m);
        }
        if (lane == 0) tma_load_2d(smem_u32(sB + s * kBBytes), &tmB, full, kb * kTileK, brow);
        ++it;
      }
    }
    if (!ok && lane == 0) {
      // wind down: let the copies already issued land before the CTA exits
      for (uint32_t j = (it > kStages ? it - kStages : 0); j < it; ++j)
        drain_wait(smem_u32(&ctl->full[j % kStages]), (j / kStages) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int64_t tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        int b, t, e;
        if (!tile_coords(p, tile, nvalid, b, t, e)) continue;
        for (int kb = 0; kb < p.nkb; ++kb) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          const uint32_t tb = it & 1u;
          const uint32_t tph = (it >> 1) & 1u;
          if (!mbar_wait(smem_u32(&ctl->full[s]), ph, abort_flag) ||
              !mbar_wait(smem_u32(&ctl->tempty[tb]), tph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * kABytes);
          const uint32_t b0 = smem_u32(sB + s * kBBytes);
          const uint32_t d = tmem_base + tb * kTileN;
#pragma unroll
          for (int kk = 0; kk < kTileK / 32; ++kk)
            umma_f8(d, sw128_kmajor_desc(a0 + 32u * kk), sw128_kmajor_desc(b0 + 32u * kk), kIdesc, kk > 0 ? 1u : 0u);
          umma_commit(smem_u32(&ctl->empty[s]));
          umma_commit(smem_u32(&ctl->tfull[tb]));
          ++it;
        }
      }
      // no MMA may still be writing TMEM when it is released
      if (it > 0) drain_wait(smem_u32(&ctl->tfull[(it - 1) & 1u]), ((it - 1) >> 1) & 1u);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t it = 0;
    int tcount = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int b, t, e;
      if (!tile_coords(p, tile, nvalid, b, t, e)) {
        if (warp == 2 && lane == 0 && t == 0 && static_cast<int64_t>(b) < nvalid) {
          const int bad = p.expert_ids[b];
          if (bad != -1) report(p.status, MOE_DEV_BAD_EXPERT);
        }
        continue;
      }
      const int64_t slot = static_cast<int64_t>(b) * p.block_m + row;
      const bool rvalid = row < p.block_m;
      const int id = rvalid ? p.sorted_ids[slot] : -1;
      const bool is_route = id >= 0 && id < p.R;

      const float* as_row;
      const float* ws0;
      const float* ws1;
      bool cols_valid = true;
      if (kUp) {
        const int tok = is_route ? id / p.top_k : 0;
        as_row = p.a_scale + static_cast<int64_t>(tok) * p.nkb;
        ws0 = p.b_scale + (static_cast<int64_t>(e) * p.b_row_blocks + t) * p.nkb;                  // gate block
        ws1 = p.b_scale + (static_cast<int64_t>(e) * p.b_row_blocks + p.I / 128 + t) * p.nkb;      // up block
      } else {
        const int hblk = 2 * t + half;
        cols_valid = hblk < p.b_row_blocks;
        as_row = p.a_scale + (rvalid ? slot : 0) * p.nkb;
        ws0 = p.b_scale + (static_cast<int64_t>(e) * p.b_row_blocks + (cols_valid ? hblk : 0)) * p.nkb;
        ws1 = ws0;
      }

      float acc[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) acc[c] = 0.f;

      for (int kb = 0; kb < p.nkb; ++kb) {
        const float as = rvalid ? __ldg(as_row + kb) : 0.f;
        const float s0 = __fmul_rn(as, __ldg(ws0 + kb));
        const float s1 = kUp ? __fmul_rn(as, __ldg(ws1 + kb)) : s0;
        const uint32_t tb = it & 1u;
        const uint32_t tph = (it >> 1) & 1u;
        if (ok) ok = warp_wait(smem_u32(&ctl->tfull[tb]), tph, abort_flag);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(lane_base + tb * kTileN + 128u * half + 32u * ch, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float sc = (kUp && (i & 8)) ? s1 : s0;
              acc[32 * ch + i] = fmaf(__uint_as_float(v[i]), sc, acc[32 * ch + i]);
            }
          }
          tc_fence_before();
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(smem_u32(&ctl->tempty[tb]));
        ++it;
      }

      if (kUp) {
        // SwiGLU on the 64 (gate, up) pairs this thread holds, then the
        // per-token 1x128 requant shared with the partner warp (other half).
        float amax = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float h = __fmul_rn(silu_f32(acc[16 * q + j]), acc[16 * q + 8 + j]);
            acc[8 * q + j] = h;  // compact in place: slot 8q+j is free once read
            amax = fmaxf(amax, fabsf(h));
          }
        }
        ctl->xchg[tcount & 1][half][row] = amax;
        named_barrier(1, 32 * kNumEpiWarps);
        amax = fmaxf(amax, ctl->xchg[tcount & 1][half ^ 1][row]);
        const float s = __fdiv_rn(amax, 448.0f);
        if (ok && rvalid) {
          uint32_t packed[16];
#pragma unroll
          for (int w = 0; w < 16; ++w) {
            uint32_t word = 0;
            if (s > 0.f) {
              const uint16_t lo = cvt_e4m3x2(__fdiv_rn(acc[4 * w + 0], s), __fdiv_rn(acc[4 * w + 1], s));
              const uint16_t hi = cvt_e4m3x2(__fdiv_rn(acc[4 * w + 2], s), __fdiv_rn(acc[4 * w + 3], s));
              word = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            }
            packed[w] = word;
          }
          const int64_t qoff = slot * p.I + 128 * t + 64 * half;
          uint4* qdst = reinterpret_cast<uint4*>(p.q_inter + qoff);
#pragma unroll
          for (int w = 0; w < 4; ++w)
            qdst[w] = make_uint4(packed[4 * w], packed[4 * w + 1], packed[4 * w + 2], packed[4 * w + 3]);
          if (half == 0) p.s_inter[slot * (p.I / 128) + t] = s;
          if (p.dbg_q) {
            uint4* ddst = reinterpret_cast<uint4*>(p.dbg_q + qoff);
#pragma unroll
            for (int w = 0; w < 4; ++w)
              ddst[w] = make_uint4(packed[4 * w], packed[4 * w + 1], packed[4 * w + 2], packed[4 * w + 3]);
            if (half == 0) p.dbg_s[slot * (p.I / 128) + t] = s;
          }
        }
      } else if (ok && is_route && cols_valid) {
        const float wr = __fmul_rn(__ldg(p.topk_w + id), p.routed_scale);
        const int tok = id / p.top_k;
        float* dst = p.acc_out + static_cast<int64_t>(tok) * p.H + (2 * t + half) * 128;
#pragma unroll
        for (int c = 0; c < 128; c += 4)
          red_add_v4(dst + c, __fmul_rn(acc[c], wr), __fmul_rn(acc[c + 1], wr), __fmul_rn(acc[c + 2], wr),
                     __fmul_rn(acc[c + 3], wr));
      }
      ++tcount;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0 && ctl->abort_flag) report(p.status, MOE_DEV_TIMEOUT);
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// out = bf16_rn(f32(out) + acc); acc = 0.  Eight elements per thread.
__global__ void __launch_bounds__(256) finalize_kernel(uint16_t* __restrict__ out, float* __restrict__ acc, int64_t n8) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    uint4 o = reinterpret_cast<uint4*>(out)[i];
    float4* ap = reinterpret_cast<float4*>(acc) + 2 * i;
    const float4 a0 = ap[0];
    const float4 a1 = ap[1];
    ap[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    ap[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float lo = __fadd_rn(__uint_as_float((ow[k] & 0xFFFFu) << 16), av[2 * k]);
      const float hi = __fadd_rn(__uint_as_float(ow[k] & 0xFFFF0000u), av[2 * k + 1]);
      const uint32_t blo = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
      const uint32_t bhi = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
      ow[k] = blo | (bhi << 16);
    }
    reinterpret_cast<uint4*>(out)[i] = o;
  }
}

struct WsLayout {
  size_t acc_off, q_off, s_off, total;
};

WsLayout ws_layout(int64_t M, int H, int I, int64_t sorted_cap) {
  WsLayout l;
  l.acc_off = 0;
  l.q_off = static_cast<size_t>(round_up(M * H * 4, 256));
  l.s_off = l.q_off + static_cast<size_t>(round_up(sorted_cap * I, 256));
  l.total = l.s_off + static_cast<size_t>(round_up(sorted_cap * (I / 128) * 4, 256));
  return l;
}

bool set_smem_attrs(int device) {
  static std::mutex mu;
  static bool done[64] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (done[device]) return true;
  if (cudaFuncSetAttribute(moe_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes)) != cudaSuccess)
    return false;
  if (cudaFuncSetAttribute(moe_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes)) != cudaSuccess)
    return false;
  done[device] = true;
  return true;
}

}  // namespace
}  // namespace moe

extern "C" {

size_t moe_forward_workspace_size(int64_t M, int H, int I, int top_k, int block_m, int64_t sorted_cap) {
  (void)top_k;
  (void)block_m;
  if (M < 0 || H < 0 || I < 0 || sorted_cap < 0) return 0;
  return moe::ws_layout(M, H, I, sorted_cap).total;
}

moe_status moe_fp8_block_scale_forward(const moe_fwd_args* a, moe_stream_t stream) {
  using namespace moe;
  if (!a) return MOE_ERR_NULL;
  if (a->M < 0 || a->H < 128 || a->H % 128 || a->I < 128 || a->I % 128 || a->E < 1 || a->top_k < 1)
    return MOE_ERR_SHAPE;
  if (a->block_m < 8 || a->block_m > 128 || a->block_m % 8) return MOE_ERR_SHAPE;
  if (a->blocks_cap < 1 || a->sorted_cap < a->blocks_cap * a->block_m) return MOE_ERR_CAPACITY;
  const int64_t R = a->M * a->top_k;
  if (R >= (int64_t(1) << 31) - 1 || static_cast<int64_t>(a->E) * 2 * a->I >= (int64_t(1) << 31) ||
      static_cast<int64_t>(a->E) * a->H >= (int64_t(1) << 31) || a->sorted_cap >= (int64_t(1) << 31))
    return MOE_ERR_SHAPE;
  if (a->M == 0) return MOE_OK;
  if (!a->a || !a->a_scale || !a->w13 || !a->w13_scale || !a->w2 || !a->w2_scale || !a->topk_weights ||
      !a->sorted_token_ids || !a->expert_ids || !a->num_tokens_post_padded || !a->out || !a->workspace)
    return MOE_ERR_NULL;
  if ((a->debug_q_inter == nullptr) != (a->debug_s_inter == nullptr)) return MOE_ERR_NULL;
  if (!aligned16(a->a) || !aligned16(a->w13) || !aligned16(a->w2) || !aligned16(a->workspace) ||
      !aligned16(a->out) || (a->debug_q_inter && !aligned16(a->debug_q_inter)))
    return MOE_ERR_ALIGN;
  const WsLayout wl = ws_layout(a->M, a->H, a->I, a->sorted_cap);
  if (a->workspace_bytes < wl.total) return MOE_ERR_CAPACITY;

  DeviceInfo dev;
  if (current_device(&dev) != MOE_OK) return MOE_ERR_CUDA;
  if (dev.major != 10 || dev.minor != 3) return MOE_ERR_DEVICE;
  const void* ptrs[] = {a->a, a->a_scale, a->w13, a->w13_scale, a->w2, a->w2_scale, a->topk_weights,
                        a->sorted_token_ids, a->expert_ids, a->num_tokens_post_padded, a->out, a->workspace};
  for (const void* ptr : ptrs)
    if (!on_device(ptr, dev.device)) return MOE_ERR_DEVICE;
  if (a->device_status && !on_device(a->device_status, dev.device)) return MOE_ERR_DEVICE;
  if (a->debug_q_inter && (!on_device(a->debug_q_inter, dev.device) || !on_device(a->debug_s_inter, dev.device)))
    return MOE_ERR_DEVICE;
  if (!set_smem_attrs(dev.device)) return MOE_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  float* acc = reinterpret_cast<float*>(ws + wl.acc_off);
  uint8_t* q_inter = ws + wl.q_off;
  float* s_inter = reinterpret_cast<float*>(ws + wl.s_off);

  const int N = 2 * a->I;
  CUtensorMap tm_a, tm_w13, tm_q, tm_w2;
  if (encode_tensor_map_2d(&tm_a, a->a, a->H, a->M, a->H, 128, 1, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_tensor_map_2d(&tm_w13, a->w13, a->H, static_cast<uint64_t>(a->E) * N, a->H, 128, 256,
                           CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_tensor_map_2d(&tm_q, q_inter, a->I, a->sorted_cap, a->I, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) !=
          CUDA_SUCCESS ||
      encode_tensor_map_2d(&tm_w2, a->w2, a->I, static_cast<uint64_t>(a->E) * a->H, a->I, 128, 256,
                           CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return MOE_ERR_CUDA;

  // Plan blocks that can hold work: P <= R + min(E, R) * (block_m - 1).
  const int64_t nonempty = R < a->E ? R : a->E;
  int64_t nblocks = ceil_div(R + nonempty * (a->block_m - 1), a->block_m);
  if (nblocks > a->blocks_cap) nblocks = a->blocks_cap;

  GemmParams p{};
  p.sorted_ids = a->sorted_token_ids;
  p.expert_ids = a->expert_ids;
  p.num_post_padded = a->num_tokens_post_padded;
  p.status = a->device_status;
  p.nblocks = nblocks;
  p.R = static_cast<int>(R);
  p.top_k = a->top_k;
  p.block_m = a->block_m;
  p.E = a->E;
  p.I = a->I;
  p.H = a->H;
  p.routed_scale = a->routed_scale;

  cudaEvent_t const* ev = reinterpret_cast<cudaEvent_t const*>(a->profile_events);
  if (ev) MOE_CUDA_TRY(cudaEventRecord(ev[0], stream));
  if (nblocks > 0) {
    GemmParams up = p;
    up.a_scale = a->a_scale;
    up.b_scale = a->w13_scale;
    up.q_inter = q_inter;
    up.s_inter = s_inter;
    up.dbg_q = a->debug_q_inter;
    up.dbg_s = a->debug_s_inter;
    up.nkb = a->H / 128;
    up.ntiles_n = N / kTileN;
    up.b_rows = N;
    up.b_row_blocks = N / 128;
    const int64_t up_tiles = nblocks * up.ntiles_n;
    const int up_grid = static_cast<int>(up_tiles < dev.sms ? up_tiles : dev.sms);
    moe_gemm_kernel<true><<<up_grid, kNumThreads, kSmemBytes, stream>>>(tm_a, tm_w13, up);
    MOE_CUDA_TRY(cudaGetLastError());
    if (ev) MOE_CUDA_TRY(cudaEventRecord(ev[1], stream));

    GemmParams dn = p;
    dn.a_scale = s_inter;
    dn.b_scale = a->w2_scale;
    dn.topk_w = a->topk_weights;
    dn.acc_out = acc;
    dn.nkb = a->I / 128;
    dn.ntiles_n = static_cast<int>(ceil_div(a->H, kTileN));
    dn.b_rows = a->H;
    dn.b_row_blocks = a->H / 128;
    const int64_t dn_tiles = nblocks * dn.ntiles_n;
    const int dn_grid = static_cast<int>(dn_tiles < dev.sms ? dn_tiles : dev.sms);
    moe_gemm_kernel<false><<<dn_grid, kNumThreads, kSmemBytes, stream>>>(tm_q, tm_w2, dn);
    MOE_CUDA_TRY(cudaGetLastError());
  } else if (ev) {
    MOE_CUDA_TRY(cudaEventRecord(ev[1], stream));
  }
  if (ev) MOE_CUDA_TRY(cudaEventRecord(ev[2], stream));

  const int64_t n8 = a->M * a->H / 8;
  int64_t fgrid = ceil_div(n8, 256);
  if (fgrid > static_cast<int64_t>(dev.sms) * 8) fgrid = static_cast<int64_t>(dev.sms) * 8;
  finalize_kernel<<<static_cast<unsigned>(fgrid), 256, 0, stream>>>(a->out, acc, n8);
  MOE_CUDA_TRY(cudaGetLastError());
  if (ev) MOE_CUDA_TRY(cudaEventRecord(ev[3], stream));
  return MOE_OK;
}

}  // extern "C"
