// Tensor-core projections of the E2M1-K32 weight x FP8 activation variant
// (sglang-glm53-flash-sm120 pull request #13, "SM120 FP8 prefill",
// description: E2M1 weights with one FP32 scale per 32 elements of K,
// applied in FP32; E4M3 activations with one FP32 scale per row).
//
// One persistent, warp-specialised kernel serves both projections.  Its
// tiles are swapped against the FP8 path's: the MMA's M operand is 128
// weight rows (tcgen05 kind::f8f6f4 takes E2M1 as one operand and E4M3 as
// the other), its N operand the route rows of a plan block group (up to 64,
// 32 or 16 by the kernel's width: consecutive plan blocks of one expert are
// taken together, so an expert's weights stream through once per group).  A weight row's K32 scale then
// belongs to one TMEM lane, and the epilogue promotes each 32-wide K block's
// partial with a single per-thread scalar.
//
//   warp 0      producer: per 128-wide K slice, the packed E2M1 weight tile
//               (the copy engine writes it in the padded form the tensor core
//               reads: 16U4_ALIGN16B, 128-byte swizzle), the weight rows' four
//               K32 scales, and the group's activation (gate/up) or
//               intermediate (down) rows gathered by token or route id
//               (tile::gather4), into a 6- or 8-stage ring, one box per
//               lane (a thread issues its copies one after another);
//   warp 1      TMEM allocation and the MMA thread: four K = 32 MMAs per
//               slice, each into its own N columns of one of the 2, 4 or 8
//               TMEM buffers;
//   warps 2..9  epilogue: warp w owns TMEM lane quarter w % 4 (32 weight
//               rows) and half of the route columns; per slice it adds each
//               K32 partial times its row's scale to FP32 registers;
//   warp 10     route tables, one tile ahead: each column's route id and its
//               scales, in two shared-memory tables.
// Gate/up tile = 64 gate rows + the 64 matching up rows of the logical W13:
// at the tile end the up rows' values pass through shared memory to the gate
// rows' threads, which write silu(g) * u by route id.  Down tile = 128 W2
// rows; the tile end writes y * s * w by route id.
#include "common.cuh"
#include "w4a8_tc.cuh"

namespace moe {
namespace {

constexpr int kTM = 128;                  // weight rows per tile (MMA M)
constexpr int kTK = 128;                  // K elements per stage
// The kernel comes in three widths: up to 64 route rows per tile with two
// TMEM buffers (each buffer: a slice's four K32 partials x 64 columns) and
// 6 stages; up to 32 rows with four buffers and 8 stages; and up to 16 rows
// with eight buffers and 8 stages.  More buffers let the MMAs run further
// ahead of the epilogue; the narrower widths serve small plans and plan
// blocks of up to 32 rows.
template <int kN>
struct W4Cfg {
  static constexpr int kMaxN = kN;                       // route rows per tile (MMA N)
  static constexpr int kTBufs = 512 / (4 * kN);          // TMEM buffers: 2 or 8
  static constexpr int kStages = kN == 64 ? 6 : 8;
  static constexpr int kBBytes = kN * 128;               // activation / intermediate rows per stage
};
constexpr int kEpiWarps = 8;
constexpr int kLoaderWarp = 2 + kEpiWarps;  // after the producer, the MMA warp and the epilogue
constexpr int kThreads = 32 * (kLoaderWarp + 1);
constexpr int kWBytes = kTM * kTK;        // 16 KiB in shared memory (padded E2M1)
constexpr int kWTx = kTM * kTK / 2;       // the packed bytes the copy engine counts
constexpr int kSBytes = kTM * 16;         // four FP32 K32 scales per weight row
constexpr int kMaxBlocks = 1024;          // plan blocks whose expert is cached in shared memory
constexpr uint32_t kTmemCols = 512;       // kTBufs buffers x 4 K32 partials x kMaxN columns

template <int kN>
struct alignas(16) W4Ctl {
  static constexpr int kMaxN = kN;
  uint64_t full[W4Cfg<kN>::kStages];
  uint64_t empty[W4Cfg<kN>::kStages];
  uint64_t tfull[W4Cfg<kN>::kTBufs];
  uint64_t tempty[W4Cfg<kN>::kTBufs];
  uint64_t rfull[2];                      // a tile's route table is written (producer)
  uint64_t rempty[2];                     // ... and has been used (every epilogue warp)
  uint32_t tmem_base;
  int abort_flag;
  int pad[2];
  // route tables of two consecutive tiles, filled by the producer
  int32_t route[2][kMaxN];                // the tile's route id per column (-1 = none)
  float cs[2][kMaxN];                     // per column: activation scale (up) / intermediate scale (down)
  float cw[2][kMaxN];                     // down: route weight x routed scale
  float xchg[64][kMaxN + 1];              // up: up-row values handed to the gate rows' threads
  int32_t expert[kMaxBlocks];
  uint8_t lead[kMaxBlocks];               // blocks in the group this block leads (0: not a group leader)
};

template <int kN>
constexpr size_t smem_bytes_w4() {
  return 1024 + static_cast<size_t>(W4Cfg<kN>::kStages) * (kWBytes + W4Cfg<kN>::kBBytes + kSBytes) + sizeof(W4Ctl<kN>);
}
static_assert(smem_bytes_w4<64>() <= 232448 && smem_bytes_w4<32>() <= 232448 && smem_bytes_w4<16>() <= 232448,
              "shared memory budget");

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  int dummy = 0;
  mbar_wait(bar, parity, &dummy);
}

__device__ __forceinline__ void tma_gather4_rows(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y0,
                                                 int y1, int y2, int y3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3)
      : "memory");
}

// Tile -> (leading plan block b, weight tile wt, expert e, blocks in the group
// nb); false if the tile has no work.
template <class Ctl>
__device__ __forceinline__ bool w4_tile(const W4GemmParams& p, const Ctl* ctl, int64_t tile, int64_t nvalid,
                                        int& b, int& wt, int& e, int& nb) {
  b = static_cast<int>(tile / p.ntw);
  wt = static_cast<int>(tile % p.ntw);
  if (b >= nvalid) return false;
  if (b < kMaxBlocks) {
    nb = ctl->lead[b];
    e = ctl->expert[b];
  } else {
    nb = 1;
    e = MOE_IN_BOUNDS(b < p.nblocks) ? p.expert_ids[b] : -1;
  }
  return nb > 0 && e >= 0 && e < p.E;
}

template <int kN>
__global__ void __launch_bounds__(kThreads, 1)
    w4a8_tc_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
                        const __grid_constant__ CUtensorMap tmB, const W4GemmParams p) {
  using C = W4Cfg<kN>;
  using W4CtlT = W4Ctl<kN>;
  constexpr int kMaxN = C::kMaxN;
  constexpr int kStages = C::kStages;
  constexpr int kBBytes = C::kBBytes;
  constexpr int kTBufs = C::kTBufs;
  constexpr uint32_t kBufCols = 4u * kMaxN;  // TMEM columns per buffer
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;
  uint8_t* sB = sW + kStages * kWBytes;
  uint8_t* sS = sB + kStages * kBBytes;
  W4CtlT* ctl = reinterpret_cast<W4CtlT*>(sS + kStages * kSBytes);
  volatile int* abort_flag = &ctl->abort_flag;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1 + kEpiWarps);  // MMA commit + every epilogue warp (reads the scales)
    }
    for (int i = 0; i < kTBufs; ++i) {
      mbar_init(smem_u32(&ctl->tfull[i]), 1);
      mbar_init(smem_u32(&ctl->tempty[i]), kEpiWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctl->rfull[i]), 1);
      mbar_init(smem_u32(&ctl->rempty[i]), kEpiWarps);
    }
    ctl->abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmS);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&ctl->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // everything this kernel reads was written before it was launched
  int64_t P = *p.num_post_padded;
  if (P < 0) P = 0;
  int64_t nvalid = P / p.block_m;
  if (nvalid > p.nblocks) nvalid = p.nblocks;
  const int64_t ncache = nvalid < kMaxBlocks ? nvalid : kMaxBlocks;
  for (int64_t b = threadIdx.x; b < ncache; b += blockDim.x) ctl->expert[b] = p.expert_ids[b];
  __syncthreads();
  // group leaders: the first block of an expert's run and every G-th after it
  for (int64_t b = threadIdx.x; b < ncache; b += blockDim.x) {
    const int e = ctl->expert[b];
    int64_t run = 0;
    while (b - run - 1 >= 0 && ctl->expert[b - run - 1] == e) ++run;
    int n = 0;
    if (run % p.group == 0)
      while (n < p.group && b + n < ncache && ctl->expert[b + n] == e) ++n;
    ctl->lead[b] = static_cast<uint8_t>(n);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  const int64_t total = nvalid * p.ntw;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t it = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      int b, wt, e, nb;
      if (!w4_tile(p, ctl, tile, nvalid, b, wt, e, nb)) continue;
      const int rows = nb * p.block_m;
      const int nmma = (rows + 15) & ~15;
      // the gather rows of lane l: group rows 4l .. 4l + 3 (tokens for gate/up,
      // route ids for down; 0 for rows without a route)
      int ids[4];
      bool mine = 4 * lane < nmma;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = 4 * lane + i;
        const int64_t slot = static_cast<int64_t>(b) * p.block_m + r;
        int id = -1;
        if (r < rows && MOE_IN_BOUNDS(slot < p.sorted_cap)) id = p.sorted_ids[slot];
        const bool route = id >= 0 && id < p.R;
        ids[i] = route ? (p.up ? id / p.top_k : id) : 0;
        if (!MOE_IN_BOUNDS(ids[i] < p.rows_total)) ids[i] = 0;
      }
      const uint32_t tx = kWTx + kSBytes + static_cast<uint32_t>(nmma) * kTK;
      const int wrow = p.up ? e * p.w_rows + wt * 64 : e * p.w_rows + wt * kTM;
      for (int kb = 0; kb < p.nkb; ++kb) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        if (!warp_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t full = smem_u32(&ctl->full[s]);
        if (lane == 0) mbar_arrive_expect_tx(full, tx);
        __syncwarp();
        {
          // one copy per lane (a thread's copies are issued one after
          // another): lanes 0/1 the weight boxes of the 64 gate and 64 up
          // rows (I rows further), or lane 0 the 128 W2 rows; lanes 2/3 the
          // matching scale boxes
          const int part = lane & 1;
          if (lane < 4 && part < (p.up ? 2 : 1)) {
            int wx = kb * kTK, wy = wrow + part * p.I, sx = kb * 4, sy = wy;
            if (lane < 2) {
              MOE_CHECK_BOX(wx, wy, static_cast<int64_t>(p.nkb) * kTK, static_cast<int64_t>(p.E) * p.w_rows, 32);
              tma_load_2d(smem_u32(sW + s * kWBytes) + part * 64 * kTK, &tmW, full, wx, wy);
            } else {
              MOE_CHECK_BOX(sx, sy, static_cast<int64_t>(p.nkb) * 4, static_cast<int64_t>(p.E) * p.w_rows, 4);
              tma_load_2d(smem_u32(sS + s * kSBytes) + part * 64 * 16, &tmS, full, sx, sy);
            }
          }
        }
        __syncwarp();
        int gx = kb * kTK;
        if (!MOE_IN_BOUNDS(gx % 16 == 0 && gx < p.nkb * kTK)) gx = 0;
        if (mine)
          tma_gather4_rows(smem_u32(sB + s * kBBytes) + 512u * lane, &tmB, full, gx, ids[0], ids[1], ids[2], ids[3]);
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
        int b, wt, e, nb;
        if (!w4_tile(p, ctl, tile, nvalid, b, wt, e, nb)) continue;
        const int nmma = (nb * p.block_m + 15) & ~15;
        const uint32_t idesc = idesc_e2m1_e4m3_f32(kTM, nmma);
        for (int kb = 0; kb < p.nkb; ++kb) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          const uint32_t tb = it % kTBufs;
          const uint32_t tph = (it / kTBufs) & 1u;
          if (!mbar_wait(smem_u32(&ctl->full[s]), ph, abort_flag) ||
              !mbar_wait(smem_u32(&ctl->tempty[tb]), tph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t w0 = smem_u32(sW + s * kWBytes);
          const uint32_t b0 = smem_u32(sB + s * kBBytes);
          // each 32-wide K block into its own columns: the epilogue scales them apart
#pragma unroll
          for (int kk = 0; kk < kTK / 32; ++kk)
            umma_f8(tmem_base + tb * kBufCols + kk * kMaxN, sw128_kmajor_desc(w0 + 32u * kk),
                    sw128_kmajor_desc(b0 + 32u * kk), idesc, 0u);
          umma_commit(smem_u32(&ctl->empty[s]));
          umma_commit(smem_u32(&ctl->tfull[tb]));
          ++it;
        }
      }
      if (it > 0) drain_wait(smem_u32(&ctl->tfull[(it - 1) % kTBufs]), ((it - 1) / kTBufs) & 1u);
    }
    __syncwarp();
  } else if (warp == kLoaderWarp) {
    // ------------------------------------------------------------ route tables
    // One tile ahead of the epilogue: the tile's route id per column and the
    // column scales (two dependent global loads), so that the epilogue starts
    // a tile without a round trip to global memory.
    uint32_t tc = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      int b, wt, e, nb;
      if (!w4_tile(p, ctl, tile, nvalid, b, wt, e, nb)) continue;
      const int rows = nb * p.block_m;
      const int par = tc & 1;
      if (!warp_wait(smem_u32(&ctl->rempty[par]), ((tc >> 1) & 1u) ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      for (int c = lane; c < kMaxN; c += 32) {
        int id = -1;
        const int64_t slot = static_cast<int64_t>(b) * p.block_m + c;
        if (c < rows && MOE_IN_BOUNDS(slot < p.sorted_cap)) id = p.sorted_ids[slot];
        const bool route = id >= 0 && id < p.R;
        ctl->route[par][c] = route ? id : -1;
        ctl->cs[par][c] = route ? (p.up ? p.a_scale[id / p.top_k] : p.s_inter[id]) : 0.f;
        ctl->cw[par][c] = (route && !p.up) ? __fmul_rn(p.topk_w[id], p.routed_scale) : 0.f;
      }
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->rfull[par]));
      ++tc;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;  // weight row of the tile
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t it = 0, tc = 0;
    bool ok = true;
    for (int64_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int b, wt, e, nb;
      if (!w4_tile(p, ctl, tile, nvalid, b, wt, e, nb)) {
        if (warp == 2 && lane == 0 && wt == 0 && b < nvalid) {
          const int bad = b < kMaxBlocks ? ctl->expert[b] : p.expert_ids[b];
          if (bad != -1 && (bad < 0 || bad >= p.E) && p.status) atomicOr(p.status, MOE_DEV_BAD_EXPERT);
        }
        continue;
      }
      const int rows = nb * p.block_m;
      const int nmma = (rows + 15) & ~15;
      const int ncols = nmma / 2;           // this thread's route columns: half * ncols ..
      const int c0 = half * ncols;
      // the tile's routes and their column scales (the producer's table)
      const int par = tc & 1;
      if (ok) ok = warp_wait(smem_u32(&ctl->rfull[par]), (tc >> 1) & 1u, abort_flag);
      const int32_t* t_route = ctl->route[par];
      const float* t_cs = ctl->cs[par];
      const float* t_cw = ctl->cw[par];

      float acc[kMaxN / 2];
#pragma unroll
      for (int c = 0; c < kMaxN / 2; ++c) acc[c] = 0.f;
      for (int kb = 0; kb < p.nkb; ++kb) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1u;
        const uint32_t tb = it % kTBufs;
        const uint32_t tph = (it / kTBufs) & 1u;
        float4 sc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (ok) ok = warp_wait(smem_u32(&ctl->full[s]), ph, abort_flag);
        if (ok) sc = *reinterpret_cast<const float4*>(sS + s * kSBytes + 16 * row);
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(smem_u32(&ctl->empty[s]));
        if (ok) ok = warp_wait(smem_u32(&ctl->tfull[tb]), tph, abort_flag);
        if (ok) {
          tc_fence_after();
          const float scl[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int c8 = 0; c8 < kMaxN / 16; ++c8) {
              if (8 * c8 < ncols) {
                uint32_t v[8];
                tmem_ld_32x32b_x8(lane_base + tb * kBufCols + kk * kMaxN + c0 + 8 * c8, v);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[8 * c8 + i] = __fmaf_rn(__uint_as_float(v[i]), scl[kk], acc[8 * c8 + i]);
              }
            }
          }
          tc_fence_before();
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(smem_u32(&ctl->tempty[tb]));
        ++it;
      }

      if (p.up) {
        // g = acc * a_scale (rows 0..63), u = acc * a_scale (rows 64..127)
        if (row >= 64) {
#pragma unroll
          for (int c = 0; c < kMaxN / 2; ++c)
            if (c < ncols) ctl->xchg[row - 64][c0 + c] = __fmul_rn(acc[c], t_cs[c0 + c]);
        }
        named_barrier(1, 32 * kEpiWarps);
        if (row < 64 && ok) {
          const int j = wt * 64 + row;  // intermediate column
#pragma unroll
          for (int c = 0; c < kMaxN / 2; ++c) {
            if (c < ncols) {
              const int rt = t_route[c0 + c];
              if (rt >= 0 && MOE_IN_BOUNDS(rt < p.R && j < p.I)) {
                const float g = __fmul_rn(acc[c], t_cs[c0 + c]);
                p.h[static_cast<int64_t>(rt) * p.I + j] = __fmul_rn(silu_f32(g), ctl->xchg[row][c0 + c]);
              }
            }
          }
        }
      } else if (ok) {
        const int hcol = wt * kTM + row;  // output column
#pragma unroll
        for (int c = 0; c < kMaxN / 2; ++c) {
          if (c < ncols) {
            const int rt = t_route[c0 + c];
            if (rt >= 0 && MOE_IN_BOUNDS(rt < p.R && hcol < p.H))
              p.y[static_cast<int64_t>(rt) * p.H + hcol] =
                  __fmul_rn(__fmul_rn(acc[c], t_cs[c0 + c]), t_cw[c0 + c]);
          }
        }
      }
      // the exchange rows are rewritten by the next tile; the route table
      // goes back to the producer
      named_barrier(1, 32 * kEpiWarps);
      if (ok && lane == 0) mbar_arrive(smem_u32(&ctl->rempty[par]));
      ++tc;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0 && ctl->abort_flag && p.status) atomicOr(p.status, MOE_DEV_TIMEOUT);
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols) : "memory");
}

}  // namespace

bool w4a8_tc_supported(int H, int I, int block_m, const void* w13, const void* w2, const void* w13_scale,
                       const void* w2_scale) {
  auto al = [](const void* q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) & (a - 1)) == 0; };
  return H % 128 == 0 && I % 128 == 0 && block_m <= 64 && al(w13, 32) && al(w2, 32) && al(w13_scale, 16) &&
         al(w2_scale, 16);
}

moe_status launch_w4a8_tc_gemm(const W4GemmTensors& t, W4GemmParams p, int sms, cudaStream_t stream) {
  static bool attr_done[64] = {};
  int dev = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MOE_ERR_DEVICE;
  if (!attr_done[dev]) {
    MOE_CUDA_TRY(cudaFuncSetAttribute(w4a8_tc_gemm_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem_bytes_w4<64>())));
    MOE_CUDA_TRY(cudaFuncSetAttribute(w4a8_tc_gemm_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem_bytes_w4<32>())));
    MOE_CUDA_TRY(cudaFuncSetAttribute(w4a8_tc_gemm_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem_bytes_w4<16>())));
    attr_done[dev] = true;
  }
  // small plans (at most 16 tokens, so at most 16 routes per expert from
  // distinct top-k ids, and plan blocks of at most 16 rows) take the 16-row
  // tiles with eight TMEM buffers; other plans with blocks of at most 32 rows
  // the 32-row tiles with four -- except the gate/up projection when an
  // expert holds 16-64 routes on average, where 32-row groups would stream
  // many experts' weights twice (measured at the page's shape, forward:
  // 64 tokens 0.91 -> 0.71 ms, 1024 tokens 1.58 -> 1.54 ms, 4096 tokens
  // 6.17 -> 5.65 ms against 64-row tiles throughout)
  const bool narrow = p.block_m <= 16 && p.R <= 16 * p.top_k;
  const int64_t touched = p.R < p.E ? p.R : p.E;
  const int64_t per_expert = touched > 0 ? p.R / touched : 0;
  const bool mid = !narrow && p.block_m <= 32 && !(p.up && per_expert > 16 && per_expert <= 64);
  const int max_n = narrow ? 16 : (mid ? 32 : 64);
  // weights: packed E2M1 rows of K codes (K/2 bytes), read as 16U4_ALIGN16B
  // boxes of 128 codes x (64 or 128) rows; scales: FP32 rows of K/32, boxes
  // of 4 x rows; gathered rows: E4M3, boxes of 128 codes x 1 row.
  const uint32_t wrows = p.up ? 64u : static_cast<uint32_t>(kTM);
  CUtensorMap mw, ms, mb;
  if (encode_tensor_map_2d_typed(&mw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, t.w, t.k, t.w_total_rows, t.k / 2, kTK,
                                 wrows, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_tensor_map_2d_typed(&ms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, t.w_scale, t.k / 32, t.w_total_rows,
                                 (t.k / 32) * 4, 4, wrows, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS ||
      encode_tensor_map_2d(&mb, t.rows, t.k, t.rows_total, t.k, kTK, 1, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
    return MOE_ERR_CUDA;
  p.group = p.block_m >= max_n ? 1 : max_n / p.block_m;
  p.rows_total = static_cast<int64_t>(t.rows_total);
  p.nkb = static_cast<int>(t.k / kTK);
  const int64_t tiles = p.nblocks * p.ntw;
  if (tiles <= 0) return MOE_OK;
  const unsigned grid = static_cast<unsigned>(tiles < sms ? tiles : sms);
  if (narrow)
    w4a8_tc_gemm_kernel<16><<<grid, kThreads, smem_bytes_w4<16>(), stream>>>(mw, ms, mb, p);
  else if (mid)
    w4a8_tc_gemm_kernel<32><<<grid, kThreads, smem_bytes_w4<32>(), stream>>>(mw, ms, mb, p);
  else
    w4a8_tc_gemm_kernel<64><<<grid, kThreads, smem_bytes_w4<64>(), stream>>>(mw, ms, mb, p);
  MOE_CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}

}  // namespace moe

MOE_BOUNDS_TU()
