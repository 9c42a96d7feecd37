// The vector path of moe_fp8_block_scale_forward, for sparse plans (decode:
// one or two routes per touched expert).  With so few activation rows per
// expert both projections are matrix-vector products: two FLOP per weight
// byte and route, so their cost is the weight stream itself.  They run on
// the CUDA cores as plain 16-byte loads with FP32 FMAs instead of 128-row
// tensor-core tiles: no staging launch, no TMA ring to fill per tile, and the
// down projection lists its routes and loads its weights before it waits for
// the gate/up kernel.
//
// Launches (programmatic dependent launch between them):
//   1. vec_up_kernel: a CTA per (plan block, 4 intermediate columns).  Its
//      eight warps (4 row pairs x 2 halves of K) stream the 8 interleaved
//      W13 rows of those columns (4 gate, 4 up; a bulk L2 prefetch starts
//      them at once) against the route's activation row, converted once to
//      FP32 in shared memory; each 16-code partial is multiplied by the
//      activation and weight block scales of its 128-wide K slice, and
//      silu(gate) * up is written in FP32 for every route of the block to
//      h[route, I].  The CTA also prefetches its share of the expert's W2
//      rows into L2 for the down kernel.
//   2. vec_down_kernel: a CTA per 16 output columns, for all tokens.  It
//      reads the plan to list the held routes in route order (the plan is
//      complete before the forward starts) and loads the first routes' W2
//      rows, then waits for h, requantises each route's row to E4M3 per 128
//      columns exactly as the tensor path does (scale amax/448, codes of
//      h * (1/scale)), and adds each route's weighted down projection, in
//      route order, to f32(out); out is rounded to BF16 once.
#include <climits>

#include "common.cuh"
#include "vector.cuh"

namespace moe {
namespace {

constexpr int kUpCols = 4;        // intermediate columns per gate/up CTA
constexpr int kDnRows = 16;       // W2 rows (output columns) per down CTA: 4 warps x 4 rows
constexpr int kDnRegs = 24;       // 16-byte W2 groups a lane holds at once

__device__ __forceinline__ uint4 ld_stream(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16 E4M3 codes -> 8 registers of two exact halves each, in byte order.
__device__ __forceinline__ void e4m3x16_to_h2(const uint4 v, uint32_t (&h)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[2 * k]) : "h"(static_cast<uint16_t>(w[k] & 0xFFFFu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[2 * k + 1]) : "h"(static_cast<uint16_t>(w[k] >> 16)));
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Plan blocks [0, nvalid) can hold work: nvalid = min(P / block_m, nblocks).
__device__ __forceinline__ int64_t valid_blocks(const int32_t* num_post_padded, int block_m, int64_t nblocks) {
  int64_t P = __ldcg(num_post_padded);
  if (P < 0) P = 0;
  const int64_t n = P / block_m;
  return n < nblocks ? n : nblocks;
}

// 16 E4M3 codes -> 16 exact floats (pairs in byte order).
__device__ __forceinline__ void e4m3x16_to_f32(const uint4 v, float2 (&f)[8]) {
  uint32_t h[8];
  e4m3x16_to_h2(v, h);
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
}

// Activation rows are converted to FP32 once per CTA and kept in shared
// memory with 16 bytes of padding after every 128: a lane's 16 values of a
// 512-byte K step start at 16 lane + 4 (lane / 2), so the 8 lanes of each
// quarter-warp read 8 different 16-byte bank groups.
__device__ __forceinline__ int apos(int k) { return k + 4 * (k >> 5); }
constexpr int kUpMaxK = 8192;            // H bound of the staged activation row
constexpr int kUpWarps = 8;              // 4 row pairs x 2 halves of K

__global__ void __launch_bounds__(32 * kUpWarps, 4) vec_up_kernel(const VecUpParams p) {
  __shared__ alignas(16) float s_act[kUpMaxK + kUpMaxK / 8];   // the current route's activations
  __shared__ float s_ws[2][kUpMaxK / 128];                     // weight scales, gate and up row blocks
  __shared__ float s_as[kUpMaxK / 128];                        // the route's activation scales
  __shared__ int s_route[128];                                 // the block's routes, in slot order
  __shared__ int s_nr;
  __shared__ float s_part[2][2][kUpCols];                      // [K half][gate, up][column]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quads = p.I / kUpCols;
  const int64_t b = blockIdx.x / quads;
  const int c0 = static_cast<int>(blockIdx.x % quads) * kUpCols;
  pdl_wait();
  // the down kernel reads the plan before its own wait: release it only now
  pdl_launch_dependents();
  if (!MOE_IN_BOUNDS(b < p.nblocks)) return;
  // extent, expert and the block's route ids in one round trip (slots of
  // blocks inside the plan capacity are always readable)
  int ids[4];
  if (warp == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int sl = 32 * i + lane;
      ids[i] = sl < p.block_m ? __ldcg(p.sorted_ids + b * p.block_m + sl) : -1;
    }
  }
  const int e = __ldcg(p.expert_ids + b);
  if (b >= valid_blocks(p.num_post_padded, p.block_m, p.nblocks)) return;
  if (e < 0 || e >= p.E) {
    if (e != -1 && c0 == 0 && threadIdx.x == 0 && p.status) atomicOr(p.status, MOE_DEV_BAD_EXPERT);
    return;
  }
  const int nkb = p.H / 128;
  const uint8_t* wg = p.w13 + (static_cast<int64_t>(e) * 2 * p.I + 16 * (c0 / 8) + c0 % 8) * p.H;
  if (threadIdx.x == 32) {
    // the CTA's 4 gate and 4 up rows (two contiguous runs) start streaming
    // into L2 now, ahead of the warps' own loads
    prefetch_l2_bulk(wg, 4u * p.H);
    prefetch_l2_bulk(wg + 8 * static_cast<int64_t>(p.H), 4u * p.H);
  } else if (threadIdx.x == 64) {
    // and this CTA's share of the expert's W2 rows, which the down kernel
    // reads next (the block's quads split the expert's H x I bytes)
    const int64_t w2b = static_cast<int64_t>(p.H) * p.I;
    const int64_t share = (w2b / quads + 15) / 16 * 16;
    const int64_t off = (blockIdx.x % quads) * share;
    if (off < w2b) prefetch_l2_bulk(p.w2 + e * w2b + off, static_cast<uint32_t>(off + share <= w2b ? share : w2b - off));
  }
  if (warp == 0) {
    int n = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const bool route = ids[i] >= 0 && ids[i] < p.R;
      const unsigned m = __ballot_sync(0xffffffffu, route);
      if (route) s_route[n + __popc(m & ((1u << lane) - 1u))] = ids[i];
      n += __popc(m);
    }
    if (lane == 0) s_nr = n;
  } else if (warp <= 2) {
    // the logical gate (warp 1) and up (warp 2) row blocks of these columns
    const float* src =
        p.w13_scale + (static_cast<int64_t>(e) * (2 * p.I / 128) + ((warp - 1) * p.I + c0) / 128) * nkb;
    for (int k = lane; k < nkb; k += 32) s_ws[warp - 1][k] = __ldg(src + k);
  }
  __syncthreads();
  const int nr = s_nr;

  // warp & 3: row pair (0, 1: gate rows of columns c0 + 2 (warp & 1) + {0, 1};
  // 2, 3: the up rows of the same columns); warp >> 2: half of K.
  // Interleaved W13 holds groups of 16 rows: 8 gate rows, then the 8 up rows
  // of the same columns.
  const int kind = (warp >> 1) & 1, half = warp >> 2;
  const uint8_t* w0 = wg + (8 * kind + 2 * (warp & 1)) * static_cast<int64_t>(p.H) + 16 * lane;
  const uint8_t* w1 = w0 + p.H;
  const int msteps = (p.H + 511) / 512;
  const int mh = (msteps + 1) / 2;
  const int m_lo = half * mh, m_hi = half ? msteps : mh;
  const int g8 = lane >> 3;  // the lane's 16 bytes of a 512-byte step lie in slice 4 m + g8

  for (int ri = 0; ri < nr; ++ri) {
    const int route = s_route[ri];
    const int64_t tok = route / p.top_k;
    // the route's activation row and scales, converted once
    const uint4* arow = reinterpret_cast<const uint4*>(p.a + tok * p.H);
    for (int c = threadIdx.x; c < p.H / 16; c += blockDim.x) {
      float2 f[8];
      e4m3x16_to_f32(__ldg(arow + c), f);
      float4* dst = reinterpret_cast<float4*>(&s_act[apos(16 * c)]);
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[i] = make_float4(f[2 * i].x, f[2 * i].y, f[2 * i + 1].x, f[2 * i + 1].y);
    }
    for (int k = threadIdx.x; k < nkb; k += blockDim.x) s_as[k] = __ldg(p.a_scale + tok * nkb + k);
    __syncthreads();
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 2
    for (int m = m_lo; m < m_hi; ++m) {
      const int kb = 4 * m + g8;
      if (kb < nkb) {
        const int64_t off = 512 * static_cast<int64_t>(m);
        float2 f0[8], f1[8];
        e4m3x16_to_f32(ld_stream(w0 + off), f0);
        e4m3x16_to_f32(ld_stream(w1 + off), f1);
        const float4* av = reinterpret_cast<const float4*>(&s_act[apos(512 * m + 16 * lane)]);
        float2 d0a = make_float2(0.f, 0.f), d0b = d0a, d1a = d0a, d1b = d0a;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 a4 = av[i];
          const float2 alo = make_float2(a4.x, a4.y), ahi = make_float2(a4.z, a4.w);
          d0a = __ffma2_rn(f0[2 * i], alo, d0a);
          d0b = __ffma2_rn(f0[2 * i + 1], ahi, d0b);
          d1a = __ffma2_rn(f1[2 * i], alo, d1a);
          d1b = __ffma2_rn(f1[2 * i + 1], ahi, d1b);
        }
        const float sc = __fmul_rn(s_as[kb], s_ws[kind][kb]);
        acc0 = fmaf((d0a.x + d0a.y) + (d0b.x + d0b.y), sc, acc0);
        acc1 = fmaf((d1a.x + d1a.y) + (d1b.x + d1b.y), sc, acc1);
      }
    }
    acc0 = warp_sum(acc0);
    acc1 = warp_sum(acc1);
    if (lane == 0) {
      s_part[half][kind][2 * (warp & 1)] = acc0;
      s_part[half][kind][2 * (warp & 1) + 1] = acc1;
    }
    __syncthreads();
    if (threadIdx.x < kUpCols) {
      const int c = threadIdx.x;
      const float g = s_part[0][0][c] + s_part[1][0][c];
      const float u = s_part[0][1][c] + s_part[1][1][c];
      if (MOE_IN_BOUNDS(route < p.R && c0 + c < p.I))
        p.h[static_cast<int64_t>(route) * p.I + c0 + c] = __fmul_rn(silu_f32(g), u);
    }
    // s_act, s_as and s_part are rewritten for the next route
    __syncthreads();
  }
}

// Shared memory of the down kernel.  The route map is needed only while the
// list of held routes is built, the requantised intermediate only afterwards.
struct HeldRoute {
  int route, slot, expert;
  float weight;  // topk_weights[route] * routed_scale
};
// The requantised intermediate is kept as exact floats in the padded layout
// of the activation rows: a lane's 16 values of W2 group g = l8 + 8u start at
// apos(16 g), so the 8 lanes of a row read 8 different 16-byte bank groups.
template <int kU>
struct DownSmem {
  static constexpr int kJB = kDnRegs / kU;  // routes per batch
  union {
    unsigned long long map[kVecMaxRoutes];  // (slot << 32 | expert) of each route, smallest slot
    struct {
      alignas(16) float q[kJB][144 * kU];   // the batch's requantised intermediate (exact floats)
      float s[kJB][kU];                     // and its scales
    } b;
  } u;
  HeldRoute held[kVecMaxRoutes];
  float weight[kVecMaxRoutes];        // topk_weights * routed_scale of every route
  float acc[kVecMaxTokens][kDnRows];  // f32(out) plus the contributions so far
  int nheld;
  int wcount[4];
};

template <int kU>
__global__ void __launch_bounds__(128) vec_down_kernel(const VecDownParams p) {
  constexpr int kJB = DownSmem<kU>::kJB;
  constexpr int kRq = (kJB + 3) / 4;  // routes a warp requantises per batch
  __shared__ DownSmem<kU> sm;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int l8 = lane & 7;
  const int row0 = blockIdx.x * kDnRows;
  const int row = row0 + 4 * warp + (lane >> 3);
  const bool rowok = row < p.H;
  const int nthreads = blockDim.x;

  // 1. Routes the plan holds (read before the wait: the plan is an input,
  //    complete before the gate/up kernel released this grid).
  for (int r = threadIdx.x; r < p.R; r += nthreads) {
    sm.u.map[r] = ~0ull;
    sm.weight[r] = __fmul_rn(__ldcg(p.topk_w + r), p.routed_scale);
  }
  if (threadIdx.x == 0) sm.nheld = 0;
  __syncthreads();
  // every slot of the plan's capacity is read, eight per thread at a time,
  // with the extent loaded alongside and checked afterwards
  {
    constexpr int kScan = 8;
    const int64_t P = __ldcg(p.num_post_padded);
    const int64_t cap_slots = p.nblocks * p.block_m;
    for (int64_t s0 = threadIdx.x; s0 < cap_slots; s0 += kScan * nthreads) {
      int id[kScan], ex[kScan];
#pragma unroll
      for (int k = 0; k < kScan; ++k) {
        const int64_t sl = s0 + k * nthreads;
        id[k] = sl < cap_slots ? __ldcg(p.sorted_ids + sl) : -1;
        ex[k] = sl < cap_slots ? __ldcg(p.expert_ids + sl / p.block_m) : -1;
      }
      int64_t nvalid = (P < 0 ? 0 : P) / p.block_m;
      if (nvalid > p.nblocks) nvalid = p.nblocks;
#pragma unroll
      for (int k = 0; k < kScan; ++k) {
        const int64_t sl = s0 + k * nthreads;
        if (sl < nvalid * p.block_m && id[k] >= 0 && id[k] < p.R && ex[k] >= 0 && ex[k] < p.E)
          atomicMin(&sm.u.map[id[k]], (static_cast<unsigned long long>(sl) << 32) | static_cast<uint32_t>(ex[k]));
      }
    }
  }
  __syncthreads();
  // compact in route order (token-major), 128 routes per round
  for (int base = 0; base < p.R; base += nthreads) {
    const int r = base + threadIdx.x;
    const unsigned long long v = r < p.R ? sm.u.map[r] : ~0ull;
    const bool held = v != ~0ull;
    const unsigned m = __ballot_sync(0xffffffffu, held);
    if (lane == 0) sm.wcount[warp] = __popc(m);
    __syncthreads();
    int off = sm.nheld;
    for (int w = 0; w < warp; ++w) off += sm.wcount[w];
    if (held) {
      HeldRoute h;
      h.route = r;
      h.slot = static_cast<int>(v >> 32);
      h.expert = static_cast<int>(v & 0xFFFFFFFFu);
      h.weight = sm.weight[r];
      sm.held[off + __popc(m & ((1u << lane) - 1u))] = h;
    }
    __syncthreads();
    if (threadIdx.x == 0) sm.nheld += sm.wcount[0] + sm.wcount[1] + sm.wcount[2] + sm.wcount[3];
    __syncthreads();
  }
  const int nh = sm.nheld;
  // every held route's 16 W2 rows of this CTA (one contiguous run each)
  // start streaming into L2; the first batch also goes to registers below
  for (int j = threadIdx.x; j < nh; j += nthreads) {
    const int rows = p.H - row0 < kDnRows ? p.H - row0 : kDnRows;
    prefetch_l2_bulk(p.w2 + (static_cast<int64_t>(sm.held[j].expert) * p.H + row0) * p.I,
                     static_cast<uint32_t>(rows * p.I));
  }

  // 2. W2 rows of a batch of held routes: group u of the lane is bytes
  //    16 (l8 + 8 u) .. + 16 of `row` (K slice u), 128 contiguous bytes per
  //    row for the 8 lanes.
  uint4 wv[kJB][kU];
  float wsc[kJB][kU];
  auto load_batch = [&](int j0) {
#pragma unroll
    for (int jj = 0; jj < kJB; ++jj) {
      const int j = j0 + jj;
      const bool live = j < nh && rowok;
      const int e = live ? sm.held[j].expert : 0;
      const uint8_t* src = p.w2 + (static_cast<int64_t>(e) * p.H + row) * p.I + 16 * l8;
      const float* scs = p.w2_scale + (static_cast<int64_t>(e) * (p.H / 128) + row / 128) * kU;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        wv[jj][u] = live ? ld_stream(src + 128 * u) : make_uint4(0u, 0u, 0u, 0u);
        wsc[jj][u] = live ? __ldg(scs + u) : 0.f;
      }
    }
  };
  load_batch(0);

  pdl_wait();
  pdl_launch_dependents();

  const int64_t tok_lo = nh > 0 ? sm.held[0].route / p.top_k : 0;
  const int ntok = nh > 0 ? static_cast<int>(sm.held[nh - 1].route / p.top_k - tok_lo) + 1 : 0;
  if (!MOE_IN_BOUNDS(ntok <= kVecMaxTokens)) return;  // (uniform over the CTA)

  for (int j0 = 0; j0 < nh; j0 += kJB) {
    if (j0 > 0) {
      load_batch(j0);
      __syncthreads();  // the previous batch's q is no longer read
    }
    // 3. the batch's intermediate rows (a warp per route), every row's loads
    //    issued before any is used
    const int nb = nh - j0 < kJB ? nh - j0 : kJB;
    float4 hv[kRq][kU];
#pragma unroll
    for (int i = 0; i < kRq; ++i) {
      const int jj = warp + 4 * i;
      int hr_route = jj < nb ? sm.held[j0 + jj].route : 0;
      if (!MOE_IN_BOUNDS(hr_route >= 0 && hr_route < p.R)) hr_route = 0;
      const float* hrow = p.h + static_cast<int64_t>(hr_route) * p.I;
#pragma unroll
      for (int g = 0; g < kU; ++g)
        hv[i][g] = jj < nb ? __ldcg(reinterpret_cast<const float4*>(hrow + 128 * g) + lane)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (j0 == 0) {
      // f32(out) of every token of the list, for this CTA's rows (these
      // loads overlap the ones above; the barrier after the requant
      // publishes them)
      for (int i = threadIdx.x; i < ntok * kDnRows; i += nthreads) {
        const int tt = i / kDnRows, rr = i % kDnRows;
        const int orow = row0 + rr;
        sm.acc[tt][rr] =
            orow < p.H ? __bfloat162float(__ushort_as_bfloat16(p.out[(tok_lo + tt) * p.H + orow])) : 0.f;
      }
    }
    // 4. requantise
#pragma unroll
    for (int i = 0; i < kRq; ++i) {
      const int jj = warp + 4 * i;
      if (jj < nb) {
        const int slot = sm.held[j0 + jj].slot;
#pragma unroll
        for (int g = 0; g < kU; ++g) {
          const float4 v = hv[i][g];
          float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          const float s = __fdiv_rn(amax, 448.0f);
          const float inv = s > 0.f ? __frcp_rn(s) : 0.f;
          const uint16_t lo = cvt_e4m3x2(__fmul_rn(v.x, inv), __fmul_rn(v.y, inv));
          const uint16_t hi = cvt_e4m3x2(__fmul_rn(v.z, inv), __fmul_rn(v.w, inv));
          const float2 qlo = e4m3x2_to_f32(lo), qhi = e4m3x2_to_f32(hi);
          *reinterpret_cast<float4*>(&sm.u.b.q[jj][apos(128 * g + 4 * lane)]) =
              make_float4(qlo.x, qlo.y, qhi.x, qhi.y);
          if (lane == 0) sm.u.b.s[jj][g] = s;
          if (p.dbg_q && blockIdx.x == 0 && MOE_IN_BOUNDS(slot >= 0 && slot < p.nblocks * p.block_m)) {
            *reinterpret_cast<uint32_t*>(p.dbg_q + static_cast<int64_t>(slot) * p.I + 128 * g + 4 * lane) =
                static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            if (lane == 0) p.dbg_s[static_cast<int64_t>(slot) * kU + g] = s;
          }
        }
      }
    }
    __syncthreads();
    // 5. the batch's contributions, in route order
#pragma unroll
    for (int jj = 0; jj < kJB; ++jj) {
      if (jj < nb) {
        float y = 0.f;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const float4* q4 = reinterpret_cast<const float4*>(&sm.u.b.q[jj][apos(16 * (l8 + 8 * u))]);
          float2 wf[8];
          e4m3x16_to_f32(wv[jj][u], wf);
          float2 da = make_float2(0.f, 0.f), db = da;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 q = q4[i];
            da = __ffma2_rn(wf[2 * i], make_float2(q.x, q.y), da);
            db = __ffma2_rn(wf[2 * i + 1], make_float2(q.z, q.w), db);
          }
          y = fmaf((da.x + da.y) + (db.x + db.y), __fmul_rn(sm.u.b.s[jj][u], wsc[jj][u]), y);
        }
        y += __shfl_xor_sync(0xffffffffu, y, 1);
        y += __shfl_xor_sync(0xffffffffu, y, 2);
        y += __shfl_xor_sync(0xffffffffu, y, 4);
        const HeldRoute hr = sm.held[j0 + jj];
        if (l8 == 0 && rowok && MOE_IN_BOUNDS(hr.route / p.top_k - tok_lo >= 0 && hr.route / p.top_k - tok_lo < ntok)) {
          float& a = sm.acc[hr.route / p.top_k - tok_lo][4 * warp + (lane >> 3)];
          a = __fadd_rn(a, __fmul_rn(y, hr.weight));
        }
      }
    }
  }
  __syncthreads();
  // 6. out = bf16_rn(acc) for the tokens from the first to the last with a held route
  for (int i = threadIdx.x; i < ntok * kDnRows; i += nthreads) {
    const int tt = i / kDnRows, rr = i % kDnRows;
    const int orow = row0 + rr;
    if (orow < p.H && MOE_IN_BOUNDS(static_cast<int64_t>(tok_lo + tt) * p.top_k < p.R))
      p.out[(tok_lo + tt) * p.H + orow] = __bfloat16_as_ushort(__float2bfloat16_rn(sm.acc[tt][rr]));
  }
}

}  // namespace

bool vector_path_supported(int64_t M, int64_t R, int H, int I) {
  return R >= 1 && R <= kVecMaxRoutes && M <= kVecMaxTokens && H <= kUpMaxK && I % 128 == 0 && I / 128 <= 8;
}

moe_status launch_vector_path(const VecUpParams& up, const VecDownParams& dn, cudaStream_t stream,
                              cudaEvent_t const* ev) {
  const int64_t up_grid = up.nblocks * (up.I / kUpCols);
  if (up_grid > 0x7FFFFFFF) return MOE_ERR_SHAPE;
  if (ev) MOE_CUDA_TRY(cudaEventRecord(ev[1], stream));  // no staging launch
  MOE_CUDA_TRY(
      launch_pdl(vec_up_kernel, dim3(static_cast<unsigned>(up_grid)), dim3(32 * kUpWarps), 0, stream, 1, up));
  if (ev) MOE_CUDA_TRY(cudaEventRecord(ev[2], stream));
  const dim3 dgrid(static_cast<unsigned>(ceil_div(dn.H, kDnRows)));
  cudaError_t err = cudaErrorInvalidValue;
  switch (dn.I / 128) {
    case 1: err = launch_pdl(vec_down_kernel<1>, dgrid, dim3(128), 0, stream, 1, dn); break;
    case 2: err = launch_pdl(vec_down_kernel<2>, dgrid, dim3(128), 0, stream, 1, dn); break;
    case 3: err = launch_pdl(vec_down_kernel<3>, dgrid, dim3(128), 0, stream, 1, dn); break;
    case 4: err = launch_pdl(vec_down_kernel<4>, dgrid, dim3(128), 0, stream, 1, dn); break;
    case 5: err = launch_pdl(vec_down_kernel<5>, dgrid, dim3(128), 0, stream, 1, dn); break;
    case 6: err = launch_pdl(vec_down_kernel<6>, dgrid, dim3(128), 0, stream, 1, dn); break;
    case 7: err = launch_pdl(vec_down_kernel<7>, dgrid, dim3(128), 0, stream, 1, dn); break;
    case 8: err = launch_pdl(vec_down_kernel<8>, dgrid, dim3(128), 0, stream, 1, dn); break;
    default: return MOE_ERR_SHAPE;
  }
  MOE_CUDA_TRY(err);
  if (ev) MOE_CUDA_TRY(cudaEventRecord(ev[3], stream));
  return MOE_OK;
}

}  // namespace moe

MOE_BOUNDS_TU()
