// E2M1-K32 weight x FP8 activation variant of the expert computation
// (sglang-glm53-flash-sm120 pull request #13, "SM120 FP8 prefill",
// description): E2M1 weight codes with one FP32 scale per 32 elements of K,
// applied in FP32, and E4M3 activations with one FP32 scale per row.
//
// Where the sizes allow (H and I multiples of 128, plan blocks of at most 64
// rows), the two projections run on the tensor cores (w4a8_tc.cu) and the
// requant and combine kernels below complete the forward.  Otherwise, or on
// request (MOE_W4A8_CUDA_CORES), the projections run on the CUDA cores; each
// CTA of the first three kernels takes one plan block (in the projections,
// and a group of columns):
//   w4a8_up_kernel       gate/up rows of the block's expert against the block's
//                        activation rows (staged in shared memory), SwiGLU;
//   w4a8_requant_kernel  each route's SwiGLU row requantised to E4M3 with one
//                        scale per row;
//   w4a8_down_kernel     W2 rows against the requantised rows, times the route
//                        weight: one FP32 contribution row per route;
//   w4a8_combine_kernel  each token's contributions added in slot order onto
//                        f32(out), rounded once to BF16.
// In the two projections a warp takes a column and its lanes the 32-wide K
// blocks (lane, lane + 32, ...): one 16-byte load of packed weight codes and
// one scale per block, the codes decoded once per chunk of kRowChunk rows,
// whose partial sums stay in registers until a warp reduction.
#include "common.cuh"
#include "w4a8_tc.cuh"
#include "../../include/moe_w4a8.h"

namespace moe {
namespace {

constexpr int kW4Threads = 256;
constexpr int kW4Warps = kW4Threads / 32;
constexpr int kRowChunk = 8;           // rows whose partial sums a lane holds at once
constexpr int kUpColsPerWarp = 2;      // gate/up column pairs per warp
constexpr int kUpCols = kW4Warps * kUpColsPerWarp;
constexpr int kDownColsPerWarp = 4;    // output columns per warp
constexpr int kDownCols = kW4Warps * kDownColsPerWarp;
constexpr int kW4MaxBlockM = 64;
constexpr int kW4MaxRowBytes = 128 * 1024;  // shared-memory rows of one plan block

__device__ __forceinline__ float bf16_to_f32(uint32_t bits) { return __uint_as_float(bits << 16); }

// E2M1 code (low 4 bits of c) -> value.  The magnitudes 0, 0.5, 1, 1.5, 2,
// 3, 4, 6 are 0, 1, 2, 3, 4, 6, 8, 12 halves, one per nibble of 0xC8643210;
// bit 3 is the sign.
__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
  const float mag = static_cast<float>((0xC8643210u >> ((c & 7u) * 4u)) & 0xFu) * 0.5f;
  return (c & 8u) ? -mag : mag;
}

// Nearest E2M1 code to v, ties to the even mantissa, saturating at 6, sign
// kept.  The midpoints between neighbouring magnitudes are 0.25, 0.75, 1.25,
// 1.75, 2.5, 3.5 and 5; a tie goes to whichever neighbour has mantissa bit 0
// (0, 1, 2 and 4 rather than 0.5, 1.5, 3 and 6).
__device__ __forceinline__ uint32_t f32_to_e2m1(float v) {
  const float a = fabsf(v);
  uint32_t m;
  if (a <= 0.25f) m = 0;
  else if (a < 0.75f) m = 1;
  else if (a <= 1.25f) m = 2;
  else if (a < 1.75f) m = 3;
  else if (a <= 2.5f) m = 4;
  else if (a < 3.5f) m = 5;
  else if (a <= 5.0f) m = 6;
  else m = 7;
  return (signbit(v) ? 8u : 0u) | m;
}

// 32 packed E2M1 codes (element 8q + n in nibble n of word q) -> values.
__device__ __forceinline__ void decode_e2m1x32(const uint4 v, float (&w)[32]) {
  const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int n = 0; n < 8; ++n) w[8 * q + n] = e2m1_to_f32(wd[q] >> (4 * n));
}

// 16 E4M3 codes (element 4q + i in byte i of word q) -> values.
__device__ __forceinline__ void decode_e4m3x16(const uint4 v, float* x) {
  const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 lo = e4m3x2_to_f32(static_cast<uint16_t>(wd[q] & 0xFFFFu));
    const float2 hi = e4m3x2_to_f32(static_cast<uint16_t>(wd[q] >> 16));
    x[4 * q] = lo.x;
    x[4 * q + 1] = lo.y;
    x[4 * q + 2] = hi.x;
    x[4 * q + 3] = hi.y;
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = red[0];
  for (int w = 1; w < kW4Warps; ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  return m;
}

// ---------------------------------------------------------------- quantisers

// One CTA per row: amax over the row, scale = amax / 448, codes E4M3(x / scale).
__global__ void __launch_bounds__(kW4Threads) quant_act_row_kernel(const uint16_t* __restrict__ x, int K,
                                                                   uint8_t* __restrict__ q,
                                                                   float* __restrict__ scale) {
  __shared__ float red[kW4Warps];
  const int64_t m = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + m * K);   // 8 values per uint4
  const int n8 = K / 8;
  float amax = 0.f;
  for (int i = threadIdx.x; i < n8; i += kW4Threads) {
    const uint4 v = xr[i];
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      amax = fmaxf(amax, fmaxf(fabsf(bf16_to_f32(wd[k] & 0xFFFFu)), fabsf(bf16_to_f32(wd[k] >> 16))));
  }
  amax = block_max(amax, red);
  const float s = __fdiv_rn(amax, 448.0f);
  uint2* qr = reinterpret_cast<uint2*>(q + m * K);               // 8 codes per uint2
  for (int i = threadIdx.x; i < n8; i += kW4Threads) {
    const uint4 v = xr[i];
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    uint32_t c[4] = {0u, 0u, 0u, 0u};
    if (s > 0.f) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        c[k] = cvt_e4m3x2(__fdiv_rn(bf16_to_f32(wd[k] & 0xFFFFu), s), __fdiv_rn(bf16_to_f32(wd[k] >> 16), s));
    }
    qr[i] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  }
  if (threadIdx.x == 0) scale[m] = s;
}

// One thread per 32-element block: amax, scale = amax / 6, codes E2M1(w / scale)
// packed into 16 bytes.
__global__ void __launch_bounds__(kW4Threads) quant_weight_k32_kernel(const uint16_t* __restrict__ w, int64_t nblk,
                                                                      uint8_t* __restrict__ q,
                                                                      float* __restrict__ scale) {
  const int64_t blk = blockIdx.x * static_cast<int64_t>(kW4Threads) + threadIdx.x;
  if (blk >= nblk) return;
  const uint4* src = reinterpret_cast<const uint4*>(w + blk * 32);
  float v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 u = src[i];
    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[8 * i + 2 * k] = bf16_to_f32(wd[k] & 0xFFFFu);
      v[8 * i + 2 * k + 1] = bf16_to_f32(wd[k] >> 16);
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const float s = __fdiv_rn(amax, 6.0f);
  uint32_t out[4] = {0u, 0u, 0u, 0u};
  if (s > 0.f) {
#pragma unroll
    for (int i = 0; i < 32; ++i) out[i / 8] |= f32_to_e2m1(__fdiv_rn(v[i], s)) << (4 * (i % 8));
  }
  reinterpret_cast<uint4*>(q)[blk] = make_uint4(out[0], out[1], out[2], out[3]);
  scale[blk] = s;
}

// ---------------------------------------------------------------- forward

struct W4Layout {
  size_t rv_off, h_off, q_off, s_off, y_off, total;
};

W4Layout w4_layout(int64_t M, int H, int I, int top_k) {
  const int64_t R = M * top_k;
  W4Layout l{};
  size_t off = 0;
  auto take = [&](int64_t bytes) {
    const size_t o = off;
    off += static_cast<size_t>(round_up(bytes, 256));
    return o;
  };
  l.rv_off = take(R * 4);
  l.h_off = take(R * static_cast<int64_t>(I) * 4);
  l.q_off = take(R * static_cast<int64_t>(I));
  l.s_off = take(R * 4);
  l.y_off = take(R * static_cast<int64_t>(H) * 4);
  l.total = off;
  return l;
}

struct W4Plan {
  const int32_t* sorted_ids;
  const int32_t* expert_ids;
  const int32_t* ntpp;
  int R, top_k, block_m, E;
  int64_t sorted_cap;  // entries of sorted_ids
  int64_t nblocks;     // entries of expert_ids
};

// The plan block's expert (or -1 when the block holds no work) and its valid
// rows: s_rid[0 .. nv) are the route ids in slot order.
__device__ __forceinline__ int block_rows(const W4Plan& pl, int b, int* s_rid, int* s_nv, int32_t* status,
                                          bool report) {
  const int64_t P = *pl.ntpp;
  if (static_cast<int64_t>(b) * pl.block_m >= P) return -1;
  if (!MOE_IN_BOUNDS(b < pl.nblocks)) return -1;
  const int e = pl.expert_ids[b];
  if (e < 0 || e >= pl.E) {
    if (report && e != -1 && threadIdx.x == 0 && status) atomicOr(status, MOE_DEV_BAD_EXPERT);
    return -1;
  }
  if (threadIdx.x == 0) {
    int nv = 0;
    for (int r = 0; r < pl.block_m; ++r) {
      const int64_t slot = static_cast<int64_t>(b) * pl.block_m + r;
      if (slot >= P) break;
      if (!MOE_IN_BOUNDS(slot < pl.sorted_cap && nv < kW4MaxBlockM)) break;
      const int id = pl.sorted_ids[slot];
      if (id >= 0 && id < pl.R) s_rid[nv++] = id;
    }
    *s_nv = nv;
  }
  __syncthreads();
  return e;
}

struct W4UpParams {
  W4Plan pl;
  const uint8_t* a;
  const float* a_scale;
  const uint8_t* w13;
  const float* w13_scale;
  float* h;                // [R, I]
  int32_t* status;
  int H, I;
};

// grid (blocks, I / kUpCols); dynamic shared memory block_m * H bytes.
__global__ void __launch_bounds__(kW4Threads) w4a8_up_kernel(const W4UpParams p) {
  extern __shared__ __align__(16) uint8_t act[];
  __shared__ int s_rid[kW4MaxBlockM];
  __shared__ float s_as[kW4MaxBlockM];
  __shared__ int s_nv;
  const int e = block_rows(p.pl, blockIdx.x, s_rid, &s_nv, p.status, blockIdx.y == 0);
  if (e < 0) return;
  const int nv = s_nv;
  if (nv == 0) return;
  const int H = p.H, I = p.I;
  const int chunks = H / 16;
  for (int i = threadIdx.x; i < nv * chunks; i += kW4Threads) {
    const int r = i / chunks, c = i - r * chunks;
    const int64_t t = s_rid[r] / p.pl.top_k;
    reinterpret_cast<uint4*>(act)[i] = reinterpret_cast<const uint4*>(p.a + t * H)[c];
  }
  if (threadIdx.x < nv) s_as[threadIdx.x] = p.a_scale[s_rid[threadIdx.x] / p.pl.top_k];
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = H / 32;
  const int64_t N = 2 * static_cast<int64_t>(I);
  for (int cw = 0; cw < kUpColsPerWarp; ++cw) {
    const int j = blockIdx.y * kUpCols + warp * kUpColsPerWarp + cw;
    const int64_t rg = static_cast<int64_t>(e) * N + j, ru = rg + I;
    const uint4* wg = reinterpret_cast<const uint4*>(p.w13 + rg * (H / 2));
    const uint4* wu = reinterpret_cast<const uint4*>(p.w13 + ru * (H / 2));
    const float* sg = p.w13_scale + rg * nkb;
    const float* su = p.w13_scale + ru * nkb;
    for (int r0 = 0; r0 < nv; r0 += kRowChunk) {
      float ag[kRowChunk], au[kRowChunk];
#pragma unroll
      for (int rr = 0; rr < kRowChunk; ++rr) ag[rr] = au[rr] = 0.f;
      for (int kb = lane; kb < nkb; kb += 32) {
        float gw[32], uw[32];
        decode_e2m1x32(wg[kb], gw);
        decode_e2m1x32(wu[kb], uw);
        const float gs = sg[kb], us = su[kb];
#pragma unroll
        for (int rr = 0; rr < kRowChunk; ++rr) {
          if (r0 + rr < nv) {
            const uint4* ar = reinterpret_cast<const uint4*>(act + static_cast<size_t>(r0 + rr) * H + 32 * kb);
            float x[32];
            decode_e4m3x16(ar[0], x);
            decode_e4m3x16(ar[1], x + 16);
            float dg = 0.f, du = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              dg = fmaf(x[i], gw[i], dg);
              du = fmaf(x[i], uw[i], du);
            }
            ag[rr] = __fadd_rn(ag[rr], __fmul_rn(dg, gs));
            au[rr] = __fadd_rn(au[rr], __fmul_rn(du, us));
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < kRowChunk; ++rr) {
        if (r0 + rr < nv) {
          const float g = warp_sum(ag[rr]), u = warp_sum(au[rr]);
          if (lane == 0 && MOE_IN_BOUNDS(j < I)) {
            const float as = s_as[r0 + rr];
            const float gv = __fmul_rn(g, as), uv = __fmul_rn(u, as);
            p.h[static_cast<int64_t>(s_rid[r0 + rr]) * I + j] = __fmul_rn(silu_f32(gv), uv);
          }
        }
      }
    }
  }
}

struct W4RequantParams {
  W4Plan pl;
  const float* h;
  uint8_t* q;              // [R, I]
  float* s;                // [R]
  int32_t* rvalid;         // [R]
  uint8_t* dbg_q;          // nullable [sorted_cap, I]
  float* dbg_s;            // nullable [sorted_cap]
  int I;
};

// grid (blocks): each valid row of the block, one after another.
__global__ void __launch_bounds__(kW4Threads) w4a8_requant_kernel(const W4RequantParams p) {
  __shared__ float red[kW4Warps];
  const int b = blockIdx.x;
  const int64_t P = *p.pl.ntpp;
  if (static_cast<int64_t>(b) * p.pl.block_m >= P) return;
  if (!MOE_IN_BOUNDS(b < p.pl.nblocks)) return;
  const int e = p.pl.expert_ids[b];
  if (e < 0 || e >= p.pl.E) return;
  const int I = p.I;
  for (int r = 0; r < p.pl.block_m; ++r) {
    const int64_t slot = static_cast<int64_t>(b) * p.pl.block_m + r;
    if (slot >= P) break;
    if (!MOE_IN_BOUNDS(slot < p.pl.sorted_cap)) break;
    const int id = p.pl.sorted_ids[slot];
    if (id < 0 || id >= p.pl.R) continue;            // the same for every thread of the CTA
    const float* hr = p.h + static_cast<int64_t>(id) * I;
    float amax = 0.f;
    for (int i = threadIdx.x; i < I; i += kW4Threads) amax = fmaxf(amax, fabsf(hr[i]));
    amax = block_max(amax, red);
    const float s = __fdiv_rn(amax, 448.0f);
    uint8_t* qr = p.q + static_cast<int64_t>(id) * I;
    for (int i = 2 * threadIdx.x; i < I; i += 2 * kW4Threads) {
      uint16_t c = 0;
      if (s > 0.f) c = cvt_e4m3x2(__fdiv_rn(hr[i], s), __fdiv_rn(hr[i + 1], s));
      *reinterpret_cast<uint16_t*>(qr + i) = c;
      if (p.dbg_q) *reinterpret_cast<uint16_t*>(p.dbg_q + slot * I + i) = c;
    }
    if (threadIdx.x == 0) {
      p.s[id] = s;
      p.rvalid[id] = 1;
      if (p.dbg_s) p.dbg_s[slot] = s;
    }
  }
}

struct W4DownParams {
  W4Plan pl;
  const uint8_t* q;
  const float* s;
  const uint8_t* w2;
  const float* w2_scale;
  const float* topk_w;
  float* y;                // [R, H]
  int H, I;
  float routed_scale;
};

// grid (blocks, H / kDownCols); dynamic shared memory block_m * I bytes.
__global__ void __launch_bounds__(kW4Threads) w4a8_down_kernel(const W4DownParams p) {
  extern __shared__ __align__(16) uint8_t qs[];
  __shared__ int s_rid[kW4MaxBlockM];
  __shared__ float s_s[kW4MaxBlockM];
  __shared__ float s_w[kW4MaxBlockM];
  __shared__ int s_nv;
  const int e = block_rows(p.pl, blockIdx.x, s_rid, &s_nv, nullptr, false);
  if (e < 0) return;
  const int nv = s_nv;
  if (nv == 0) return;
  const int H = p.H, I = p.I;
  const int chunks = I / 16;
  for (int i = threadIdx.x; i < nv * chunks; i += kW4Threads) {
    const int r = i / chunks, c = i - r * chunks;
    reinterpret_cast<uint4*>(qs)[i] = reinterpret_cast<const uint4*>(p.q + static_cast<int64_t>(s_rid[r]) * I)[c];
  }
  if (threadIdx.x < nv) {
    const int id = s_rid[threadIdx.x];
    s_s[threadIdx.x] = p.s[id];
    s_w[threadIdx.x] = __fmul_rn(p.topk_w[id], p.routed_scale);
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = I / 32;
  for (int cw = 0; cw < kDownColsPerWarp; ++cw) {
    const int hh = blockIdx.y * kDownCols + warp * kDownColsPerWarp + cw;
    const int64_t row = static_cast<int64_t>(e) * H + hh;
    const uint4* wr = reinterpret_cast<const uint4*>(p.w2 + row * (I / 2));
    const float* sr = p.w2_scale + row * nkb;
    for (int r0 = 0; r0 < nv; r0 += kRowChunk) {
      float acc[kRowChunk];
#pragma unroll
      for (int rr = 0; rr < kRowChunk; ++rr) acc[rr] = 0.f;
      for (int kb = lane; kb < nkb; kb += 32) {
        float w[32];
        decode_e2m1x32(wr[kb], w);
        const float ws = sr[kb];
#pragma unroll
        for (int rr = 0; rr < kRowChunk; ++rr) {
          if (r0 + rr < nv) {
            const uint4* xr = reinterpret_cast<const uint4*>(qs + static_cast<size_t>(r0 + rr) * I + 32 * kb);
            float x[32];
            decode_e4m3x16(xr[0], x);
            decode_e4m3x16(xr[1], x + 16);
            float d = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) d = fmaf(x[i], w[i], d);
            acc[rr] = __fadd_rn(acc[rr], __fmul_rn(d, ws));
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < kRowChunk; ++rr) {
        if (r0 + rr < nv) {
          const float v = warp_sum(acc[rr]);
          if (lane == 0 && MOE_IN_BOUNDS(hh < H)) {
            const float yv = __fmul_rn(v, s_s[r0 + rr]);
            p.y[static_cast<int64_t>(s_rid[r0 + rr]) * H + hh] = __fmul_rn(yv, s_w[r0 + rr]);
          }
        }
      }
    }
  }
}

// grid (M, ceil(H / (4 * 256))): four columns of one token per thread.
__global__ void __launch_bounds__(kW4Threads) w4a8_combine_kernel(uint16_t* __restrict__ out,
                                                                  const float* __restrict__ y,
                                                                  const int32_t* __restrict__ rvalid, int H,
                                                                  int top_k) {
  const int64_t t = blockIdx.x;
  const int c = 4 * (blockIdx.y * kW4Threads + threadIdx.x);
  if (c >= H) return;
  uint2* op = reinterpret_cast<uint2*>(out + t * H + c);
  const uint2 raw = *op;
  float acc[4] = {bf16_to_f32(raw.x & 0xFFFFu), bf16_to_f32(raw.x >> 16), bf16_to_f32(raw.y & 0xFFFFu),
                  bf16_to_f32(raw.y >> 16)};
  for (int j = 0; j < top_k; ++j) {
    const int64_t id = t * top_k + j;
    if (!rvalid[id]) continue;
    const float4 v = *reinterpret_cast<const float4*>(y + id * H + c);
    acc[0] = __fadd_rn(acc[0], v.x);
    acc[1] = __fadd_rn(acc[1], v.y);
    acc[2] = __fadd_rn(acc[2], v.z);
    acc[3] = __fadd_rn(acc[3], v.w);
  }
  uint32_t b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) b[i] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[i]));
  *op = make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
}

}  // namespace
}  // namespace moe

extern "C" {

moe_status moe_quantize_act_per_row(const uint16_t* x, int64_t M, int K, uint8_t* q, float* scale,
                                    moe_stream_t stream) {
  using namespace moe;
  if (M < 0 || K < 32 || K % 32 != 0) return MOE_ERR_SHAPE;
  if (M == 0) return MOE_OK;
  if (!x || !q || !scale) return MOE_ERR_NULL;
  if (M > 0x7FFFFFFF) return MOE_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(q)) return MOE_ERR_ALIGN;
  DeviceInfo dev;
  if (current_device(&dev) != MOE_OK) return MOE_ERR_CUDA;
  if (!on_device(x, dev.device) || !on_device(q, dev.device) || !on_device(scale, dev.device)) return MOE_ERR_DEVICE;
  quant_act_row_kernel<<<static_cast<unsigned>(M), kW4Threads, 0, stream>>>(x, K, q, scale);
  MOE_CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}

moe_status moe_quantize_weight_k32(const uint16_t* w, int64_t rows, int K, uint8_t* q_packed, float* scale,
                                   moe_stream_t stream) {
  using namespace moe;
  if (rows < 1 || K < 32 || K % 32 != 0) return MOE_ERR_SHAPE;
  if (!w || !q_packed || !scale) return MOE_ERR_NULL;
  const int64_t nblk = rows * (K / 32);
  const int64_t grid = ceil_div(nblk, kW4Threads);
  if (grid > 0x7FFFFFFF) return MOE_ERR_SHAPE;
  if (!aligned16(w) || !aligned16(q_packed)) return MOE_ERR_ALIGN;
  DeviceInfo dev;
  if (current_device(&dev) != MOE_OK) return MOE_ERR_CUDA;
  if (!on_device(w, dev.device) || !on_device(q_packed, dev.device) || !on_device(scale, dev.device))
    return MOE_ERR_DEVICE;
  quant_weight_k32_kernel<<<static_cast<unsigned>(grid), kW4Threads, 0, stream>>>(w, nblk, q_packed, scale);
  MOE_CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}

size_t moe_w4a8_workspace_size(int64_t M, int H, int I, int top_k) {
  if (M < 0 || H < 0 || I < 0 || top_k < 1) return 0;
  return moe::w4_layout(M, H, I, top_k).total;
}

moe_status moe_w4a8_forward(const moe_w4a8_args* a, moe_stream_t stream) {
  using namespace moe;
  if (!a) return MOE_ERR_NULL;
  if (a->M < 0 || a->H < 32 || a->H % 32 || a->I < 32 || a->I % 32 || a->E < 1 || a->top_k < 1 || a->top_k > 64)
    return MOE_ERR_SHAPE;
  if (a->block_m < 8 || a->block_m > kW4MaxBlockM || a->block_m % 8) return MOE_ERR_SHAPE;
  if (a->path != MOE_W4A8_AUTO && a->path != MOE_W4A8_CUDA_CORES) return MOE_ERR_SHAPE;
  if (static_cast<int64_t>(a->block_m) * a->H > kW4MaxRowBytes ||
      static_cast<int64_t>(a->block_m) * a->I > kW4MaxRowBytes)
    return MOE_ERR_SHAPE;
  if (a->blocks_cap < 1 || a->sorted_cap < a->blocks_cap * a->block_m) return MOE_ERR_CAPACITY;
  const int64_t R = a->M * a->top_k;
  if (R >= (int64_t(1) << 31) - 1 || a->sorted_cap >= (int64_t(1) << 30)) return MOE_ERR_SHAPE;
  if (a->M == 0) return MOE_OK;
  if (!a->a || !a->a_scale || !a->w13 || !a->w13_scale || !a->w2 || !a->w2_scale || !a->topk_weights ||
      !a->sorted_token_ids || !a->expert_ids || !a->num_tokens_post_padded || !a->out || !a->workspace)
    return MOE_ERR_NULL;
  if ((a->debug_q_inter == nullptr) != (a->debug_s_inter == nullptr)) return MOE_ERR_NULL;
  if (!aligned16(a->a) || !aligned16(a->w13) || !aligned16(a->w2) || !aligned16(a->workspace) ||
      !aligned16(a->out) || (a->debug_q_inter && !aligned16(a->debug_q_inter)))
    return MOE_ERR_ALIGN;
  const W4Layout wl = w4_layout(a->M, a->H, a->I, a->top_k);
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
  MOE_CUDA_TRY(cudaFuncSetAttribute(w4a8_up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kW4MaxRowBytes));
  MOE_CUDA_TRY(cudaFuncSetAttribute(w4a8_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kW4MaxRowBytes));

  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  int32_t* rvalid = reinterpret_cast<int32_t*>(ws + wl.rv_off);
  float* h = reinterpret_cast<float*>(ws + wl.h_off);
  uint8_t* q = ws + wl.q_off;
  float* s = reinterpret_cast<float*>(ws + wl.s_off);
  float* y = reinterpret_cast<float*>(ws + wl.y_off);
  const W4Plan pl{a->sorted_token_ids, a->expert_ids, a->num_tokens_post_padded, static_cast<int>(R), a->top_k,
                  a->block_m, a->E, a->sorted_cap, a->blocks_cap};
  const unsigned nblocks = static_cast<unsigned>(a->blocks_cap);

  MOE_CUDA_TRY(cudaMemsetAsync(rvalid, 0, static_cast<size_t>(R) * 4, stream));
  const bool tc = a->path == MOE_W4A8_AUTO &&
                  w4a8_tc_supported(a->H, a->I, a->block_m, a->w13, a->w2, a->w13_scale, a->w2_scale);
  if (tc) {
    W4GemmParams gp{};
    gp.sorted_ids = a->sorted_token_ids;
    gp.expert_ids = a->expert_ids;
    gp.num_post_padded = a->num_tokens_post_padded;
    gp.status = a->device_status;
    gp.nblocks = a->blocks_cap;
    gp.sorted_cap = a->sorted_cap;
    gp.R = static_cast<int>(R);
    gp.top_k = a->top_k;
    gp.block_m = a->block_m;
    gp.E = a->E;
    gp.H = a->H;
    gp.I = a->I;
    gp.routed_scale = a->routed_scale;
    W4GemmParams gu = gp;
    gu.up = 1;
    gu.a_scale = a->a_scale;
    gu.h = h;
    gu.ntw = a->I / 64;
    gu.w_rows = 2 * a->I;
    const W4GemmTensors tu{a->w13, a->w13_scale, static_cast<uint64_t>(a->E) * 2 * a->I, a->a,
                           static_cast<uint64_t>(a->M), static_cast<uint64_t>(a->H)};
    moe_status st = launch_w4a8_tc_gemm(tu, gu, dev.sms, stream);
    if (st != MOE_OK) return st;
    const W4RequantParams rq{pl, h, q, s, rvalid, a->debug_q_inter, a->debug_s_inter, a->I};
    w4a8_requant_kernel<<<nblocks, kW4Threads, 0, stream>>>(rq);
    MOE_CUDA_TRY(cudaGetLastError());
    W4GemmParams gd = gp;
    gd.up = 0;
    gd.s_inter = s;
    gd.topk_w = a->topk_weights;
    gd.y = y;
    gd.ntw = a->H / 128;
    gd.w_rows = a->H;
    const W4GemmTensors td{a->w2, a->w2_scale, static_cast<uint64_t>(a->E) * a->H, q, static_cast<uint64_t>(R),
                           static_cast<uint64_t>(a->I)};
    st = launch_w4a8_tc_gemm(td, gd, dev.sms, stream);
    if (st != MOE_OK) return st;
    w4a8_combine_kernel<<<dim3(static_cast<unsigned>(a->M), static_cast<unsigned>(ceil_div(a->H, 4 * kW4Threads))),
                          kW4Threads, 0, stream>>>(a->out, y, rvalid, a->H, a->top_k);
    MOE_CUDA_TRY(cudaGetLastError());
    return MOE_OK;
  }
  const W4UpParams up{pl, a->a, a->a_scale, a->w13, a->w13_scale, h, a->device_status, a->H, a->I};
  w4a8_up_kernel<<<dim3(nblocks, static_cast<unsigned>(a->I / kUpCols)), kW4Threads,
                   static_cast<size_t>(a->block_m) * a->H, stream>>>(up);
  MOE_CUDA_TRY(cudaGetLastError());
  const W4RequantParams rq{pl, h, q, s, rvalid, a->debug_q_inter, a->debug_s_inter, a->I};
  w4a8_requant_kernel<<<nblocks, kW4Threads, 0, stream>>>(rq);
  MOE_CUDA_TRY(cudaGetLastError());
  const W4DownParams dn{pl, q, s, a->w2, a->w2_scale, a->topk_weights, y, a->H, a->I, a->routed_scale};
  w4a8_down_kernel<<<dim3(nblocks, static_cast<unsigned>(a->H / kDownCols)), kW4Threads,
                     static_cast<size_t>(a->block_m) * a->I, stream>>>(dn);
  MOE_CUDA_TRY(cudaGetLastError());
  w4a8_combine_kernel<<<dim3(static_cast<unsigned>(a->M), static_cast<unsigned>(ceil_div(a->H, 4 * kW4Threads))),
                        kW4Threads, 0, stream>>>(a->out, y, rvalid, a->H, a->top_k);
  MOE_CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}

}  // extern "C"

MOE_BOUNDS_TU()
