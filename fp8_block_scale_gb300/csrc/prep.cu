// Offline weight preparation and the quantisers that produce the path's FP8
// inputs.
//  - moe_prep_weights: the eight-row gate/up interleave the forward expects
//    (FlashInfer PR #4287, "Public contract and review fixes").
//  - moe_requant_scales_ue8m0: FP32 -> power-of-two block scales (SGLang PR
//    #43556, "Motivation" and "Modifications").
//  - moe_quantize_act_1x128 / moe_quantize_weight_128x128: one FP32 scale
//    per token and 128 columns of activations, one per 128x128 weight block
//    (PR #4287, "Public contract and review fixes").
// All of them stream HBM once: coalesced 16-byte loads and stores.
#include "common.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------- interleave

__global__ void interleave_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t E, int N, int chunks_per_row) {
  const int I = N / 2;
  const int64_t total = E * N * static_cast<int64_t>(chunks_per_row);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / chunks_per_row;
    const int c = static_cast<int>(i - row * chunks_per_row);
    const int64_t e = row / N;
    const int o = static_cast<int>(row - e * N);
    const int q = o >> 4, j = o & 15;
    const int src_row = j < 8 ? 8 * q + j : I + 8 * q + (j - 8);
    dst[i] = src[(e * N + src_row) * chunks_per_row + c];
  }
}

// ---------------------------------------------------------------- UE8M0

// Smallest power of two >= s (s > 0, finite), computed on the bit pattern.
__device__ __forceinline__ float pow2_round_up(float s) {
  const uint32_t b = __float_as_uint(s);
  const uint32_t ex = (b >> 23) & 0xFFu;
  const uint32_t man = b & 0x7FFFFFu;
  if (ex != 0) {
    if (man == 0) return s;
    if (ex >= 254) return s;  // 2^128 does not exist in FP32: leave such scales alone
    return __uint_as_float((ex + 1) << 23);
  }
  // subnormal: value = man * 2^-149
  const int p = 31 - __clz(man);  // highest set bit
  if ((man & (man - 1)) == 0) return s;
  if (p + 1 >= 23) return __uint_as_float(1u << 23);  // 2^-126, the smallest normal
  return __uint_as_float(1u << (p + 1));
}

__global__ void __launch_bounds__(256) requant_ue8m0_kernel(uint8_t* __restrict__ w, float* __restrict__ scale,
                                                            uint8_t* __restrict__ exp_out, int rows, int cols) {
  const int rb_n = rows / 128, cb_n = cols / 128;
  const int64_t blk = blockIdx.x;
  const int64_t e = blk / (static_cast<int64_t>(rb_n) * cb_n);
  const int rb = static_cast<int>((blk / cb_n) % rb_n);
  const int cb = static_cast<int>(blk % cb_n);
  const float s = scale[blk];
  const bool active = s > 0.f && isfinite(s);
  float sp = s;
  if (active) sp = pow2_round_up(s);
  if (active && sp != s) {
    const float ratio = __fdiv_rn(s, sp);
    uint8_t* base = w + (e * rows + static_cast<int64_t>(rb) * 128) * cols + static_cast<int64_t>(cb) * 128;
    // 128 rows x 128 bytes = 1024 chunks of 16 bytes; 4 per thread
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int chunk = threadIdx.x + 256 * k;
      const int r = chunk >> 3, c16 = chunk & 7;
      uint4* p = reinterpret_cast<uint4*>(base + static_cast<int64_t>(r) * cols + c16 * 16);
      uint4 v = *p;
      uint32_t* words = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t x = words[q];
        const float2 a = e4m3x2_to_f32(static_cast<uint16_t>(x & 0xFFFFu));
        const float2 b = e4m3x2_to_f32(static_cast<uint16_t>(x >> 16));
        const uint16_t lo = cvt_e4m3x2(__fmul_rn(a.x, ratio), __fmul_rn(a.y, ratio));
        const uint16_t hi = cvt_e4m3x2(__fmul_rn(b.x, ratio), __fmul_rn(b.y, ratio));
        words[q] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      }
      *p = v;
    }
  }
  if (threadIdx.x == 0) {
    if (active) scale[blk] = sp;
    if (exp_out) {
      int eb = 0;
      if (active) {
        const uint32_t b = __float_as_uint(sp);
        const int ex = static_cast<int>((b >> 23) & 0xFFu);
        if (ex != 0) {
          eb = ex;  // biased exponent of a normal power of two is log2 + 127
        } else {
          eb = 0;   // subnormal powers of two lie below 2^-127's neighbourhood: clamp
        }
        if (eb > 254) eb = 254;
      }
      exp_out[blk] = static_cast<uint8_t>(eb);
    }
  }
}

// ---------------------------------------------------------------- quantisers

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// One warp per (row, 128-column group): lane l holds columns 4l..4l+3.
// kPow2: the group's scale amax/448 is rounded up to a power of two (UE8M0),
// as the weight requant rounds block scales.
template <bool kPow2>
__global__ void __launch_bounds__(256) quant_act_kernel(const uint16_t* __restrict__ x, int64_t M, int H,
                                                        uint8_t* __restrict__ q, float* __restrict__ scale) {
  const int groups = H / 128;
  const int64_t gw = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (gw >= M * groups) return;
  const int64_t m = gw / groups;
  const int g = static_cast<int>(gw - m * groups);
  const int64_t off = m * H + static_cast<int64_t>(g) * 128 + 4 * lane;
  const uint2 raw = *reinterpret_cast<const uint2*>(x + off);
  float v[4] = {bf16_bits_to_f32(raw.x & 0xFFFFu), bf16_bits_to_f32(raw.x >> 16), bf16_bits_to_f32(raw.y & 0xFFFFu),
                bf16_bits_to_f32(raw.y >> 16)};
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  float s = __fdiv_rn(amax, 448.0f);
  if (kPow2 && s > 0.f) s = pow2_round_up(s);
  uint32_t packed = 0;
  if (s > 0.f) {
    const uint16_t lo = cvt_e4m3x2(__fdiv_rn(v[0], s), __fdiv_rn(v[1], s));
    const uint16_t hi = cvt_e4m3x2(__fdiv_rn(v[2], s), __fdiv_rn(v[3], s));
    packed = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  *reinterpret_cast<uint32_t*>(q + off) = packed;
  if (lane == 0) scale[m * groups + g] = s;
}

// One CTA (256 threads) per 128x128 block: thread t holds rows t/2 (two
// threads per row), 64 columns each.
__global__ void __launch_bounds__(256) quant_weight_kernel(const uint16_t* __restrict__ w, int rows, int cols,
                                                           uint8_t* __restrict__ q, float* __restrict__ scale) {
  __shared__ float red[8];
  const int rb_n = rows / 128, cb_n = cols / 128;
  const int64_t blk = blockIdx.x;
  const int64_t e = blk / (static_cast<int64_t>(rb_n) * cb_n);
  const int rb = static_cast<int>((blk / cb_n) % rb_n);
  const int cb = static_cast<int>(blk % cb_n);
  const int r = threadIdx.x >> 1, half = threadIdx.x & 1;
  const int64_t off = (e * rows + static_cast<int64_t>(rb) * 128 + r) * cols + static_cast<int64_t>(cb) * 128 + 64 * half;
  uint4 raw[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) raw[i] = reinterpret_cast<const uint4*>(w + off)[i];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t* u = reinterpret_cast<const uint32_t*>(&raw[i]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      amax = fmaxf(amax, fabsf(bf16_bits_to_f32(u[k] & 0xFFFFu)));
      amax = fmaxf(amax, fabsf(bf16_bits_to_f32(u[k] >> 16)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const float s = __fdiv_rn(amax, 448.0f);
  uint4 out[4];
  uint32_t* ow = reinterpret_cast<uint32_t*>(out);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t* u = reinterpret_cast<const uint32_t*>(&raw[i]);
#pragma unroll
    for (int k = 0; k < 4; k += 2) {
      uint32_t packed = 0;
      if (s > 0.f) {
        const uint16_t lo = cvt_e4m3x2(__fdiv_rn(bf16_bits_to_f32(u[k] & 0xFFFFu), s),
                                       __fdiv_rn(bf16_bits_to_f32(u[k] >> 16), s));
        const uint16_t hi = cvt_e4m3x2(__fdiv_rn(bf16_bits_to_f32(u[k + 1] & 0xFFFFu), s),
                                       __fdiv_rn(bf16_bits_to_f32(u[k + 1] >> 16), s));
        packed = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      }
      ow[i * 2 + k / 2] = packed;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) reinterpret_cast<uint4*>(q + off)[i] = out[i];
  if (threadIdx.x == 0) scale[blk] = s;
}

int grid_for(int64_t work, int threads, int sms) {
  int64_t g = ceil_div(work, threads);
  const int64_t cap = static_cast<int64_t>(sms) * 16;
  if (g > cap) g = cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace
}  // namespace moe

namespace moe {
namespace {
template <bool kPow2>
moe_status quantize_act(const uint16_t* x, int64_t M, int H, uint8_t* q, float* scale, cudaStream_t stream) {
  if (M == 0) return MOE_OK;
  if (!x || !q || !scale) return MOE_ERR_NULL;
  if (M < 0 || H < 128 || H % 128 != 0) return MOE_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(q)) return MOE_ERR_ALIGN;
  DeviceInfo dev;
  if (current_device(&dev) != MOE_OK) return MOE_ERR_CUDA;
  if (!on_device(x, dev.device) || !on_device(q, dev.device) || !on_device(scale, dev.device)) return MOE_ERR_DEVICE;
  const int64_t warps = M * (H / 128);
  const int64_t blocks = ceil_div(warps * 32, 256);
  if (blocks > 0x7FFFFFFF) return MOE_ERR_SHAPE;
  quant_act_kernel<kPow2><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x, M, H, q, scale);
  MOE_CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}
}  // namespace
}  // namespace moe

extern "C" {

moe_status moe_prep_weights(const uint8_t* w13, uint8_t* w13_interleaved, int E, int N, int H, moe_stream_t stream) {
  using namespace moe;
  if (!w13 || !w13_interleaved) return MOE_ERR_NULL;
  if (E < 1 || N < 256 || N % 256 != 0 || H < 16 || H % 16 != 0) return MOE_ERR_SHAPE;
  if (!aligned16(w13) || !aligned16(w13_interleaved)) return MOE_ERR_ALIGN;
  const int64_t bytes = static_cast<int64_t>(E) * N * H;
  const uint8_t* a = w13;
  const uint8_t* b = w13_interleaved;
  if (a < b + bytes && b < a + bytes) return MOE_ERR_SHAPE;  // overlapping buffers
  DeviceInfo dev;
  if (current_device(&dev) != MOE_OK) return MOE_ERR_CUDA;
  if (!on_device(w13, dev.device) || !on_device(w13_interleaved, dev.device)) return MOE_ERR_DEVICE;
  const int chunks = H / 16;
  interleave_kernel<<<grid_for(bytes / 16, 256, dev.sms), 256, 0, stream>>>(
      reinterpret_cast<const uint4*>(w13), reinterpret_cast<uint4*>(w13_interleaved), E, N, chunks);
  MOE_CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}

moe_status moe_requant_scales_ue8m0(uint8_t* w, float* scale, uint8_t* ue8m0_exp, int E, int rows, int cols,
                                    moe_stream_t stream) {
  using namespace moe;
  if (!w || !scale) return MOE_ERR_NULL;
  if (E < 1 || rows < 128 || cols < 128 || rows % 128 || cols % 128) return MOE_ERR_SHAPE;
  if (!aligned16(w)) return MOE_ERR_ALIGN;
  DeviceInfo dev;
  if (current_device(&dev) != MOE_OK) return MOE_ERR_CUDA;
  if (!on_device(w, dev.device) || !on_device(scale, dev.device) || (ue8m0_exp && !on_device(ue8m0_exp, dev.device)))
    return MOE_ERR_DEVICE;
  const int64_t nblk = static_cast<int64_t>(E) * (rows / 128) * (cols / 128);
  if (nblk > 0x7FFFFFFF) return MOE_ERR_SHAPE;
  requant_ue8m0_kernel<<<static_cast<unsigned>(nblk), 256, 0, stream>>>(w, scale, ue8m0_exp, rows, cols);
  MOE_CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}


moe_status moe_quantize_act_1x128(const uint16_t* x, int64_t M, int H, uint8_t* q, float* scale, moe_stream_t stream) {
  return moe::quantize_act<false>(x, M, H, q, scale, stream);
}

moe_status moe_quantize_act_1x128_ue8m0(const uint16_t* x, int64_t M, int H, uint8_t* q, float* scale,
                                        moe_stream_t stream) {
  return moe::quantize_act<true>(x, M, H, q, scale, stream);
}

moe_status moe_quantize_weight_128x128(const uint16_t* w, int64_t E, int rows, int cols, uint8_t* q, float* scale,
                                       moe_stream_t stream) {
  using namespace moe;
  if (!w || !q || !scale) return MOE_ERR_NULL;
  if (E < 1 || rows < 128 || cols < 128 || rows % 128 || cols % 128) return MOE_ERR_SHAPE;
  if (!aligned16(w) || !aligned16(q)) return MOE_ERR_ALIGN;
  DeviceInfo dev;
  if (current_device(&dev) != MOE_OK) return MOE_ERR_CUDA;
  if (!on_device(w, dev.device) || !on_device(q, dev.device) || !on_device(scale, dev.device)) return MOE_ERR_DEVICE;
  const int64_t nblk = E * (rows / 128) * (cols / 128);
  if (nblk > 0x7FFFFFFF) return MOE_ERR_SHAPE;
  quant_weight_kernel<<<static_cast<unsigned>(nblk), 256, 0, stream>>>(w, rows, cols, q, scale);
  MOE_CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}

}  // extern "C"

MOE_BOUNDS_TU()
