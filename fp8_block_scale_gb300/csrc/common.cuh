// Shared helpers of the GB300 (sm_103a) MoE FP8 library: status handling,
// host-side argument checks, and thin inline-PTX wrappers for mbarrier, TMA
// (cp.async.bulk.tensor), tcgen05 (MMA into tensor memory) and FP8 conversion.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <cstddef>

#include "../../include/moe_fp8.h"

namespace moe {

// ---------------------------------------------------------------- host side

#define MOE_CUDA_TRY(expr)                                   \
  do {                                                       \
    cudaError_t err__ = (expr);                              \
    if (err__ != cudaSuccess) return MOE_ERR_CUDA;           \
  } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Current device's ordinal, SM count and compute capability (cached per device).
struct DeviceInfo {
  int device = -1;
  int sms = 0;
  int major = 0, minor = 0;
};
moe_status current_device(DeviceInfo* info);

// True if `p` is device (or managed) memory that the current device can use.
bool on_device(const void* p, int device);

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Launch with programmatic stream serialization (the kernel calls
// pdl_wait), optionally as clusters of `cluster` CTAs.
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, int cluster,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// cuTensorMapEncodeTiled fetched through the runtime (no -lcuda needed).
CUresult encode_tensor_map_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                              uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                              CUtensorMapSwizzle swizzle);
// The same for another element type (sizes in elements, the stride in bytes).
CUresult encode_tensor_map_2d_typed(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                                    uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                                    uint32_t box_outer, CUtensorMapSwizzle swizzle);

// ---------------------------------------------------------------- bounds checks
//
// MOE_IN_BOUNDS(c) guards a global access or a tensor copy whose index is
// derived from data (plan entries, route and token ids, expert ids) or from
// tiling arithmetic.  In a library built with -DMOE_DEBUG_BOUNDS it counts a
// failed check in this translation unit's bounds record (and keeps the first
// failing source line), then returns false: the caller skips the access, or
// moves a tensor copy to coordinate 0 so that its barrier still receives the
// bytes it expects.  Nothing traps.  In the normal build it is the constant
// true and the checks compile away.  Each translation unit ends with
// MOE_BOUNDS_TU(), which registers a host reader of its record for
// moe_debug_bounds_read.
struct BoundsRecord {
  unsigned long long failures;
  int first_line;
  int pad;
};
using BoundsReader = cudaError_t (*)(BoundsRecord* out, int reset);
void bounds_register(BoundsReader reader, const char* file);

#ifdef MOE_DEBUG_BOUNDS
static __device__ BoundsRecord g_bounds;
__device__ __forceinline__ bool bounds_note(bool ok, int line) {
  if (!ok) {
    atomicAdd(&g_bounds.failures, 1ull);
    atomicCAS(&g_bounds.first_line, 0, line);
  }
  return ok;
}
#define MOE_IN_BOUNDS(c) ::moe::bounds_note(static_cast<bool>(c), __LINE__)
#define MOE_BOUNDS_TU()                                                                      \
  namespace {                                                                                \
  cudaError_t bounds_read_tu(::moe::BoundsRecord* out, int reset) {                          \
    cudaError_t err = cudaMemcpyFromSymbol(out, ::moe::g_bounds, sizeof(::moe::BoundsRecord)); \
    if (err == cudaSuccess && reset) {                                                       \
      const ::moe::BoundsRecord zero = {};                                                   \
      err = cudaMemcpyToSymbol(::moe::g_bounds, &zero, sizeof(zero));                        \
    }                                                                                        \
    return err;                                                                              \
  }                                                                                          \
  const bool bounds_registered_tu = (::moe::bounds_register(bounds_read_tu, __FILE__), true); \
  }
#else
#define MOE_IN_BOUNDS(c) true
#define MOE_BOUNDS_TU()
#endif

// A 2D tensor copy's coordinates: the innermost one (x, in elements) a
// multiple of `x_align` (16 bytes' worth) and inside the row, the outer one
// inside the tensor.  A failing copy is moved to the origin, which every
// tensor the library copies from has.
#define MOE_CHECK_BOX(x, y, x_extent, y_extent, x_align)                                               \
  do {                                                                                                 \
    if (!MOE_IN_BOUNDS((x) >= 0 && (x) % (x_align) == 0 && static_cast<int64_t>(x) < (x_extent) &&     \
                       (y) >= 0 && static_cast<int64_t>(y) < (y_extent))) {                            \
      (x) = 0;                                                                                         \
      (y) = 0;                                                                                         \
    }                                                                                                  \
  } while (0)

// ---------------------------------------------------------------- device side

// A bounded wait gives up after this long (the whole forward takes well under
// a millisecond; one second means something is stuck).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;
// ... or after this many polls, whichever comes first: a second bound that
// does not rely on %globaltimer advancing.  A failed poll takes at least some
// ten nanoseconds (at most a short, hardware-defined suspension), so the cap
// is a few tenths of a second or more; either bound lies far above any wait
// of a healthy forward (milliseconds at most).
constexpr uint32_t kWaitMaxPolls = 1u << 25;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Adds `bytes` to the transaction count of the current phase without
// arriving: the phase cannot complete before the expected arrival.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false, and
// raises *abort_flag, if the wait runs past `limit_ns` (or kWaitMaxPolls
// polls); returns false at once if another thread of the CTA has already
// raised *abort_flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  unsigned long long t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 31u) {
      if (*abort_flag) return false;
      unsigned long long now = global_timer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > limit_ns || i >= kWaitMaxPolls) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while its predecessor finishes; it must wait here
// before touching memory the predecessor writes (the wait returns once the
// predecessor grid has completed and its writes are visible).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel on the stream begin launching.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Named barrier over `count` threads (a multiple of 32) with id `id` (1..15).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// Four rows (y0..y3) of a 2D tensor, each `box inner` elements wide starting at
// column x, land one after another at dst (the map's box is one row high).
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y0, int y1,
                                            int y2, int y3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3)
      : "memory");
}

// Contiguous global -> shared copy of `bytes` (a multiple of 16; both
// addresses 16-byte aligned), completing on the mbarrier like a tensor load.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// ---- tcgen05 (tensor memory + 5th generation tensor core MMA)

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f8f6f4, issued by one thread.
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier completes one arrival once every tcgen05 operation this thread
// issued before has finished.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// D[tmem] (+)= (A * 2^sfa) * (B * 2^sfb)^T, kind::mxf8f6f4 with one UE8M0
// scale per row of A and per column of B for the instruction's 32-wide K
// block (scale_vec::1X), read from tensor memory: row m of A at lane m,
// column sfa + m / 32; column n of B at lane 32 (m / 32) + n % 32 (each lane
// quarter holds a copy), column sfb + n / 32; the byte of each 32-bit cell
// is chosen by the instruction descriptor's scale-factor ids.
__device__ __forceinline__ void umma_mx8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Shared memory -> tensor memory copy of 32 rows x 16 bytes, written to the
// same 32 lanes of all four lane quarters (columns taddr .. taddr + 3: row r
// lands in lane 32 q + r, bytes 4 i .. 4 i + 3 of the row in column
// taddr + i).  Ordered with the MMAs the same thread issues.
__device__ __forceinline__ void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Shared-memory descriptor of 32 rows x 16 bytes stored row after row
// (no swizzle: 8-row core matrices 128 bytes apart).
__device__ __forceinline__ uint64_t rows16_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);  // start address
  d |= static_cast<uint64_t>(128 >> 4) << 16;          // leading byte offset (one 16-byte column: unused)
  d |= static_cast<uint64_t>(128 >> 4) << 32;          // stride byte offset: next 8-row core matrix
  d |= static_cast<uint64_t>(1) << 46;                 // descriptor version (sm_100 family)
  return d;                                            // swizzle: none
}

// Make this thread's generic-proxy shared-memory writes visible to the
// tensor core's (async proxy) reads.
// Tensor store of a 2D box from shared memory, tracked as a bulk group of
// the issuing thread (commit, then wait for its reads or its completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map), "r"(src),
               "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The shared memory of every committed group has been read (it may be reused).
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Every committed group has completed (its writes are done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, rows of 128 bytes stored
// with the 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);  // start address
  d |= static_cast<uint64_t>(1) << 16;                 // leading byte offset (unused with swizzle)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;         // stride byte offset: next 8-row group
  d |= static_cast<uint64_t>(1) << 46;                 // descriptor version (sm_100 family)
  d |= static_cast<uint64_t>(2) << 61;                 // swizzle: 128 bytes
  return d;
}

// Instruction descriptor, kind::f8f6f4: E4M3 x E4M3 -> F32, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n) {
  return (1u << 4)                                 // D format F32
         | (0u << 7) | (0u << 10)                  // A, B format E4M3
         | (static_cast<uint32_t>(n >> 3) << 17)   // N / 8
         | (static_cast<uint32_t>(m >> 4) << 24);  // M / 16
}

// Instruction descriptor, kind::mxf8f6f4 with UE8M0 block scales: E4M3 x
// E4M3 -> F32, both K-major, scale-factor byte 0 of A's and B's cells.
__host__ __device__ constexpr uint32_t idesc_mx_e4m3(int m, int n) {
  return (0u << 4)                                 // B scale-factor id
         | (0u << 7) | (0u << 10)                  // A, B format E4M3
         | (static_cast<uint32_t>(n >> 3) << 17)   // N / 8
         | (1u << 23)                              // scale format UE8M0
         | (static_cast<uint32_t>(m >> 4) << 24)   // M / 16
         | (0u << 29);                             // A scale-factor id
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (taddr.lane + i), columns taddr.col .. taddr.col + 31.
// 32 lanes x 16 consecutive 32-bit columns (the epilogue's chunk: with ten
// warps per CTA a thread may use 168 registers, 128 of which hold the FP32
// accumulators, so wider chunks would spill).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 8 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}

// Instruction descriptor, kind::f8f6f4: A E2M1 (FP4, in the padded shared-
// memory form the copy engine writes for 16U4_ALIGN16B tensors) x B E4M3
// -> F32, both K-major.
__host__ __device__ constexpr uint32_t idesc_e2m1_e4m3_f32(int m, int n) {
  return (1u << 4)                                 // D format F32
         | (5u << 7) | (0u << 10)                  // A E2M1, B E4M3
         | (static_cast<uint32_t>(n >> 3) << 17)   // N / 8
         | (static_cast<uint32_t>(m >> 4) << 24);  // M / 16
}

// ---- FP8 conversion

// Two floats -> two E4M3 codes (round to nearest even, finite overflow
// saturates to +-448).  Byte 0 of the result holds lo, byte 1 holds hi.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 codes (byte 0, byte 1) -> two exact floats.
__device__ __forceinline__ float2 e4m3x2_to_f32(uint16_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// Start moving `bytes` (a multiple of 16, 16-byte aligned) from global
// memory into L2 without waiting for them.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// silu(g) = g / (1 + exp(-g)) with the hardware exp2 and divide
// approximations (a few ulp; for g below about -88 the quotient is 0).
__device__ __forceinline__ float silu_f32(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

}  // namespace moe
