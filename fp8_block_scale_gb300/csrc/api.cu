// Host-side entry points shared by the library: status strings, device
// queries, tensor-map encoding, plan capacity and workspace helpers.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace moe {

moe_status current_device(DeviceInfo* info) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  int dev = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MOE_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev].device != dev) {
    DeviceInfo d;
    d.device = dev;
    MOE_CUDA_TRY(cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev));
    MOE_CUDA_TRY(cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev));
    MOE_CUDA_TRY(cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev));
    cache[dev] = d;
  }
  *info = cache[dev];
  return MOE_OK;
}

bool on_device(const void* p, int device) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (attr.type == cudaMemoryTypeDevice) return attr.device == device;
  if (attr.type == cudaMemoryTypeManaged) return true;
  return false;
}

CUresult encode_tensor_map_2d_typed(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                                    uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                                    uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_tensor_map_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                              uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                              CUtensorMapSwizzle swizzle) {
  return encode_tensor_map_2d_typed(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, inner, outer, row_stride_bytes,
                                    box_inner, box_outer, swizzle);
}

// Readers of the translation units' bounds records (registered while the
// library loads; empty in the normal build).
namespace {
struct BoundsEntry {
  BoundsReader reader;
  const char* file;
};
std::vector<BoundsEntry>& bounds_registry() {
  static std::vector<BoundsEntry> v;
  return v;
}
}  // namespace

void bounds_register(BoundsReader reader, const char* file) { bounds_registry().push_back({reader, file}); }

// Self-test of the bounds checks: reads data[probe] into *out only when the
// check passes (-1 otherwise).
__global__ void bounds_selftest_kernel(const int32_t* data, int n, int probe, int32_t* out) {
  int32_t v = -1;
  if (MOE_IN_BOUNDS(probe >= 0 && probe < n)) v = data[probe];
  *out = v;
}

}  // namespace moe

extern "C" {

int moe_debug_bounds_enabled(void) {
#ifdef MOE_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

moe_status moe_debug_bounds_selftest(const int32_t* data, int n, int probe, int32_t* out, moe_stream_t stream) {
  using namespace moe;
  if (!data || !out) return MOE_ERR_NULL;
  if (n < 1) return MOE_ERR_SHAPE;
  // without the device-side checks an out-of-range probe is refused here
  if (!moe_debug_bounds_enabled() && (probe < 0 || probe >= n)) return MOE_ERR_SHAPE;
  DeviceInfo dev;
  if (current_device(&dev) != MOE_OK) return MOE_ERR_CUDA;
  if (!on_device(data, dev.device) || !on_device(out, dev.device)) return MOE_ERR_DEVICE;
  bounds_selftest_kernel<<<1, 1, 0, stream>>>(data, n, probe, out);
  MOE_CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}

moe_status moe_debug_bounds_read(uint64_t* failures, const char** first_file, int32_t* first_line, int reset) {
  if (!failures) return MOE_ERR_NULL;
  *failures = 0;
  if (first_file) *first_file = nullptr;
  if (first_line) *first_line = 0;
  if (moe::bounds_registry().empty()) return MOE_OK;
  MOE_CUDA_TRY(cudaDeviceSynchronize());
  for (const auto& entry : moe::bounds_registry()) {
    moe::BoundsRecord r = {};
    MOE_CUDA_TRY(entry.reader(&r, reset));
    if (r.failures != 0 && *failures == 0) {
      const char* base = std::strrchr(entry.file, '/');
      if (first_file) *first_file = base ? base + 1 : entry.file;
      if (first_line) *first_line = r.first_line;
    }
    *failures += r.failures;
  }
  return MOE_OK;
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_NULL: return "MOE_ERR_NULL: a required pointer is NULL";
    case MOE_ERR_SHAPE: return "MOE_ERR_SHAPE: a size violates the documented constraints";
    case MOE_ERR_ALIGN: return "MOE_ERR_ALIGN: a pointer is not 16-byte aligned";
    case MOE_ERR_CAPACITY: return "MOE_ERR_CAPACITY: plan or workspace buffer too small";
    case MOE_ERR_DTYPE: return "MOE_ERR_DTYPE: unsupported id width";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE: pointer not on the current device, or device is not sm_103";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call failed";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    default: return "unknown moe_status";
  }
}

moe_status moe_plan_capacity(int64_t M, int top_k, int E, int block_m, int64_t* sorted_cap,
                             int64_t* blocks_cap) {
  if (!sorted_cap || !blocks_cap) return MOE_ERR_NULL;
  if (M < 0 || top_k < 1 || E < 1 || block_m < 1) return MOE_ERR_SHAPE;
  const int64_t R = M * top_k;
  const int64_t nonempty = R < E ? R : E;
  int64_t cap = moe::round_up(R + nonempty * (block_m - 1), block_m);
  if (cap == 0) cap = block_m;  // keep one block so buffers are never empty
  *sorted_cap = cap;
  *blocks_cap = cap / block_m;
  return MOE_OK;
}

moe_status moe_workspace_init(void* workspace, size_t bytes, moe_stream_t stream) {
  if (!workspace) return bytes == 0 ? MOE_OK : MOE_ERR_NULL;
  MOE_CUDA_TRY(cudaMemsetAsync(workspace, 0, bytes, stream));
  return MOE_OK;
}

}  // extern "C"

MOE_BOUNDS_TU()
