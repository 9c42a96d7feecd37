// moe_fp8_block_scale_forward_noalloc: the fused forward for callers that
// cannot allocate device memory.  Its scratch lives in a file-scope static
// device array of fixed size instead of a caller-provided workspace.
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB

__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch, looked up once per device with that
// device current (in host code the symbol is only a host-side stand-in).
moe_status static_scratch_address(int device, void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  if (device < 0 || device >= 64) return MOE_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[device] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    addr[device] = p;
  }
  *out = addr[device];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" {

size_t moe_noalloc_scratch_bytes(void) { return moe::kStaticScratchBytes; }

moe_status moe_fp8_block_scale_forward_noalloc(const moe_fwd_args* args, moe_stream_t stream) {
  using namespace moe;
  if (!args) return MOE_ERR_NULL;
  if (args->M < 0 || args->H < 0 || args->I < 0 || args->sorted_cap < 0) return MOE_ERR_SHAPE;
  const size_t need = moe_forward_workspace_size(args->M, args->H, args->I, args->E, args->top_k, args->block_m,
                                                 args->sorted_cap);
  if (need == 0) return MOE_ERR_SHAPE;
  if (need > kStaticScratchBytes) return MOE_ERR_CAPACITY;
  if (args->M == 0) return MOE_OK;
  DeviceInfo dev;
  if (current_device(&dev) != MOE_OK) return MOE_ERR_CUDA;
  void* scratch = nullptr;
  const moe_status st = static_scratch_address(dev.device, &scratch);
  if (st != MOE_OK) return st;
  // The array keeps whatever the previous call left; the forward needs its
  // scratch zeroed on entry.
  MOE_CUDA_TRY(cudaMemsetAsync(scratch, 0, need, stream));
  moe_fwd_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = kStaticScratchBytes;
  return moe_fp8_block_scale_forward(&a, stream);
}

}  // extern "C"

MOE_BOUNDS_TU()
