// bsq_scratch.cu -- bsq_gemm_splitk with its fp32 workspace in a fixed device array of the
// library instead of a caller buffer: a call allocates nothing.
//
// The array is a file-scope __device__ variable: the loader places it with the module, once per
// device, and no call allocates or frees it. Its address on the current device is looked up
// once per device (cudaGetSymbolAddress) and then passed to bsq_gemm_splitk as the workspace, so
// validation, the two kernels and every error code are bsq_gemm_splitk's own; a request larger
// than the array fails there like one with too small a workspace. Nothing in it needs to start
// at zero: the split-K GEMM overwrites every element of the slices it uses before the finalize
// kernel reads them. The array is shared by all callers in the process on a device, so calls that
// may overlap in time race on it.
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "bsq.h"
#include "bsq_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t{64} << 20;  // 64 MiB: splits * M * N * 4 bytes at most
static __device__ __align__(256) unsigned char g_splitk_scratch[kScratchBytes];

using bsq::kMaxDevices;
std::once_flag g_scratch_once[kMaxDevices];
void* g_scratch_addr[kMaxDevices];

// The array's address on the current device (nullptr if unavailable), looked up once per device.
void* scratch_address() {
  const bsq::DeviceInfo* dev = bsq::current_device();
  if (dev == nullptr || dev->device < 0 || dev->device >= kMaxDevices) return nullptr;
  const int d = dev->device;
  std::call_once(g_scratch_once[d], [d] {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_splitk_scratch) == cudaSuccess) {
      g_scratch_addr[d] = p;
    } else {
      g_scratch_addr[d] = nullptr;
      cudaGetLastError();  // the failed lookup leaves no error pending for a later launch check
    }
  });
  return g_scratch_addr[d];
}

}  // namespace

int bsq_gemm_splitk_scratch(int fmt, const void* A, const void* A_scales, const void* B, const void* B_scales,
                            const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K, int splits,
                            bsq_stream_t stream) {
  void* ws = scratch_address();
  // a usable device whose array could not be found: say so rather than report a workspace too
  // small (without a usable device bsq_gemm_splitk itself returns the argument or device error)
  if (ws == nullptr && splits > 1 && bsq::current_device() != nullptr) return bsq::record_error(BSQ_ERR_LAUNCH);
  return bsq_gemm_splitk(fmt, A, A_scales, B, B_scales, bias_bf16, out_bf16, M, N, K, splits, ws,
                         ws != nullptr ? kScratchBytes : 0, stream);
}
