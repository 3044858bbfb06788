// bsq_api.cu -- the extern "C" entry points of libbsq.so: argument validation, per-device
// properties, the device status word, and dispatch to the kernel launchers.
#include <cuda_runtime.h>

#include <cmath>
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "bsq.h"
#include "bsq_device.cuh"
#include "bsq_internal.h"

namespace bsq {

// One status word per device (each device holds its own copy of this module's globals).
// Kernels record the first failure with atomicCAS; bsq_get_device_status reads and clears.
__device__ int g_status_word;

namespace {

DeviceInfo g_dev[kMaxDevices];
thread_local int t_stall_kernel = 0;  // BSQ_KERNEL_* of the armed stall, 0 = none
thread_local StallInjection t_stall;
std::once_flag g_dev_once[kMaxDevices];
thread_local int t_last_error = 0;

int fail(int code) {
  t_last_error = code;
  return code;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

__global__ void selftest_timeout_kernel(int64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing ever arrives on `bar`: the bounded wait must give up and record the timeout
    mbar_wait_bounded(&bar, 0, &abort_flag, status, static_cast<uint64_t>(limit_ns));
  }
}

}  // namespace

int record_error(int code) { return fail(code); }

StallInjection take_stall(int kernel) {
  if (t_stall_kernel != kernel) return StallInjection{};
  t_stall_kernel = 0;
  return t_stall;
}

const DeviceInfo* current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::call_once(g_dev_once[dev], [dev] {
    DeviceInfo d;
    d.device = dev;
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return;
    if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return;
    if (cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return;
    if (d.cc_major != 10 || d.cc_minor != 3) {
      g_dev[dev] = d;  // recorded, status stays nullptr -> BSQ_ERR_ARCH
      return;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return;
    d.status = static_cast<int*>(p);
    g_dev[dev] = d;
  });
  const DeviceInfo& d = g_dev[dev];
  return d.status != nullptr ? &d : nullptr;
}

namespace {
// One thread evaluating an index check that fails: records BSQ_ERR_DEVICE_CHECK in the checked
// build, nothing in the normal one.
__global__ void selftest_device_check_kernel(int* status) {
  const volatile int index = 1, size = 1;
  volatile int sink = 0;
  if (in_bounds(index < size, status)) sink = index;  // the guarded access touches nothing shared
  (void)sink;
}
}  // namespace

int launch_selftest_timeout(int64_t limit_ns, cudaStream_t stream, const DeviceInfo& dev) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, dev.status);
  return cudaGetLastError() == cudaSuccess ? BSQ_OK : BSQ_ERR_LAUNCH;
}

}  // namespace bsq

using bsq::aligned16;
using bsq::fail;

extern "C" {

size_t bsq_codes_bytes(int fmt, int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= 0) return 0;
  if (fmt == BSQ_MXFP8) return static_cast<size_t>(rows * cols);
  if (fmt == BSQ_NVFP4 || fmt == BSQ_MXFP4) return static_cast<size_t>(rows * cols / 2);
  return 0;
}

size_t bsq_scales_bytes(int fmt, int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= 0 || (fmt != BSQ_MXFP8 && fmt != BSQ_NVFP4 && fmt != BSQ_MXFP4)) return 0;
  const int64_t body = bsq::scales_body_bytes(fmt, rows, cols);
  return static_cast<size_t>(fmt == BSQ_NVFP4 ? body + 16 : body);
}

namespace {
// Validation shared by bsq_quantize and bsq_quantize_batch; BSQ_OK or the error code.
int check_quant_item(int fmt, bool given, const bsq_quant_item& it) {
  if (it.src == nullptr || it.codes == nullptr || it.scales == nullptr || it.rows <= 0 || it.cols <= 0)
    return BSQ_ERR_ARG;
  if (fmt == BSQ_NVFP4 && given && it.global_scale == nullptr) return BSQ_ERR_ARG;
  if (it.cols % bsq::block_size(fmt) != 0 || it.rows > INT32_MAX || it.cols > INT32_MAX) return BSQ_ERR_SHAPE;
  if (!aligned16(it.src) || !aligned16(it.codes) || !aligned16(it.scales)) return BSQ_ERR_ALIGN;
  if (it.global_scale != nullptr && (reinterpret_cast<uintptr_t>(it.global_scale) & 3u)) return BSQ_ERR_ALIGN;
  return BSQ_OK;
}
}  // namespace

int bsq_quantize_batch(int fmt_flags, int count, const bsq_quant_item* items, bsq_stream_t stream) {
  const int fmt = fmt_flags & BSQ_FMT_MASK;
  const int flags = fmt_flags & ~BSQ_FMT_MASK;
  if (fmt != BSQ_MXFP8 && fmt != BSQ_NVFP4 && fmt != BSQ_MXFP4) return fail(BSQ_ERR_ARG);
  if (flags & ~(BSQ_FLAG_SRC_F32 | BSQ_FLAG_GLOBAL_GIVEN)) return fail(BSQ_ERR_ARG);
  if (items == nullptr || count < 1 || count > BSQ_MAX_BATCH) return fail(BSQ_ERR_ARG);
  const bool given = (flags & BSQ_FLAG_GLOBAL_GIVEN) != 0;
  if (fmt != BSQ_NVFP4 && given) return fail(BSQ_ERR_ARG);
  bsq_quant_item local[BSQ_MAX_BATCH];
  for (int i = 0; i < count; ++i) {
    const int st = check_quant_item(fmt, given, items[i]);
    if (st != BSQ_OK) return fail(st);
    local[i] = items[i];
    if (fmt != BSQ_NVFP4) local[i].global_scale = nullptr;
  }
  const bsq::DeviceInfo* dev = bsq::current_device();
  if (dev == nullptr) return fail(BSQ_ERR_ARCH);
  const int st = bsq::launch_quantize_batch(fmt, (flags & BSQ_FLAG_SRC_F32) != 0, given, count, local,
                                            reinterpret_cast<cudaStream_t>(stream), *dev);
  return st == BSQ_OK ? BSQ_OK : fail(st);
}

int bsq_layernorm_quantize(int fmt_flags, const void* src, const void* gamma_bf16, const void* beta_bf16, float eps,
                           int64_t rows, int64_t cols, void* codes, void* scales, bsq_stream_t stream) {
  const int fmt = fmt_flags & BSQ_FMT_MASK;
  const int flags = fmt_flags & ~BSQ_FMT_MASK;
  if (fmt != BSQ_MXFP8 && fmt != BSQ_MXFP4) return fail(BSQ_ERR_ARG);
  if (flags & ~BSQ_FLAG_SRC_F32) return fail(BSQ_ERR_ARG);
  if (gamma_bf16 == nullptr || beta_bf16 == nullptr || !(eps >= 0.0f) || !(eps < INFINITY)) return fail(BSQ_ERR_ARG);
  const bsq_quant_item item = {src, rows, cols, codes, scales, nullptr};
  int st = check_quant_item(fmt, false, item);
  if (st != BSQ_OK) return fail(st);
  const bool f32 = (flags & BSQ_FLAG_SRC_F32) != 0;
  if (cols * (f32 ? 4 : 2) > 16384) return fail(BSQ_ERR_SHAPE);
  if (!aligned16(gamma_bf16) || !aligned16(beta_bf16)) return fail(BSQ_ERR_ALIGN);
  const bsq::DeviceInfo* dev = bsq::current_device();
  if (dev == nullptr) return fail(BSQ_ERR_ARCH);
  st = bsq::launch_layernorm_quantize(fmt, f32, item, static_cast<const uint16_t*>(gamma_bf16),
                                      static_cast<const uint16_t*>(beta_bf16), eps,
                                      reinterpret_cast<cudaStream_t>(stream), *dev);
  return st == BSQ_OK ? BSQ_OK : fail(st);
}

int bsq_quantize(int fmt_flags, const void* src, int64_t rows, int64_t cols, void* codes, void* scales,
                 float* global_scale, bsq_stream_t stream) {
  const bsq_quant_item item = {src, rows, cols, codes, scales, global_scale};
  return bsq_quantize_batch(fmt_flags, 1, &item, stream);
}

int bsq_quantize_dual(int fmt_flags, const void* src, int64_t rows, int64_t cols, uint64_t seed, void* row_codes,
                      void* row_scales, void* col_codes, void* col_scales, float* global_scale, bsq_stream_t stream) {
  const int fmt = fmt_flags & BSQ_FMT_MASK;
  const int flags = fmt_flags & ~BSQ_FMT_MASK;
  if (fmt != BSQ_MXFP8 && fmt != BSQ_NVFP4 && fmt != BSQ_MXFP4) return fail(BSQ_ERR_ARG);
  if (flags & ~(BSQ_FLAG_SRC_F32 | BSQ_FLAG_STOCHASTIC | BSQ_FLAG_GLOBAL_GIVEN)) return fail(BSQ_ERR_ARG);
  const bool given = (flags & BSQ_FLAG_GLOBAL_GIVEN) != 0;
  if (given && (fmt != BSQ_NVFP4 || global_scale == nullptr)) return fail(BSQ_ERR_ARG);
  if (src == nullptr || row_codes == nullptr || row_scales == nullptr || col_codes == nullptr ||
      col_scales == nullptr || rows <= 0 || cols <= 0)
    return fail(BSQ_ERR_ARG);
  if (rows % 32 != 0 || cols % 32 != 0 || rows > INT32_MAX || cols > INT32_MAX) return fail(BSQ_ERR_SHAPE);
  if (!aligned16(src) || !aligned16(row_codes) || !aligned16(row_scales) || !aligned16(col_codes) ||
      !aligned16(col_scales))
    return fail(BSQ_ERR_ALIGN);
  if (fmt == BSQ_NVFP4 && global_scale != nullptr && (reinterpret_cast<uintptr_t>(global_scale) & 3u))
    return fail(BSQ_ERR_ALIGN);
  const bsq::DeviceInfo* dev = bsq::current_device();
  if (dev == nullptr) return fail(BSQ_ERR_ARCH);
  const int st = bsq::launch_quantize_dual(fmt, (flags & BSQ_FLAG_SRC_F32) != 0, (flags & BSQ_FLAG_STOCHASTIC) != 0,
                                           given, seed, src, rows, cols, row_codes, row_scales, col_codes, col_scales,
                                           fmt == BSQ_NVFP4 ? global_scale : nullptr,
                                           reinterpret_cast<cudaStream_t>(stream), *dev);
  return st == BSQ_OK ? BSQ_OK : fail(st);
}

int bsq_delayed_global_scale(const void* prev_scales, int64_t rows, int64_t cols, float headroom, float* g_out,
                             bsq_stream_t stream) {
  if (prev_scales == nullptr || g_out == nullptr || rows <= 0 || cols <= 0) return fail(BSQ_ERR_ARG);
  if (!(headroom > 0.0f) || !(headroom < INFINITY)) return fail(BSQ_ERR_ARG);
  if (cols % 16 != 0 || rows > INT32_MAX || cols > INT32_MAX) return fail(BSQ_ERR_SHAPE);
  if (!aligned16(prev_scales) || (reinterpret_cast<uintptr_t>(g_out) & 3u)) return fail(BSQ_ERR_ALIGN);
  const bsq::DeviceInfo* dev = bsq::current_device();
  if (dev == nullptr) return fail(BSQ_ERR_ARCH);
  const int st = bsq::launch_delayed_scale(prev_scales, rows, cols, headroom, g_out,
                                           reinterpret_cast<cudaStream_t>(stream));
  return st == BSQ_OK ? BSQ_OK : fail(st);
}

namespace {
// Validation shared by the GEMM entry points; BSQ_OK or the error code.
int check_gemm(int fmt, const void* A, const void* A_scales, const void* B, const void* B_scales,
               const void* bias_bf16, const void* out, int64_t M, int64_t N, int64_t K) {
  if (fmt != BSQ_MXFP8 && fmt != BSQ_NVFP4 && fmt != BSQ_MXFP4) return BSQ_ERR_ARG;
  if (A == nullptr || A_scales == nullptr || B == nullptr || B_scales == nullptr || out == nullptr) return BSQ_ERR_ARG;
  if (M <= 0 || N <= 0 || K <= 0) return BSQ_ERR_ARG;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return BSQ_ERR_SHAPE;
  if (K % (fmt == BSQ_MXFP8 ? 128 : 256) != 0 || N % 8 != 0) return BSQ_ERR_SHAPE;
  if (!aligned16(A) || !aligned16(A_scales) || !aligned16(B) || !aligned16(B_scales) || !aligned16(out))
    return BSQ_ERR_ALIGN;
  if (bias_bf16 != nullptr && (reinterpret_cast<uintptr_t>(bias_bf16) & 1u)) return BSQ_ERR_ALIGN;
  return BSQ_OK;
}

int gemm_common(int fmt, int epi, const void* A, const void* A_scales, const void* B, const void* B_scales,
                const void* bias_bf16, void* out, void* out_scales, int64_t M, int64_t N, int64_t K,
                bsq_stream_t stream) {
  const bsq::DeviceInfo* dev = bsq::current_device();
  if (dev == nullptr) return fail(BSQ_ERR_ARCH);
  const int st = bsq::launch_gemm(fmt, epi, A, A_scales, B, B_scales, bias_bf16, out, out_scales, M, N, K,
                                  reinterpret_cast<cudaStream_t>(stream), *dev);
  return st == BSQ_OK ? BSQ_OK : fail(st);
}
}  // namespace

int bsq_gemm(int fmt, const void* A, const void* A_scales, const void* B, const void* B_scales,
             const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K, bsq_stream_t stream) {
  const int st = check_gemm(fmt, A, A_scales, B, B_scales, bias_bf16, out_bf16, M, N, K);
  if (st != BSQ_OK) return fail(st);
  return gemm_common(fmt, 0, A, A_scales, B, B_scales, bias_bf16, out_bf16, nullptr, M, N, K, stream);
}

int bsq_gemm_splitk(int fmt, const void* A, const void* A_scales, const void* B, const void* B_scales,
                    const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K, int splits,
                    void* workspace, size_t workspace_bytes, bsq_stream_t stream) {
  const int st = check_gemm(fmt, A, A_scales, B, B_scales, bias_bf16, out_bf16, M, N, K);
  if (st != BSQ_OK) return fail(st);
  const int64_t stages = K / (fmt == BSQ_MXFP8 ? 128 : 256);
  if (splits < 1 || splits > 8 || splits > stages) return fail(BSQ_ERR_ARG);
  if (splits == 1) return gemm_common(fmt, 0, A, A_scales, B, B_scales, bias_bf16, out_bf16, nullptr, M, N, K, stream);
  if (workspace == nullptr || workspace_bytes / 4 / static_cast<size_t>(splits) / static_cast<size_t>(M) <
                                  static_cast<size_t>(N))
    return fail(BSQ_ERR_ARG);
  if (!aligned16(workspace)) return fail(BSQ_ERR_ALIGN);
  const bsq::DeviceInfo* dev = bsq::current_device();
  if (dev == nullptr) return fail(BSQ_ERR_ARCH);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc = bsq::launch_gemm(fmt, 6, A, A_scales, B, B_scales, nullptr, workspace, nullptr, M, N, K, s, *dev, 1, splits);
  if (rc == BSQ_OK)
    rc = bsq::launch_splitk_finalize(fmt, static_cast<const float*>(workspace), splits, M, N, K, bias_bf16, A_scales,
                                     B_scales, out_bf16, s, *dev);
  return rc == BSQ_OK ? BSQ_OK : fail(rc);
}

int bsq_gemm_splitk_splits(int fmt, int64_t M, int64_t N, int64_t K) {
  if (fmt != BSQ_MXFP8 && fmt != BSQ_NVFP4 && fmt != BSQ_MXFP4) return fail(BSQ_ERR_ARG);
  if (M <= 0 || N <= 0 || K <= 0) return fail(BSQ_ERR_ARG);
  const bsq::DeviceInfo* dev = bsq::current_device();
  if (dev == nullptr) return fail(BSQ_ERR_ARCH);
  const int64_t tiles = bsq::ceil_div(bsq::ceil_div(M, 128), 2) * bsq::ceil_div(N, 256);
  const int64_t stages = K / (fmt == BSQ_MXFP8 ? 128 : 256);
  const int64_t s = std::min<int64_t>(std::min<int64_t>(dev->num_sms / 2 / tiles, 8), stages / 8);
  return static_cast<int>(std::max<int64_t>(s, 1));
}

int bsq_gemm_gelu(int fmt, const void* A, const void* A_scales, const void* B, const void* B_scales,
                  const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K, bsq_stream_t stream) {
  const int st = check_gemm(fmt, A, A_scales, B, B_scales, bias_bf16, out_bf16, M, N, K);
  if (st != BSQ_OK) return fail(st);
  return gemm_common(fmt, 1, A, A_scales, B, B_scales, bias_bf16, out_bf16, nullptr, M, N, K, stream);
}

int bsq_gemm_gelu_quantize(int fmt, const void* A, const void* A_scales, const void* B, const void* B_scales,
                           const void* bias_bf16, int out_fmt, void* out_codes, void* out_scales, int64_t M,
                           int64_t N, int64_t K, bsq_stream_t stream) {
  if (out_fmt != BSQ_MXFP8 && out_fmt != BSQ_MXFP4) return fail(BSQ_ERR_ARG);
  if (out_scales == nullptr) return fail(BSQ_ERR_ARG);
  int st = check_gemm(fmt, A, A_scales, B, B_scales, bias_bf16, out_codes, M, N, K);
  if (st != BSQ_OK) return fail(st);
  if (N % 32 != 0) return fail(BSQ_ERR_SHAPE);
  if (!aligned16(out_scales)) return fail(BSQ_ERR_ALIGN);
  return gemm_common(fmt, out_fmt == BSQ_MXFP8 ? 2 : 3, A, A_scales, B, B_scales, bias_bf16, out_codes, out_scales,
                     M, N, K, stream);
}

int bsq_convt2x2(int fmt, const void* A, const void* A_scales, const void* B, const void* B_scales,
                 const void* bias_bf16, void* out_bf16, int64_t batch, int64_t H, int64_t W, int64_t C_in,
                 int64_t C_out, int gelu, bsq_stream_t stream) {
  if (batch <= 0 || H <= 0 || W <= 0 || C_in <= 0 || C_out <= 0) return fail(BSQ_ERR_ARG);
  if (batch * H > INT32_MAX || batch * H * W > INT32_MAX || 4 * C_out > INT32_MAX) return fail(BSQ_ERR_SHAPE);
  if (C_out % 32 != 0 || (32 % W != 0 && W % 32 != 0)) return fail(BSQ_ERR_SHAPE);
  const int64_t M = batch * H * W, N = 4 * C_out;
  const int st = check_gemm(fmt, A, A_scales, B, B_scales, bias_bf16, out_bf16, M, N, C_in);
  if (st != BSQ_OK) return fail(st);
  const bsq::DeviceInfo* dev = bsq::current_device();
  if (dev == nullptr) return fail(BSQ_ERR_ARCH);
  const int rc = bsq::launch_gemm(fmt, gelu ? 5 : 4, A, A_scales, B, B_scales, bias_bf16, out_bf16, nullptr, M, N,
                                  C_in, reinterpret_cast<cudaStream_t>(stream), *dev, W);
  return rc == BSQ_OK ? BSQ_OK : fail(rc);
}

int bsq_get_device_status(bsq_stream_t stream) {
  const bsq::DeviceInfo* dev = bsq::current_device();
  if (dev == nullptr) return fail(BSQ_ERR_ARCH);
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return fail(BSQ_ERR_LAUNCH);
  int v = 0;
  const int zero = 0;
  if (cudaMemcpy(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return fail(BSQ_ERR_LAUNCH);
  if (cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return fail(BSQ_ERR_LAUNCH);
  return v;
}

int bsq_selftest_timeout(int64_t limit_ns, bsq_stream_t stream) {
  if (limit_ns < 1000 || limit_ns > 10000000000ll) return fail(BSQ_ERR_ARG);
  const bsq::DeviceInfo* dev = bsq::current_device();
  if (dev == nullptr) return fail(BSQ_ERR_ARCH);
  const int st = bsq::launch_selftest_timeout(limit_ns, reinterpret_cast<cudaStream_t>(stream), *dev);
  return st == BSQ_OK ? BSQ_OK : fail(st);
}

int bsq_test_inject_stall(int kernel, int64_t after_stages, int64_t wait_limit_ns) {
  if (kernel != BSQ_KERNEL_GEMM && kernel != BSQ_KERNEL_DUAL && kernel != BSQ_KERNEL_LAYERNORM) return fail(BSQ_ERR_ARG);
  if (after_stages < -1 || wait_limit_ns < 1000 || wait_limit_ns > 10000000000ll) return fail(BSQ_ERR_ARG);
  if (after_stages == -1) {  // disarm
    bsq::t_stall_kernel = 0;
    return BSQ_OK;
  }
  bsq::t_stall_kernel = kernel;
  bsq::t_stall.after = after_stages;
  bsq::t_stall.limit_ns = static_cast<uint64_t>(wait_limit_ns);
  return BSQ_OK;
}

int bsq_selftest_device_check(bsq_stream_t stream) {
  const bsq::DeviceInfo* dev = bsq::current_device();
  if (dev == nullptr) return fail(BSQ_ERR_ARCH);
  bsq::selftest_device_check_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(dev->status);
  return cudaGetLastError() == cudaSuccess ? BSQ_OK : fail(BSQ_ERR_LAUNCH);
}

int bsq_last_error(void) { return bsq::t_last_error; }

const char* bsq_strerror(int status) {
  switch (status) {
    case BSQ_OK: return "ok";
    case BSQ_ERR_ARG: return "invalid argument (null pointer, non-positive size, unknown format or flag)";
    case BSQ_ERR_SHAPE: return "unsupported shape (block size, K or N multiple)";
    case BSQ_ERR_ALIGN: return "pointer not 16-byte aligned";
    case BSQ_ERR_ARCH: return "no compute capability 10.3 (GB300) device";
    case BSQ_ERR_LAUNCH: return "CUDA launch or runtime error";
    case BSQ_ERR_TIMEOUT: return "a kernel's bounded wait timed out";
    case BSQ_ERR_DEVICE_CHECK: return "a kernel's index check failed (checked build)";
    default: return "unknown status";
  }
}

}  // extern "C"
