// bsq_internal.h -- host-side declarations shared by the translation units of libbsq.so.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>

#include "bsq.h"

namespace bsq {

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline int64_t block_size(int fmt) { return fmt == 2 /*BSQ_NVFP4*/ ? 16 : 32; }

// Bytes of the tiled scale body (128-row x 4-column tiles of 512 bytes), without the NVFP4 tail.
inline int64_t scales_body_bytes(int fmt, int64_t rows, int64_t cols) {
  const int64_t nsc = cols / block_size(fmt);
  return ceil_div(rows, 128) * ceil_div(nsc, 4) * 512;
}

struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  int cc_major = 0, cc_minor = 0;
  int* status = nullptr;  // device address of the status word
};

// Current device's cached properties (and the status word's address); nullptr when no
// usable device. Thread-safe.
const DeviceInfo* current_device();

// Kernel attributes (the dynamic shared-memory opt-in) and occupancy queries hold per device, so
// each kernel instance does its setup once per device: PerDevice<T> keeps one flag and one
// result per device index, and run(device, f) calls f() the first time that device asks.
constexpr int kMaxDevices = 64;
template <typename T>
struct PerDevice {
  std::once_flag once[kMaxDevices];
  T value[kMaxDevices] = {};
  template <typename F>
  const T& run(int device, F&& f) {
    std::call_once(once[device], [&] { value[device] = f(); });
    return value[device];
  }
};

// A stall injected into the next launch of one kernel class on the calling thread
// (bsq_test_inject_stall): the producers stop issuing loads after `after` pipeline stages (-1:
// none) and the launch's bounded waits give up after `limit_ns`.
struct StallInjection {
  int64_t after = -1;
  uint64_t limit_ns = 2000000000ull;
};
// Takes (and clears) the calling thread's injection if it names `kernel` (BSQ_KERNEL_*); else none.
StallInjection take_stall(int kernel);

// Record `code` as the calling thread's last error (bsq_last_error) and return it.
int record_error(int code);

// cuTensorMapEncodeTiled, obtained once through the runtime's driver entry-point query
// (nullptr if unavailable).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();

// 2-D tensor map over `outer` rows of `inner` elements (row pitch `row_bytes`), box
// box_inner x box_outer, zero fill out of bounds. False if the encoder refused.
bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

// Items already validated (shapes, alignment); count in [1, BSQ_MAX_BATCH].
using QuantItem = bsq_quant_item;
int launch_quantize_batch(int fmt, bool src_f32, bool global_given, int count, const QuantItem* items,
                          cudaStream_t stream, const DeviceInfo& dev);

// For each of n (1..BSQ_MAX_BATCH) sources: the largest |x| of its elems[i] bf16 / fp32 values
// (elems * size a multiple of 16 bytes), atomically max-ed into *outs[i] as fp32 bits (which
// must hold 0 or an earlier maximum). One launch.
int launch_amax(const void* const* srcs, const int64_t* elems, uint32_t* const* outs, int n, bool src_f32,
                cudaStream_t stream, const DeviceInfo& dev);

// g_out = fp32(fp32(amax * headroom) / 2688), amax from the tail of an NVFP4 scale buffer of a
// rows x cols matrix.
int launch_delayed_scale(const void* prev_scales, int64_t rows, int64_t cols, float headroom, float* g_out,
                         cudaStream_t stream);

// Row LayerNorm then MX quantization of one matrix (fmt MXFP8 / MXFP4); rows must fit a chunk
// (BSQ_ERR_SHAPE otherwise).
int launch_layernorm_quantize(int fmt, bool src_f32, const QuantItem& item, const uint16_t* gamma,
                              const uint16_t* beta, float eps, cudaStream_t stream, const DeviceInfo& dev);

// Dual-layout quantization (MXFP8 / MXFP4 / NVFP4) of one rows x cols matrix, arguments
// validated (rows, cols multiples of 32). NVFP4: global_scale as bsq_quantize's (given mode
// when global_given).
int launch_quantize_dual(int fmt, bool src_f32, bool stochastic, bool global_given, uint64_t seed, const void* src,
                         int64_t rows, int64_t cols, void* row_codes, void* row_scales, void* col_codes,
                         void* col_scales, float* global_scale, cudaStream_t stream, const DeviceInfo& dev);

// epi: 0 bf16 out, 1 GELU -> bf16, 2 GELU -> MXFP8 codes + scales, 3 GELU -> MXFP4 (out_scales
// used by 2 and 3 only), 4 / 5 kernel-2 stride-2 transposed convolution to NHWC bf16 (without /
// with GELU; N = 4 C_out, M = batch H W, convt_w = W), 6 split-K partial sums: `out` is an fp32
// workspace of splits x M x N (slice s = K stages [s nk / splits, (s + 1) nk / splits), raw
// accumulator; 1 <= splits <= K stages).
int launch_gemm(int fmt, int epi, const void* A, const void* A_scales, const void* B, const void* B_scales,
                const void* bias, void* out, void* out_scales, int64_t M, int64_t N, int64_t K, cudaStream_t stream,
                const DeviceInfo& dev, int64_t convt_w = 1, int splits = 1);

// out_bf16 = bf16(alpha * sum of the workspace's slices + bias), after launch_gemm epi 6.
int launch_splitk_finalize(int fmt, const float* ws, int splits, int64_t M, int64_t N, int64_t K, const void* bias,
                           const void* A_scales, const void* B_scales, void* out, cudaStream_t stream,
                           const DeviceInfo& dev);

int launch_selftest_timeout(int64_t limit_ns, cudaStream_t stream, const DeviceInfo& dev);

}  // namespace bsq
