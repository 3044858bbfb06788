// bsq_quantize.cu -- memory-bound block quantizers: bf16/fp32 -> MXFP8, NVFP4, MXFP4.
//
// Formats ("lightly-train - DINOv3 + EoMT on RTX 5090" README, section 2 number formats):
//   MXFP8  E4M3 codes, UE8M0 scale per 1x32 block;
//   NVFP4  e2m1 codes, E4M3 scale per 1x16 block, fp32 per-tensor scale g = amax / (6 * 448);
//   MXFP4  e2m1 codes, UE8M0 scale per 1x32 block.
// Elements round to nearest even and saturate at the largest finite value (448 for E4M3,
// the BF16 ledger blog section 5.4; 6 for e2m1). The UE8M0 exponent of a block is
// floor(log2(amax)) - emax with emax the exponent of the element format's top binade.
//
// Work mapping: one warp quantizes a 256-element segment of one row per step, each lane
// 8 consecutive elements (one 16-byte bf16 load). A 1x32 block is 4 lanes, a 1x16 block 2
// lanes; block maxima come from two (one) xor-shuffles. Each warp keeps kUnroll segments
// of loads in flight. Codes leave as one 8-byte (E4M3) or 4-byte (e2m1) store per lane,
// i.e. 256 or 128 contiguous bytes per warp. The scales of 4 consecutive blocks of a row
// are 4 contiguous bytes in the tiled layout (128 rows x 4 columns per 512-byte tile, row
// r at byte (r % 32) * 16 + ((r / 32) % 4) * 4), so each group of 4 scales is gathered with
// shuffles and written as one 32-bit word.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "bsq_device.cuh"
#include "bsq_internal.h"

namespace bsq {
namespace {

constexpr int kThreads = 256;
// Resident CTAs per SM (and so the register budget: 65536 / (256 * n)). fp32 sources and
// NVFP4 hold more live values per lane.
template <int FMT, bool F32>
__host__ __device__ constexpr int ctas_per_sm() {
  return F32 ? 2 : (FMT == BSQ_NVFP4 ? 3 : 4);
}
constexpr int kUnroll = 4;
constexpr int kSeg = 256;  // elements per warp step

enum NvMode { kMx = 0, kNvComputed = 1, kNvGiven = 2 };

struct QuantArgs {
  const void* src;
  int64_t rows, cols;
  uint8_t* codes;
  uint8_t* scales;
  uint32_t* tail;       // NVFP4: {g, amax bits, 0, 0}
  const float* g_in;    // NVFP4 given-scale mode
  float* g_out;         // NVFP4 computed mode (nullable)
  int64_t segs_per_row;
  int64_t total_segs;
  int64_t nsc;          // scale columns per row
  int64_t nct;          // 4-column scale tiles per row
};

template <bool F32>
struct Loaded {
  uint4 v[F32 ? 2 : 1];
};

__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  const uint32_t E = (c >> 3) & 15u, m = c & 7u;
  if (E == 0u) return static_cast<float>(m) * 0.001953125f;  // m * 2^-9, exact
  return __uint_as_float(((E + 120u) << 23) | (m << 20));
}

// 8 source elements of one lane -> fp32 values and the max of their magnitude bits
// (bf16: 15-bit magnitudes, fp32: 31-bit magnitudes; both order like the values).
template <bool F32>
__device__ __forceinline__ void unpack8(const Loaded<F32>& L, float (&x)[8], uint32_t& mag_max) {
  uint32_t mm = 0;
  if constexpr (F32) {
    const uint32_t w[8] = {L.v[0].x, L.v[0].y, L.v[0].z, L.v[0].w, L.v[1].x, L.v[1].y, L.v[1].z, L.v[1].w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[i] = __uint_as_float(w[i]);
      mm = max(mm, w[i] & 0x7FFFFFFFu);
    }
  } else {
    const uint32_t w[4] = {L.v[0].x, L.v[0].y, L.v[0].z, L.v[0].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      mm = max(mm, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
    }
  }
  mag_max = mm;
}

template <bool F32>
__device__ __forceinline__ uint32_t exp_field(uint32_t mag) {
  return F32 ? (mag >> 23) : (mag >> 7);
}

template <bool F32>
__device__ __forceinline__ float mag_to_f32(uint32_t mag) {
  return F32 ? __uint_as_float(mag) : __uint_as_float(mag << 16);
}

// Byte offset of the 32-bit scale word holding scale columns [c4, c4 + 4) of row r.
__device__ __forceinline__ int64_t scale_word_offset(int64_t r, int64_t c4, int64_t nct) {
  return ((r >> 7) * nct + (c4 >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
}

template <int FMT, bool F32, int NV>
__global__ void __launch_bounds__(kThreads, (ctas_per_sm<FMT, F32>())) quantize_kernel(QuantArgs a) {
  constexpr bool kFp4 = (FMT != BSQ_MXFP8);
  constexpr int kLanesPerBlock = (FMT == BSQ_NVFP4) ? 2 : 4;
  constexpr uint32_t kEmax = (FMT == BSQ_MXFP8) ? 8u : 2u;
  const uint32_t lane = threadIdx.x & 31u;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kThreads) >> 5;

  float g = 0.f, six_g = 0.f;
  if constexpr (NV != kMx) {
    if constexpr (NV == kNvComputed) {
      g = __fdiv_rn(__uint_as_float(a.tail[1]), 2688.0f);  // amax / (6 * 448)
    } else {
      g = *a.g_in;
    }
    six_g = __fmul_rn(6.0f, g);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      a.tail[0] = __float_as_uint(g);
      if constexpr (NV == kNvComputed) {
        if (a.g_out != nullptr) *a.g_out = g;
      }
    }
  }
  uint32_t run_max = 0;  // NVFP4 given-scale mode: running magnitude max for the tail

  // Work unit: one batch = up to kUnroll consecutive 256-element segments of one row. Warps
  // walk the batches with a grid stride and prefetch the next batch's loads before working
  // on the current one, so every warp keeps two batches of 16-byte loads in flight.
  const uint32_t bpr = static_cast<uint32_t>((a.segs_per_row + kUnroll - 1) / kUnroll);
  const uint32_t total = static_cast<uint32_t>(a.rows) * bpr;
  auto load_batch = [&](uint32_t b, Loaded<F32> (&dst)[kUnroll]) {
    const uint32_t row = b / bpr;
    const int64_t seg0 = static_cast<int64_t>(b - row * bpr) * kUnroll;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t k0 = (seg0 + u) * kSeg + lane * 8;
      if (k0 < a.cols) {
        const int64_t e = static_cast<int64_t>(row) * a.cols + k0;
        if constexpr (F32) {
          const uint4* p = reinterpret_cast<const uint4*>(static_cast<const float*>(a.src) + e);
          dst[u].v[0] = __ldcs(p);
          dst[u].v[1] = __ldcs(p + 1);
        } else {
          dst[u].v[0] = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.src) + e));
        }
      } else {
#pragma unroll
        for (int i = 0; i < (F32 ? 2 : 1); ++i) dst[u].v[i] = make_uint4(0, 0, 0, 0);
      }
    }
  };
  Loaded<F32> cur[kUnroll], nxt[kUnroll];
  uint32_t b = static_cast<uint32_t>(warp);
  if (b < total) load_batch(b, cur);
  for (; b < total; b += static_cast<uint32_t>(nwarps)) {
    const uint32_t bn = b + static_cast<uint32_t>(nwarps);
    if (bn < total) load_batch(bn, nxt);
    const uint32_t row = b / bpr;
    const int64_t seg0 = static_cast<int64_t>(b - row * bpr) * kUnroll;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (seg0 + u >= a.segs_per_row) break;  // warp-uniform
      const int64_t brow = row;
      const int64_t bk0 = (seg0 + u) * kSeg + lane * 8;
      const bool blive = bk0 < a.cols;
      float x[8];
      uint32_t mag;
      unpack8<F32>(cur[u], x, mag);
      // block maximum across the lanes of one block
      mag = max(mag, __shfl_xor_sync(0xFFFFFFFFu, mag, 1));
      if (kLanesPerBlock == 4) mag = max(mag, __shfl_xor_sync(0xFFFFFFFFu, mag, 2));
      if constexpr (NV == kNvGiven) run_max = max(run_max, mag);

      uint32_t sbyte;
      uint32_t code_lo = 0, code_hi = 0;
      if constexpr (FMT == BSQ_NVFP4) {
        uint32_t scode = 0;
        if (g != 0.0f) scode = cvt_e4m3x2(__fdiv_rn(mag_to_f32<F32>(mag), six_g), 0.0f) & 0xFFu;
        sbyte = scode;
        const float s = e4m3_to_f32(scode);
        const float sg = __fmul_rn(s, g);
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          uint32_t c;
          if (s == 0.0f) {
            c = ((__float_as_uint(x[i]) >> 31) << 3) | ((__float_as_uint(x[i + 1]) >> 31) << 7);
          } else {
            c = cvt_e2m1x2(__fdiv_rn(x[i], sg), __fdiv_rn(x[i + 1], sg));
          }
          code_lo |= c << (4 * i);
        }
      } else {
        const uint32_t ef = exp_field<F32>(mag);
        sbyte = ef > kEmax ? ef - kEmax : 0u;
        const float mul = __uint_as_float((254u - sbyte) << 23);  // 2^(127 - sbyte), exact
        if constexpr (FMT == BSQ_MXFP8) {
          code_lo = cvt_e4m3x2(x[0] * mul, x[1] * mul) | (cvt_e4m3x2(x[2] * mul, x[3] * mul) << 16);
          code_hi = cvt_e4m3x2(x[4] * mul, x[5] * mul) | (cvt_e4m3x2(x[6] * mul, x[7] * mul) << 16);
        } else {
#pragma unroll
          for (int i = 0; i < 8; i += 2) code_lo |= cvt_e2m1x2(x[i] * mul, x[i + 1] * mul) << (4 * i);
        }
      }

      if (blive) {
        const int64_t e = brow * a.cols + bk0;
        if constexpr (kFp4) {
          *reinterpret_cast<uint32_t*>(a.codes + (e >> 1)) = code_lo;
        } else {
          *reinterpret_cast<uint2*>(a.codes + e) = make_uint2(code_lo, code_hi);
        }
      } else {
        sbyte = 0;  // padding scale columns of a partial segment hold 0
      }
      // gather 4 consecutive block scales into one word: blocks are kLanesPerBlock lanes apart
      const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, sbyte, kLanesPerBlock);
      const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, sbyte, 2 * kLanesPerBlock);
      const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, sbyte, 3 * kLanesPerBlock);
      if ((lane % (4 * kLanesPerBlock)) == 0) {
        const int64_t seg_k0 = bk0 - lane * 8;
        const int64_t c4 = seg_k0 / (FMT == BSQ_NVFP4 ? 16 : 32) + lane / kLanesPerBlock;
        if (c4 < a.nsc) {
          const uint32_t word = sbyte | (s1 << 8) | (s2 << 16) | (s3 << 24);
          *reinterpret_cast<uint32_t*>(a.scales + scale_word_offset(brow, c4, a.nct)) = word;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) cur[u] = nxt[u];
  }

  if constexpr (NV == kNvGiven) {
    // per-CTA maximum of |x| -> tail word 1 (the amax of this tensor)
    __shared__ uint32_t red[kThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) run_max = max(run_max, __shfl_xor_sync(0xFFFFFFFFu, run_max, o));
    if (lane == 0) red[threadIdx.x >> 5] = run_max;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t m = 0;
      for (int i = 0; i < kThreads / 32; ++i) m = max(m, red[i]);
      atomicMax(&a.tail[1], __float_as_uint(mag_to_f32<F32>(m)));
    }
  }
}

// Tensor amax (NVFP4 computed-scale mode): max |x| -> atomicMax on the fp32 bits at `out`
// (non-negative floats order like their bit patterns). Reads use the default cache policy
// so that the quantize pass that follows finds the tensor in L2 when it fits.
template <bool F32>
__global__ void __launch_bounds__(kThreads) amax_kernel(const uint4* src, int64_t nvec, uint32_t* out) {
  constexpr int kU = 4;
  uint32_t m = 0;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t i = tid; i < nvec; i += nthr * kU) {
    uint4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t j = i + u * nthr;
      v[u] = j < nvec ? __ldg(src + j) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if constexpr (F32) {
          m = max(m, w[q] & 0x7FFFFFFFu);
        } else {
          m = max(m, max(w[q] & 0x7FFFu, (w[q] >> 16) & 0x7FFFu));
        }
      }
    }
  }
  __shared__ uint32_t red[kThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = 0;
    for (int i = 0; i < kThreads / 32; ++i) b = max(b, red[i]);
    atomicMax(out, F32 ? b : (b << 16));
  }
}

template <int FMT, bool F32, int NV>
cudaError_t launch_q(const QuantArgs& a, int grid, cudaStream_t stream) {
  quantize_kernel<FMT, F32, NV><<<grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

int launch_quantize(int fmt, bool src_f32, bool global_given, const void* src, int64_t rows, int64_t cols,
                    void* codes, void* scales, float* global_scale, cudaStream_t stream, const DeviceInfo& dev) {
  QuantArgs a{};
  a.src = src;
  a.rows = rows;
  a.cols = cols;
  a.codes = static_cast<uint8_t*>(codes);
  a.scales = static_cast<uint8_t*>(scales);
  a.nsc = cols / block_size(fmt);
  a.nct = ceil_div(a.nsc, 4);
  a.segs_per_row = ceil_div(cols, kSeg);
  a.total_segs = rows * a.segs_per_row;
  const int64_t body = scales_body_bytes(fmt, rows, cols);

  // Padding scale bytes must read 0. Padding columns of real rows are written (as zero
  // bytes inside the last scale word of a row); padding rows of the last row tile are not,
  // so that tile row is cleared first.
  cudaError_t err = cudaSuccess;
  if (rows % 128 != 0) {
    const int64_t last = (rows / 128) * a.nct * 512;
    err = cudaMemsetAsync(a.scales + last, 0, static_cast<size_t>(body - last), stream);
  }
  if (err != cudaSuccess) return BSQ_ERR_LAUNCH;

  // Persistent grid: as many CTAs as stay resident (a second wave would serialise a kernel
  // that lasts only a few microseconds), never more than there are batches of work.
  const int64_t batches = rows * ceil_div(a.segs_per_row, kUnroll);
  const int per_sm = fmt == BSQ_NVFP4 ? (src_f32 ? ctas_per_sm<BSQ_NVFP4, true>() : ctas_per_sm<BSQ_NVFP4, false>())
                                      : (src_f32 ? ctas_per_sm<BSQ_MXFP8, true>() : ctas_per_sm<BSQ_MXFP8, false>());
  const int64_t max_grid = static_cast<int64_t>(dev.num_sms) * per_sm;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(ceil_div(batches, kThreads / 32), max_grid)));

  if (fmt == BSQ_NVFP4) {
    a.tail = reinterpret_cast<uint32_t*>(a.scales + body);
    a.g_in = global_scale;
    a.g_out = global_scale;
    if (cudaMemsetAsync(a.tail, 0, 16, stream) != cudaSuccess) return BSQ_ERR_LAUNCH;
    if (!global_given) {
      const int64_t nvec = rows * cols * (src_f32 ? 4 : 2) / 16;
      const int agrid = static_cast<int>(std::min<int64_t>(ceil_div(nvec, kThreads * 4), max_grid));
      if (src_f32) amax_kernel<true><<<agrid, kThreads, 0, stream>>>(static_cast<const uint4*>(src), nvec, a.tail + 1);
      else amax_kernel<false><<<agrid, kThreads, 0, stream>>>(static_cast<const uint4*>(src), nvec, a.tail + 1);
      if (cudaGetLastError() != cudaSuccess) return BSQ_ERR_LAUNCH;
      err = src_f32 ? launch_q<BSQ_NVFP4, true, kNvComputed>(a, grid, stream)
                    : launch_q<BSQ_NVFP4, false, kNvComputed>(a, grid, stream);
    } else {
      err = src_f32 ? launch_q<BSQ_NVFP4, true, kNvGiven>(a, grid, stream)
                    : launch_q<BSQ_NVFP4, false, kNvGiven>(a, grid, stream);
    }
  } else if (fmt == BSQ_MXFP8) {
    err = src_f32 ? launch_q<BSQ_MXFP8, true, kMx>(a, grid, stream) : launch_q<BSQ_MXFP8, false, kMx>(a, grid, stream);
  } else {
    err = src_f32 ? launch_q<BSQ_MXFP4, true, kMx>(a, grid, stream) : launch_q<BSQ_MXFP4, false, kMx>(a, grid, stream);
  }
  return err == cudaSuccess ? BSQ_OK : BSQ_ERR_LAUNCH;
}

}  // namespace bsq
