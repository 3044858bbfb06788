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
// Work mapping (four CTAs per SM for MX, two for NVFP4; persistent). The source is cut into chunks of whole rows
// (or, for rows longer than a chunk, row pieces of whole 1024-element segments); a chunk is
// contiguous in memory and comes in with one 1-D TMA bulk copy. A producer thread per CTA
// keeps a ring of up to kRing chunk buffers in flight -- for a 22 MB matrix that is nearly
// every chunk of the SM's share, requested at kernel start -- and the consumer warps (dealt
// warp steps round-robin over the CTA's chunks) quantize a chunk straight from shared memory,
// walking it as one flat array: each warp step covers 1024 consecutive elements, each lane 32,
// i.e. exactly one MX block or two NVFP4 blocks, so a lane finds its block maxima without any
// shuffle and computes one scale position per block. Codes leave as 32 (E4M3) or 16 (e2m1)
// contiguous bytes per lane; each block's scale byte is stored at its place in the tiled
// layout (128 rows x 4 columns per 512-byte tile, row r at byte (r % 32) * 16 +
// ((r / 32) % 4) * 4), the lane of a row's last block also zeroing the padding columns of that
// 4-column group. Scale bytes of the padding rows of the last row tile are written as zeros by
// the kernel itself. (A lane-per-16-elements version with shuffles for the block maxima spent
// ~14 instructions per element against ~10 here.) In LayerNorm mode each warp instead owns whole
// rows of a chunk: the row's statistics, then its affine step and quantization.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "bsq_device.cuh"
#include "bsq_internal.h"

namespace bsq {
namespace {

constexpr int kLaneElems = 32;         // elements per lane per step: one MX block, two NVFP4 blocks
constexpr int kSeg = 32 * kLaneElems;   // elements per warp step
constexpr int kChunkMax = 16384;        // bytes per chunk buffer
constexpr int kChunkMin = 4096;         // smallest chunk worth a copy (small tensors)
constexpr int kAmaxThreads = 256;
constexpr int kMaxBatch = BSQ_MAX_BATCH;
constexpr int kLnMaxRows = kChunkMax / (32 * 2);  // rows of a chunk: rows of at least 32 bf16

enum NvMode { kMx = 0, kNvComputed = 1, kNvGiven = 2 };

// Occupancy per format (warp 0's lane 0 is the TMA producer, the other warps consume): MX, four
// resident CTAs of 256 threads with a 3-chunk ring each (28 consumer warps per SM to hide
// latency, 64 registers); NVFP4, whose IEEE divisions need more registers, two CTAs of 384
// threads with a 6-chunk ring (72 registers; at 64 it spilled and ran 8-15 % slower).
template <bool NV>
struct QCfg {
  static constexpr int kThreads = NV ? 384 : 256;
  static constexpr int kCtasPerSm = NV ? 2 : 4;
  static constexpr int kRing = NV ? 6 : 3;
  static constexpr int kConsumerWarps = kThreads / 32 - 1;
  static constexpr int kSmem = kRing * kChunkMax + 128;
};
inline int ctas_per_sm(int fmt) { return fmt == BSQ_NVFP4 ? QCfg<true>::kCtasPerSm : QCfg<false>::kCtasPerSm; }

struct QuantArgs {
  const uint8_t* src;
  int64_t rows, cols;
  uint8_t* codes;
  uint8_t* scales;
  uint32_t* tail;       // NVFP4: {g, amax bits, 0, 0}
  const float* g_in;    // NVFP4 given-scale mode
  float* g_out;         // NVFP4 computed mode (nullable)
  int64_t nsc;          // scale columns per row
  int64_t nct;          // 4-column scale tiles per row
  // chunking: either `rows_per_chunk` whole rows (cspan == cols) or one row piece of `cspan`
  // elements (rows_per_chunk == 1, chunks_per_row pieces per row)
  int64_t rows_per_chunk;
  int64_t cspan;
  int64_t chunks_per_row;
  int64_t nchunks;
  uint32_t cols_magic;  // floor(2^32 / cols) + 1: f / cols == umulhi(f, cols_magic) for f * cols < 2^32
  // LayerNorm mode: y = (x - mean) / sqrt(var + eps) * gamma + beta per row before quantizing
  const uint16_t* gamma;  // cols bf16
  const uint16_t* beta;   // cols bf16
  float eps;
};

// Up to kMaxBatch matrices of one format and source type quantized by one launch: their
// chunk lists are concatenated, matrix t owning global chunks [chunk_start[t], chunk_start[t+1]).
struct QuantBatch {
  int n;
  int64_t chunk_start[kMaxBatch + 1];
  QuantArgs t[kMaxBatch];
  int* status;
};

// The first N (16 or 32) source elements of one lane's piece (bf16 or fp32) -> fp32 values.
template <bool F32, int N = 32>
__device__ __forceinline__ void load32(const uint8_t* p, float* x) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  if constexpr (F32) {
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
      const uint4 v = q[i];
      x[4 * i + 0] = __uint_as_float(v.x);
      x[4 * i + 1] = __uint_as_float(v.y);
      x[4 * i + 2] = __uint_as_float(v.z);
      x[4 * i + 3] = __uint_as_float(v.w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < N / 8; ++i) {
      const uint4 v = q[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[8 * i + 2 * k] = __uint_as_float(w[k] << 16);
        x[8 * i + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
      }
    }
  }
}

// Largest |x[i]| over n values. The maximum starts at 0 and skips NaN (fmaxf returns the other
// operand), as a block maximum taken with "if (|x| > amax) amax = |x|" does.
template <int N>
__device__ __forceinline__ float abs_max(const float* x) {
  float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int i = 0; i < N; ++i) m[i & 3] = fmaxf(m[i & 3], fabsf(x[i]));
  return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

// Byte offset of the 32-bit scale word holding scale columns [c4, c4 + 4) of row r.
__device__ __forceinline__ int64_t scale_word_offset(int64_t r, int64_t c4, int64_t nct) {
  return ((r >> 7) * nct + (c4 >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
}

// Codes of 16 elements of one NVFP4 block with block maximum `amax` -> 8 bytes in w[0..1]; returns
// the block's E4M3 scale code.
__device__ __forceinline__ uint32_t nv_block16(const float* x, float amax, float g, float six_g, uint32_t* w) {
  uint32_t scode = 0;
  if (g != 0.0f) scode = cvt_e4m3x2(__fdiv_rn(amax, six_g), 0.0f) & 0xFFu;
  const float sc = e4m3_to_f32(scode);
  const float sg = __fmul_rn(sc, g);
  w[0] = w[1] = 0;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    uint32_t c;
    if (sc == 0.0f) {
      c = ((__float_as_uint(x[i]) >> 31) << 3) | ((__float_as_uint(x[i + 1]) >> 31) << 7);
    } else {
      c = cvt_e2m1x2(__fdiv_rn(x[i], sg), __fdiv_rn(x[i + 1], sg));
    }
    w[i >> 3] |= c << (4 * (i & 7));
  }
  return scode;
}

// Quantize the 32 elements of one lane: MX one block (scale byte returned in bits 0..7), NVFP4
// two blocks (scale codes in bits 0..7 and 8..15). Codes go to w: 8 words (E4M3) or 4 (e2m1).
template <int FMT>
__device__ __forceinline__ uint32_t quantize32(const float (&x)[32], float g, float six_g, uint32_t* w) {
  if constexpr (FMT == BSQ_NVFP4) {
    const uint32_t s0 = nv_block16(x, abs_max<16>(x), g, six_g, w);
    const uint32_t s1 = nv_block16(x + 16, abs_max<16>(x + 16), g, six_g, w + 2);
    return s0 | (s1 << 8);
  } else {
    constexpr uint32_t kEmax = (FMT == BSQ_MXFP8) ? 8u : 2u;
    const uint32_t ef = __float_as_uint(abs_max<32>(x)) >> 23;  // biased exponent of the block maximum
    const uint32_t sbyte = ef > kEmax ? ef - kEmax : 0u;
    const float mul = __uint_as_float((254u - sbyte) << 23);  // 2^(127 - sbyte), exact
    if constexpr (FMT == BSQ_MXFP8) {
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = cvt_e4m3x4(x[4 * i] * mul, x[4 * i + 1] * mul, x[4 * i + 2] * mul, x[4 * i + 3] * mul);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float y[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) y[k] = x[8 * i + k] * mul;
        w[i] = cvt_e2m1x8(y);
      }
    }
    return sbyte;
  }
}

template <int FMT, bool F32, int NV, bool LN>
__global__ void __launch_bounds__(QCfg<NV != kMx>::kThreads, QCfg<NV != kMx>::kCtasPerSm)
    quantize_kernel(const __grid_constant__ QuantBatch batch) {
  constexpr int kThreads = QCfg<NV != kMx>::kThreads;
  constexpr int kRing = QCfg<NV != kMx>::kRing;
  constexpr int kConsumerWarps = QCfg<NV != kMx>::kConsumerWarps;
  constexpr int kEsize = F32 ? 4 : 2;
  extern __shared__ uint8_t q_smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(q_smem_raw) + 127) & ~uintptr_t(127));
  __shared__ uint64_t full_bar[kRing], empty_bar[kRing];
  __shared__ int abort_flag;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kConsumerWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  launch_dependents();
  grid_dependency_wait();  // inputs and outputs may belong to the previous kernel until here

  const int64_t nchunks = batch.chunk_start[batch.n];
  // global chunk c -> its matrix and local chunk index
  auto chunk_owner = [&](int64_t c, int64_t& local) {
    int t = 0;
    while (t + 1 < batch.n && c >= batch.chunk_start[t + 1]) ++t;
    local = c - batch.chunk_start[t];
    return t;
  };
  // local chunk c of matrix a -> first row, rows, first column, columns
  auto chunk_geom = [&](const QuantArgs& a, int64_t c, int64_t& r0, int64_t& nr, int64_t& c0, int64_t& nc) {
    if (a.chunks_per_row > 1) {
      r0 = c / a.chunks_per_row;
      c0 = (c - r0 * a.chunks_per_row) * a.cspan;
      nr = 1;
      nc = min(a.cspan, a.cols - c0);
    } else {
      r0 = c * a.rows_per_chunk;
      nr = min(a.rows_per_chunk, a.rows - r0);
      c0 = 0;
      nc = a.cols;
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
        if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, &abort_flag, batch.status)) break;
        int64_t local;
        const QuantArgs& a = batch.t[chunk_owner(c, local)];
        int64_t r0, nr, c0, nc;
        chunk_geom(a, local, r0, nr, c0, nc);
        const uint32_t bytes = static_cast<uint32_t>(nr * nc * kEsize);
        mbar_arrive_expect_tx(&full_bar[stage], bytes);
        bulk_load(ring + stage * kChunkMax, a.src + (r0 * a.cols + c0) * kEsize, bytes, &full_bar[stage]);
        if (++stage == kRing) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    uint32_t run_max = 0;  // NVFP4 given-scale mode: running max |x| (fp32 bits) of matrix `cur`
    int cur = -1;          // matrix of the previous chunk
    float g = 0.f, six_g = 0.f;
    const int cw = static_cast<int>(warp) - 1;
    // Warp steps are dealt round-robin over the concatenation of the CTA's chunks (not per
    // chunk), so that a chunk whose step count is not a multiple of the warp count does not
    // give the same warps an extra step every time. `lead`: this warp's first step in the
    // current chunk.
    uint32_t lead = static_cast<uint32_t>(cw);
    int stage = 0;
    uint32_t phase = 0;
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
      if (!mbar_wait_bounded_warp(&full_bar[stage], phase, &abort_flag, batch.status)) break;
      int64_t local;
      const int t = chunk_owner(c, local);
      const QuantArgs& a = batch.t[t];
      if (t != cur) {
        if constexpr (NV == kNvGiven) {
          // the previous matrix's share of |x| maxima -> its tail word 1
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) run_max = max(run_max, __shfl_xor_sync(0xFFFFFFFFu, run_max, o));
          if (cur >= 0 && lane == 0 && run_max != 0) atomicMax(&batch.t[cur].tail[1], run_max);
          run_max = 0;
        }
        cur = t;
        if constexpr (NV != kMx) {
          if constexpr (NV == kNvComputed) {
            g = __fdiv_rn(__uint_as_float(a.tail[1]), 2688.0f);  // amax / (6 * 448)
          } else {
            g = *a.g_in;
          }
          six_g = __fmul_rn(6.0f, g);
        }
      }
      if constexpr (NV != kMx) {
        if (local == 0 && warp == 1 && lane == 0) {
          a.tail[0] = __float_as_uint(g);
          if constexpr (NV == kNvComputed) {
            if (a.g_out != nullptr) *a.g_out = g;
          }
        }
      }
      int64_t r0, nr, c0, nc;
      chunk_geom(a, local, r0, nr, c0, nc);
      const uint8_t* buf = ring + stage * kChunkMax;
      // the chunk as one flat array of nr * nc elements; lane piece f = 32 elements
      const uint32_t flat = static_cast<uint32_t>(nr * nc);
      const uint64_t elem0 = static_cast<uint64_t>(r0) * static_cast<uint64_t>(a.cols) + static_cast<uint64_t>(c0);
      const uint32_t steps = (flat + kSeg - 1) / kSeg;
      if constexpr (LN) {
        // LayerNorm mode (whole rows, MX formats): each warp owns whole rows of the chunk, dealt
        // round-robin over the CTA's chunks like the warp steps below (`lead` is this warp's first
        // row here): the row's mean and rstd (fp32, two passes over the row -- in registers for
        // rows of at most 1024 elements, else in shared memory -- with butterfly warp sums), then
        // y = (x - mean) * rstd * gamma + beta and the quantization of the row, 32 columns per
        // lane -- no barrier between the warps
        const int nci = static_cast<int>(nc);
        const int pieces = nci * kEsize / 16;  // 16-byte pieces of a row
        for (uint32_t rr = lead; rr < static_cast<uint32_t>(nr); rr += kConsumerWarps) {
          const uint8_t* rowp = buf + static_cast<size_t>(rr) * nci * kEsize;
          auto piece_sum = [&](float mean, bool sq) {
            float acc_s = 0.0f;
            for (int q = static_cast<int>(lane); q < pieces; q += 32) {
              const uint4 v = reinterpret_cast<const uint4*>(rowp)[q];
              const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                if constexpr (F32) {
                  const float d = __uint_as_float(w[i]) - mean;
                  acc_s += sq ? d * d : d;
                } else {
                  const float d0 = __uint_as_float(w[i] << 16) - mean, d1 = __uint_as_float(w[i] & 0xFFFF0000u) - mean;
                  acc_s += sq ? d0 * d0 + d1 * d1 : d0 + d1;
                }
              }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc_s += __shfl_xor_sync(0xFFFFFFFFu, acc_s, o);
            return acc_s;
          };
          const uint32_t row = static_cast<uint32_t>(r0) + rr;
          // y = (x - mean) * rstd * gamma + beta for the 32 elements at column cc (x holds the
          // source values), then their MX block: codes and scale byte
          auto finish = [&](int cc, float (&x)[32], float mean, float rstd) {
            const uint4* gp = reinterpret_cast<const uint4*>(a.gamma + cc);
            const uint4* bp = reinterpret_cast<const uint4*>(a.beta + cc);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const uint4 gv = __ldg(gp + h), bv = __ldg(bp + h);
              const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                float& y0 = x[8 * h + 2 * i];
                float& y1 = x[8 * h + 2 * i + 1];
                y0 = __fadd_rn(__fmul_rn(__fmul_rn(y0 - mean, rstd), __uint_as_float(gw[i] << 16)),
                               __uint_as_float(bw[i] << 16));
                y1 = __fadd_rn(__fmul_rn(__fmul_rn(y1 - mean, rstd), __uint_as_float(gw[i] & 0xFFFF0000u)),
                               __uint_as_float(bw[i] & 0xFFFF0000u));
              }
            }
            const uint64_t e = static_cast<uint64_t>(row) * static_cast<uint64_t>(a.cols) + static_cast<uint64_t>(cc);
            uint32_t w[FMT == BSQ_MXFP8 ? 8 : 4];
            const uint32_t sb = quantize32<FMT>(x, g, six_g, w);
            if constexpr (FMT == BSQ_MXFP8) {
              uint4* dst = reinterpret_cast<uint4*>(a.codes + e);
              dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
              dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            } else {
              *reinterpret_cast<uint4*>(a.codes + (e >> 1)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            const uint32_t sc = static_cast<uint32_t>(cc) >> 5;
            uint8_t* sp = a.scales + static_cast<uint64_t>((row >> 7) * static_cast<uint32_t>(a.nct) + (sc >> 2)) * 512 +
                          (((row & 31u) << 4) | (((row >> 5) & 3u) << 2) | (sc & 3u));
            *sp = static_cast<uint8_t>(sb);
            if (sc + 1 == static_cast<uint32_t>(a.nsc)) {
              for (uint32_t j = (sc & 3u) + 1; j < 4; ++j) sp[j - (sc & 3u)] = 0;
            }
          };
          if (nci <= 32 * kLaneElems) {
            // rows of at most 1024 elements: each lane reads its 32 elements from shared memory
            // once and keeps them in registers for both statistics passes and the quantization
            const int cc = static_cast<int>(lane) * kLaneElems;
            const bool act = cc < nci;
            float x[32];
            if (act) {
              load32<F32>(rowp + cc * kEsize, x);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) x[i] = 0.0f;
            }
            float p4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int i = 0; i < 32; ++i) p4[i & 3] += x[i];
            float acc_s = (p4[0] + p4[1]) + (p4[2] + p4[3]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc_s += __shfl_xor_sync(0xFFFFFFFFu, acc_s, o);
            const float mean = __fdiv_rn(acc_s, static_cast<float>(nci));
#pragma unroll
            for (int i = 0; i < 4; ++i) p4[i] = 0.0f;
            if (act) {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const float d = x[i] - mean;
                p4[i & 3] += d * d;
              }
            }
            acc_s = (p4[0] + p4[1]) + (p4[2] + p4[3]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc_s += __shfl_xor_sync(0xFFFFFFFFu, acc_s, o);
            const float var = __fdiv_rn(acc_s, static_cast<float>(nci));
            const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(var + a.eps));
            if (act) finish(cc, x, mean, rstd);
          } else {
            const float mean = __fdiv_rn(piece_sum(0.0f, false), static_cast<float>(nci));
            const float var = __fdiv_rn(piece_sum(mean, true), static_cast<float>(nci));
            const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(var + a.eps));
            for (int cc = static_cast<int>(lane) * kLaneElems; cc < nci; cc += 32 * kLaneElems) {
              float x[32];
              load32<F32>(rowp + cc * kEsize, x);
              finish(cc, x, mean, rstd);
            }
          }
        }
        lead = (lead + (kConsumerWarps - static_cast<uint32_t>(nr) % kConsumerWarps)) % kConsumerWarps;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[stage]);
        if (++stage == kRing) {
          stage = 0;
          phase ^= 1u;
        }
      } else {
        for (uint32_t base = lead * kSeg; base < flat; base += kConsumerWarps * kSeg) {
          const uint32_t f = base + lane * kLaneElems;
          // MX chunks hold whole 32-element blocks; an NVFP4 chunk may end half-way through a
          // lane's piece (rows of 16k elements): then only its first block is live
          const bool live = f < flat;
          const bool live_hi = f + 16 < flat;
          float x[32];
          if (live_hi) {
            load32<F32>(buf + f * kEsize, x);
          } else {
  #pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = 0.0f;
            if (live) load32<F32, 16>(buf + f * kEsize, x);  // the first block only: nothing past the chunk is read
          }
          if constexpr (NV == kNvGiven) run_max = max(run_max, __float_as_uint(abs_max<32>(x)));
          if (live) {
            const uint64_t e = elem0 + f;
            uint32_t w[FMT == BSQ_MXFP8 ? 8 : 4];
            const uint32_t sb = quantize32<FMT>(x, g, six_g, w);
            if constexpr (FMT == BSQ_MXFP8) {
              uint4* dst = reinterpret_cast<uint4*>(a.codes + e);
              dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
              dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            } else if constexpr (FMT == BSQ_MXFP4) {
              *reinterpret_cast<uint4*>(a.codes + (e >> 1)) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {  // NVFP4 codes are only 8-byte aligned when rows are 16k elements long
              uint2* dst = reinterpret_cast<uint2*>(a.codes + (e >> 1));
              dst[0] = make_uint2(w[0], w[1]);
              if (live_hi) dst[1] = make_uint2(w[2], w[3]);
            }
            // each block's scale byte at its place in the tiled layout (32-bit arithmetic: rows and
            // columns stay below 2^31, the number of 512-byte scale tiles below 2^32)
            constexpr int kBlocks = FMT == BSQ_NVFP4 ? 2 : 1;
  #pragma unroll
            for (int h = 0; h < kBlocks; ++h) {
              if (h == 1 && !live_hi) break;
              const uint32_t fh = f + 16u * h;
              const uint32_t rr = nr > 1 ? __umulhi(fh, a.cols_magic) : 0u;
              const uint32_t row = static_cast<uint32_t>(r0) + rr;
              const uint32_t col = static_cast<uint32_t>(c0) + (fh - rr * static_cast<uint32_t>(nc));
              const uint32_t sc = col >> (FMT == BSQ_NVFP4 ? 4 : 5);
              const uint32_t tile = (row >> 7) * static_cast<uint32_t>(a.nct) + (sc >> 2);
              uint8_t* sp = a.scales + static_cast<uint64_t>(tile) * 512 +
                            (((row & 31u) << 4) | (((row >> 5) & 3u) << 2) | (sc & 3u));
              *sp = static_cast<uint8_t>(sb >> (8 * h));
              if (sc + 1 == static_cast<uint32_t>(a.nsc)) {
                // padding columns of the row's last 4-column group read 0
                for (uint32_t j = (sc & 3u) + 1; j < 4; ++j) sp[j - (sc & 3u)] = 0;
              }
            }
          }
        }
        // first step in the next chunk: continue the round-robin where this chunk ended
        lead = (lead + (kConsumerWarps - steps % kConsumerWarps)) % kConsumerWarps;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[stage]);
        if (++stage == kRing) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }

    if constexpr (NV == kNvGiven) {
      // the last matrix's share of |x| maxima -> its tail word 1
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) run_max = max(run_max, __shfl_xor_sync(0xFFFFFFFFu, run_max, o));
      if (cur >= 0 && lane == 0 && run_max != 0) atomicMax(&batch.t[cur].tail[1], run_max);
    }
  }

  // scale bytes of the padding rows of each matrix's last row tile read 0
  for (int m = 0; m < batch.n; ++m) {
    const QuantArgs& a = batch.t[m];
    const int64_t pad_rows = (128 - a.rows % 128) % 128;
    if (pad_rows == 0) continue;
    const int64_t words = pad_rows * a.nct;
    for (int64_t w = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; w < words;
         w += static_cast<int64_t>(gridDim.x) * kThreads) {
      const int64_t r = a.rows + w / a.nct, tc = w % a.nct;
      *reinterpret_cast<uint32_t*>(a.scales + scale_word_offset(r, 4 * tc, a.nct)) = 0u;
    }
  }
}

// Tensor amax (NVFP4 computed-scale mode): max |x| over the tensor, NaN skipped like the block
// maxima -> atomicMax on the fp32 bits at `out` (non-negative floats order like their bit
// patterns). Reads use the default cache policy so that the quantize pass that follows finds
// the tensor in L2 when it fits.
template <bool F32>
__global__ void __launch_bounds__(kAmaxThreads) amax_kernel(const uint4* src, int64_t nvec, uint32_t* out) {
  constexpr int kU = 4;
  float m = 0.0f;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kAmaxThreads + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * kAmaxThreads;
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
          m = fmaxf(m, fabsf(__uint_as_float(w[q])));
        } else {
          m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[q] << 16)), fabsf(__uint_as_float(w[q] & 0xFFFF0000u))));
        }
      }
    }
  }
  __shared__ float red[kAmaxThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.0f;
    for (int i = 0; i < kAmaxThreads / 32; ++i) b = fmaxf(b, red[i]);
    atomicMax(out, __float_as_uint(b));
  }
}

template <int FMT, bool F32, int NV, bool LN = false>
cudaError_t launch_q(const QuantBatch& b, int grid, cudaStream_t stream, int device) {
  using Q = QCfg<NV != kMx>;
  static PerDevice<cudaError_t> setup;  // the shared-memory opt-in holds per device
  const cudaError_t attr = setup.run(device, [] {
    return cudaFuncSetAttribute(quantize_kernel<FMT, F32, NV, LN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Q::kSmem);
  });
  if (attr != cudaSuccess) return attr;
  // programmatic dependent launch: the kernel may be launched while the previous kernel in
  // the stream finishes; it waits for it (grid_dependency_wait) before touching memory
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Q::kThreads);
  cfg.dynamicSmemBytes = Q::kSmem;
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quantize_kernel<FMT, F32, NV, LN>, b);
}

}  // namespace

namespace {
// Delayed per-tensor scale: g = fp32(fp32(amax_prev * headroom) / 2688), amax_prev from the tail
// of an earlier NVFP4 quantization of the tensor.
__global__ void delayed_scale_kernel(const uint32_t* tail, float headroom, float* g_out) {
  grid_dependency_wait();
  *g_out = __fdiv_rn(__fmul_rn(__uint_as_float(tail[1]), headroom), 2688.0f);
  launch_dependents();
}
}  // namespace

int launch_delayed_scale(const void* prev_scales, int64_t rows, int64_t cols, float headroom, float* g_out,
                         cudaStream_t stream) {
  const uint32_t* tail = reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(prev_scales) +
                                                           scales_body_bytes(BSQ_NVFP4, rows, cols));
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(1);
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, delayed_scale_kernel, tail, headroom, g_out) == cudaSuccess ? BSQ_OK
                                                                                            : BSQ_ERR_LAUNCH;
}

int launch_amax(const void* src, bool src_f32, int64_t elems, uint32_t* out, cudaStream_t stream,
                const DeviceInfo& dev) {
  const int64_t nvec = elems * (src_f32 ? 4 : 2) / 16;
  const int agrid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(ceil_div(nvec, kAmaxThreads * 4), dev.num_sms * 8)));
  if (src_f32) amax_kernel<true><<<agrid, kAmaxThreads, 0, stream>>>(static_cast<const uint4*>(src), nvec, out);
  else amax_kernel<false><<<agrid, kAmaxThreads, 0, stream>>>(static_cast<const uint4*>(src), nvec, out);
  return cudaGetLastError() == cudaSuccess ? BSQ_OK : BSQ_ERR_LAUNCH;
}

// The batch's chunking (chunk size, per-matrix chunk counts) and per-matrix arguments.
void build_batch(QuantBatch& b, int fmt, bool src_f32, int count, const QuantItem* items, const DeviceInfo& dev) {
  const int64_t esize = src_f32 ? 4 : 2;
  b.n = count;
  b.status = dev.status;
  // Chunk size: at most one ring buffer, and small enough that every SM gets a few chunks
  // (a 5 MB matrix is then still spread over all SMs and copied in parallel).
  int64_t total_bytes = 0;
  for (int i = 0; i < count; ++i) total_bytes += items[i].rows * items[i].cols * esize;
  const int64_t target = std::max<int64_t>(
      kChunkMin, std::min<int64_t>(kChunkMax, total_bytes / (4 * ctas_per_sm(fmt) * static_cast<int64_t>(dev.num_sms))));
  b.chunk_start[0] = 0;
  for (int i = 0; i < count; ++i) {
    const QuantItem& it = items[i];
    QuantArgs& a = b.t[i];
    a.src = static_cast<const uint8_t*>(it.src);
    a.rows = it.rows;
    a.cols = it.cols;
    a.codes = static_cast<uint8_t*>(it.codes);
    a.scales = static_cast<uint8_t*>(it.scales);
    a.nsc = it.cols / block_size(fmt);
    a.nct = ceil_div(a.nsc, 4);
    a.cols_magic = static_cast<uint32_t>((uint64_t{1} << 32) / static_cast<uint64_t>(it.cols) + 1);
    const int64_t row_bytes = it.cols * esize;
    if (row_bytes <= target) {
      a.rows_per_chunk = target / row_bytes;
      a.cspan = it.cols;
      a.chunks_per_row = 1;
      a.nchunks = ceil_div(it.rows, a.rows_per_chunk);
    } else {
      a.rows_per_chunk = 1;
      a.cspan = std::max<int64_t>(1, kChunkMax / (esize * kSeg)) * kSeg;  // whole segments per piece
      a.chunks_per_row = ceil_div(it.cols, a.cspan);
      a.nchunks = it.rows * a.chunks_per_row;
    }
    b.chunk_start[i + 1] = b.chunk_start[i] + a.nchunks;
    if (fmt == BSQ_NVFP4) {
      a.tail = reinterpret_cast<uint32_t*>(a.scales + scales_body_bytes(fmt, it.rows, it.cols));
      a.g_in = it.global_scale;
      a.g_out = it.global_scale;
    }
  }
}

int launch_quantize_batch(int fmt, bool src_f32, bool global_given, int count, const QuantItem* items,
                          cudaStream_t stream, const DeviceInfo& dev) {
  if (count < 1 || count > kMaxBatch) return BSQ_ERR_ARG;
  QuantBatch b{};
  build_batch(b, fmt, src_f32, count, items, dev);
  const int grid =
      static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(b.chunk_start[count], ctas_per_sm(fmt) * dev.num_sms)));

  cudaError_t err = cudaSuccess;
  if (fmt == BSQ_NVFP4) {
    for (int i = 0; i < count; ++i) {
      const QuantArgs& a = b.t[i];
      if (cudaMemsetAsync(a.tail, 0, 16, stream) != cudaSuccess) return BSQ_ERR_LAUNCH;
      if (!global_given && launch_amax(a.src, src_f32, a.rows * a.cols, a.tail + 1, stream, dev) != BSQ_OK)
        return BSQ_ERR_LAUNCH;
    }
    if (!global_given) {
      err = src_f32 ? launch_q<BSQ_NVFP4, true, kNvComputed>(b, grid, stream, dev.device)
                    : launch_q<BSQ_NVFP4, false, kNvComputed>(b, grid, stream, dev.device);
    } else {
      err = src_f32 ? launch_q<BSQ_NVFP4, true, kNvGiven>(b, grid, stream, dev.device)
                    : launch_q<BSQ_NVFP4, false, kNvGiven>(b, grid, stream, dev.device);
    }
  } else if (fmt == BSQ_MXFP8) {
    err = src_f32 ? launch_q<BSQ_MXFP8, true, kMx>(b, grid, stream, dev.device) : launch_q<BSQ_MXFP8, false, kMx>(b, grid, stream, dev.device);
  } else {
    err = src_f32 ? launch_q<BSQ_MXFP4, true, kMx>(b, grid, stream, dev.device) : launch_q<BSQ_MXFP4, false, kMx>(b, grid, stream, dev.device);
  }
  return err == cudaSuccess ? BSQ_OK : BSQ_ERR_LAUNCH;
}

int launch_layernorm_quantize(int fmt, bool src_f32, const QuantItem& item, const uint16_t* gamma,
                              const uint16_t* beta, float eps, cudaStream_t stream, const DeviceInfo& dev) {
  QuantBatch b{};
  build_batch(b, fmt, src_f32, 1, &item, dev);
  if (b.t[0].chunks_per_row != 1 || b.t[0].rows_per_chunk > kLnMaxRows) return BSQ_ERR_SHAPE;  // whole rows only
  b.t[0].gamma = gamma;
  b.t[0].beta = beta;
  b.t[0].eps = eps;
  const int grid =
      static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(b.chunk_start[1], ctas_per_sm(fmt) * dev.num_sms)));
  cudaError_t err;
  if (fmt == BSQ_MXFP8) {
    err = src_f32 ? launch_q<BSQ_MXFP8, true, kMx, true>(b, grid, stream, dev.device) : launch_q<BSQ_MXFP8, false, kMx, true>(b, grid, stream, dev.device);
  } else {
    err = src_f32 ? launch_q<BSQ_MXFP4, true, kMx, true>(b, grid, stream, dev.device) : launch_q<BSQ_MXFP4, false, kMx, true>(b, grid, stream, dev.device);
  }
  return err == cudaSuccess ? BSQ_OK : BSQ_ERR_LAUNCH;
}

}  // namespace bsq
