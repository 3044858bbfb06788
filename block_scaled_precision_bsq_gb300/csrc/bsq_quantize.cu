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
// Work mapping. bsq_quantize / bsq_quantize_batch run stream_kernel: every matrix of a batch is
// one flat array, a warp step is 1024 consecutive elements of one matrix and a lane's piece 32 of
// them -- one MX block, two NVFP4 blocks -- loaded straight into registers (two 32-byte loads for
// bf16; the MX formats one step ahead of the piece being quantized); no shared-memory staging
// and no barriers, so the instructions are the element arithmetic itself: block maxima on packed
// bf16 pairs, the scaling (MX: a power of two) or the IEEE quotient (NVFP4: Markstein's remainder
// step from a table of correctly rounded reciprocals) on packed fp32 pairs, cvt.rn.satfinite to
// E4M3 / e2m1. Codes leave as 32 (E4M3) or 16 (e2m1) contiguous bytes per lane; each block's scale
// byte is stored at its place in the tiled layout (128 rows x 4 columns per 512-byte tile, row r at
// byte (r % 32) * 16 + ((r / 32) % 4) * 4), as 32-bit words of two lanes for NVFP4 when the row
// length allows; the padding of the tiled scales is zeroed after the loop. NVFP4 with a computed
// per-tensor scale first runs amax_kernel, one launch over every matrix of the batch.
// bsq_layernorm_quantize runs ln_stream_kernel for bf16 rows of at most 1024 elements (one row per
// warp step, in registers) and layernorm_kernel otherwise: chunks of whole rows brought into
// shared memory by 1-D TMA bulk copies, each consumer warp owning whole rows (the row's
// statistics, then its affine step and quantization).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "bsq_device.cuh"
#include "bsq_internal.h"

namespace bsq {
namespace {

constexpr int kLaneElems = 32;         // elements per lane per step: one MX block, two NVFP4 blocks
constexpr int kChunkMax = 16384;        // bytes per chunk buffer
constexpr int kChunkMin = 4096;         // smallest chunk worth a copy (small tensors)
constexpr int kAmaxThreads = 256;
constexpr int kMaxBatch = BSQ_MAX_BATCH;
constexpr int kLnMaxRows = kChunkMax / (32 * 2);  // rows of a chunk: rows of at least 32 bf16

enum NvMode { kMx = 0, kNvComputed = 1, kNvGiven = 2 };

// LayerNorm kernel: four resident CTAs of 256 threads per SM (warp 0's lane 0 is the TMA producer,
// the other warps consume), a 3-chunk ring each.
struct QCfg {
  static constexpr int kThreads = 256;
  static constexpr int kCtasPerSm = 4;
  static constexpr int kRing = 3;
  static constexpr int kConsumerWarps = kThreads / 32 - 1;
  static constexpr int kSmem = kRing * kChunkMax + 128;
};

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
  int64_t rows_per_chunk;  // LayerNorm kernel: whole rows per chunk
  uint32_t cols_magic;  // floor(2^32 / cols) + 1: f / cols == umulhi(f, cols_magic) for f * cols < 2^32
  uint64_t cols_magic64;  // floor((2^64 - 1) / cols): f / cols is umul64hi(f, .) or one more
  int64_t elems;        // rows * cols
  int64_t codes_bytes;  // sizes of the code buffer and of the tiled scale body (index checks)
  int64_t scales_bytes;
  bool scale_words;     // NVFP4 with cols a multiple of 64: scale bytes stored as words
  // LayerNorm mode: y = (x - mean) / sqrt(var + eps) * gamma + beta per row before quantizing
  const uint16_t* gamma;  // cols bf16
  const uint16_t* beta;   // cols bf16
  float eps;
};

// Up to kMaxBatch matrices of one format and source type quantized by one launch: their
// chunk lists are concatenated, matrix t owning global chunks [chunk_start[t], chunk_start[t+1]).
struct QuantBatch {
  int n;
  int64_t chunk_start[kMaxBatch + 1];  // LayerNorm kernel: chunks; streaming kernel: warp steps
  QuantArgs t[kMaxBatch];
  int* status;
  int64_t stall_after;  // LayerNorm kernel, injected stall (tests): loads stop after this many chunks; -1 = none
  uint64_t wait_ns;     // LayerNorm kernel: limit of every bounded wait
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

// NVFP4 divisors of one matrix: g, 6 g and its reciprocal, and a table holding for every E4M3
// scale code s the block divisor d = fp32(s g) and r = fp32(1 / d) (NaN where the remainder step
// of markstein_quotient is not valid for that d: the block then divides).
struct NvCtx {
  float g = 0.0f, six_g = 0.0f, r6 = 0.0f;
  const float2* tab = nullptr;
};

// Fill `tab` (128 entries, shared by the warp's lanes) for per-tensor scale g; returns the
// context. Called by the whole warp.
// With g = 0 the scale quotient is taken as amax * 0 (r6 = 0): every block scale is then 0. The
// entry of scale code 0 is {0, 0}: the quotient step then yields a zero carrying the sign of x,
// the code the format's rule gives a block whose scale is 0.
__device__ __forceinline__ NvCtx nv_context(float g, float2* tab) {
  NvCtx c;
  c.g = g;
  c.six_g = __fmul_rn(6.0f, g);
  const float r6 = __frcp_rn(c.six_g);
  if (g == 0.0f) {
    c.r6 = 0.0f;
  } else {
    c.r6 = markstein_ok(c.six_g, r6, 0.0f) ? r6 : __uint_as_float(0x7FC00000u);
  }
  __syncwarp();  // every lane is done with the previous matrix's table
  for (uint32_t code = lane_id(); code < 128u; code += 32u) {
    const float d = __fmul_rn(e4m3_to_f32(code), g);
    const float r = __frcp_rn(d);
    tab[code] = code == 0u ? make_float2(0.0f, 0.0f)
                           : make_float2(d, markstein_ok(d, r, 0.0f) ? r : __uint_as_float(0x7FC00000u));
  }
  __syncwarp();
  c.tab = tab;
  return c;
}

// Codes of 16 elements of one NVFP4 block with block maximum `amax` -> 8 bytes in w[0..1]; returns
// the block's E4M3 scale code s = E4M3(fp32(amax / fp32(6 g))), then e2m1(fp32(x / fp32(s g)))
// per element, both quotients the IEEE ones (markstein_quotient where valid, else the division).
__device__ __forceinline__ uint32_t nv_block16(const float* x, float amax, const NvCtx& c, uint32_t* w) {
  uint32_t scode = 0;
  if (c.g != 0.0f) {
    float qs;
    if (__fmul_rn(amax, c.r6) < 0x1p100f) qs = markstein_quotient(amax, c.six_g, c.r6);
    else qs = __fdiv_rn(amax, c.six_g);
    scode = cvt_e4m3x2(qs, 0.0f) & 0xFFu;
  }
  if (scode == 0u) {  // s = 0: zero codes carrying the sign of each element
    uint32_t c0 = 0, c1 = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      c0 |= (__float_as_uint(x[i]) >> 31) << (4 * i + 3);
      c1 |= (__float_as_uint(x[8 + i]) >> 31) << (4 * i + 3);
    }
    w[0] = c0;
    w[1] = c1;
    return 0u;
  }
  const float2 dr = c.tab[scode];
  float q[16];
  if (__fmul_rn(amax, dr.y) < 0x1p100f) {
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = markstein_quotient(x[i], dr.x, dr.y);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = __fdiv_rn(x[i], dr.x);
  }
  w[0] = cvt_e2m1x8(q);
  w[1] = cvt_e2m1x8(q + 8);
  return scode;
}

// ---------------------------------------------------------------------------- bf16 fast paths
// max(|a|, |b|) of each bf16 half (the result's sign bits are those of a and b XOR-ed; callers
// mask them); a NaN operand gives the other one, as fmaxf does.
__device__ __forceinline__ uint32_t bf16x2_maxabs(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Largest |x| of the 2 N bf16 values in w[0..N) (N a power of two), as an fp32 value (exact).
template <int N>
__device__ __forceinline__ float bf16_block_amax(const uint32_t* w) {
  uint32_t m[N];
#pragma unroll
  for (int i = 0; i < N; ++i) m[i] = w[i];
#pragma unroll
  for (int n = N / 2; n >= 1; n /= 2) {
#pragma unroll
    for (int i = 0; i < n; ++i) m[i] = bf16x2_maxabs(m[i], m[i + n]);
  }
  return __uint_as_float(max(m[0] & 0x7FFFu, (m[0] >> 16) & 0x7FFFu) << 16);
}

// The bf16 pair of word v as packed fp32 (element 2i of the word in the low lane).
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t v) {
  return f2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// MX block of one lane: 32 bf16 values in raw[0..16) -> codes in w (8 words E4M3, 4 e2m1);
// returns the scale byte. The same rule as quantize32, on packed pairs.
template <int FMT>
__device__ __forceinline__ uint32_t mx_piece_bf16(const uint32_t* raw, uint32_t* w) {
  constexpr uint32_t kEmax = (FMT == BSQ_MXFP8) ? 8u : 2u;
  const uint32_t ef = __float_as_uint(bf16_block_amax<16>(raw)) >> 23;  // biased exponent of the block maximum
  const uint32_t sbyte = ef > kEmax ? ef - kEmax : 0u;
  const uint64_t m2 = f2_splat(__uint_as_float((254u - sbyte) << 23));  // 2^(127 - sbyte), exact
  if constexpr (FMT == BSQ_MXFP8) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float a, b, c, d;
      f2_split(f2_mul(bf16x2_to_f2(raw[2 * j]), m2), a, b);
      f2_split(f2_mul(bf16x2_to_f2(raw[2 * j + 1]), m2), c, d);
      w[j] = cvt_e4m3x4(a, b, c, d);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float y[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) f2_split(f2_mul(bf16x2_to_f2(raw[4 * j + i]), m2), y[2 * i], y[2 * i + 1]);
      w[j] = cvt_e2m1x8(y);
    }
  }
  return sbyte;
}

// NVFP4 blocks of one lane: 32 bf16 values in raw[0..16) -> codes in w[0..4), scale codes in bits
// 0..7 and 8..15 of `sb`. Quotients by markstein_quotient's remainder step in packed form, with
// the reciprocal negated: q0' = x (-r) = -q0, t = q0' d + x (the exact remainder x - q0 d), y =
// t (-r) + q0' = -(q0 + t r), the negated IEEE quotient, whose code is the quotient's with the sign
// flipped back by one XOR per eight codes. Working on -q keeps signed zeros exact without
// negating x (x = +-0 gives -+0). Returns false when the step is not valid for some block (then
// the caller takes the exact path).
__device__ __forceinline__ bool nv_piece_bf16(const uint32_t* raw, const NvCtx& c, uint32_t* w, uint32_t& sb) {
  bool quick = true;
  sb = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t* wb = raw + 8 * h;
    const float amax = bf16_block_amax<8>(wb);
    quick = quick && __fmul_rn(amax, c.r6) < 0x1p100f;
    const uint32_t scode = cvt_e4m3x2(markstein_quotient(amax, c.six_g, c.r6), 0.0f) & 0xFFu;
    const float2 dr = c.tab[scode];
    quick = quick && __fmul_rn(amax, dr.y) < 0x1p100f;
    sb |= scode << (8 * h);
    const uint64_t d2 = f2_splat(dr.x), nr2 = f2_splat(-dr.y);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float y[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint64_t x2 = bf16x2_to_f2(wb[4 * j + i]);
        const uint64_t q0 = f2_mul(x2, nr2);
        f2_split(f2_fma(f2_fma(q0, d2, x2), nr2, q0), y[2 * i], y[2 * i + 1]);
      }
      w[2 * h + j] = cvt_e2m1x8(y) ^ 0x88888888u;
    }
  }
  return quick;
}

// Quantize the 32 elements of one lane: MX one block (scale byte returned in bits 0..7), NVFP4
// two blocks (scale codes in bits 0..7 and 8..15). Codes go to w: 8 words (E4M3) or 4 (e2m1).
template <int FMT>
__device__ __forceinline__ uint32_t quantize32(const float (&x)[32], const NvCtx& nv, uint32_t* w) {
  if constexpr (FMT == BSQ_NVFP4) {
    const uint32_t s0 = nv_block16(x, abs_max<16>(x), nv, w);
    const uint32_t s1 = nv_block16(x + 16, abs_max<16>(x + 16), nv, w + 2);
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

// ---------------------------------------------------------------------------- streaming kernel
// Every matrix of the batch is one flat array of rows * cols elements; a warp step is 1024
// consecutive elements of one matrix and a lane's piece 32 of them (one MX block, two NVFP4
// blocks: a piece never crosses a row for MX, cols being a multiple of 32; an NVFP4 piece may
// when cols % 32 == 16, and each block then finds its own row). Warps walk the concatenated step
// list with a grid-wide stride, each lane loading its piece straight from global memory into
// registers (two 32-byte loads for bf16, whole sectors): no shared-memory staging, no barriers, so
// nearly every instruction is the element arithmetic. After the NVFP4 amax pass (which reads
// every source front to back) the step list is walked back to front, to meet the lines still in
// L2.
// Latency hiding, per SM: the MX formats from bf16 load each piece one step ahead of the piece
// they quantize, with three CTAs (up to 80 registers); NVFP4 from bf16 keeps no second piece in
// registers and relies on three CTAs (up to 80 registers) alone; fp32 sources prefetch with two
// CTAs (up to 128). Measured on GB300 (51200 x 4096 bf16, L2 flushed): NVFP4 (amax pass
// included) 192 us this way against 200 us with the prefetch at two CTAs, 191-230 us at 128
// threads per CTA with 4 to 6 CTAs; MXFP8 103.3 us with three CTAs against 115.8 with two and
// 110.8 with four. A deeper prefetch ring in shared memory (cp.async, 2 to 8 pieces per thread)
// gained nothing for NVFP4 and lost 8-10% for the MX formats.
constexpr int kSThreads = 256;
template <bool F32, bool NV>
struct SCfg {
  static constexpr bool kPrefetch = F32 || !NV;
  static constexpr int kCtasPerSm = F32 ? 2 : 3;
};
constexpr int kSWarps = kSThreads / 32;

// f / cols for f < 2^63: one 64-bit high multiply and at most one correction.
__device__ __forceinline__ int64_t div_cols(int64_t f, int64_t cols, uint64_t magic) {
  int64_t q = static_cast<int64_t>(__umul64hi(static_cast<uint64_t>(f), magic));
  if (f - q * cols >= cols) ++q;
  return q;
}

// Read-only 32-byte and 16-byte loads that do not allocate in L1 (each byte is read once).
__device__ __forceinline__ void ld32(const uint8_t* p, uint32_t* r) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "l"(p));
}
__device__ __forceinline__ void ld16(const uint8_t* p, uint32_t* r) {
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "l"(p));
}

// One lane's piece in flight: its matrix, element index and source words.
template <bool F32>
struct Piece {
  static constexpr int kWords = F32 ? 32 : 16;
  int t;      // matrix
  int64_t f;  // first element of the piece in the matrix
  int live;   // elements present: 32, 16 (NVFP4: the matrix ends after the first block) or 0
  uint32_t w[kWords];
};

// The fields of one batch matrix a warp works with, held in registers while its steps last
// (the batch itself lives in the constant bank, where a dynamically indexed read costs an
// address computation and a load every time).
struct Mat {
  int t = -1;
  int64_t s0 = 0, s1 = 0;  // its warp steps [s0, s1) in the concatenated list
  const uint8_t* src;
  uint8_t* codes;
  uint8_t* scales;
  int64_t elems, cols, nct;
  uint64_t magic;
  bool aligned32;
  int64_t codes_bytes, scales_bytes;
  bool words;  // NVFP4: every 4-column group of scale bytes lies in one row and one lane pair
};

__device__ __forceinline__ Mat find_mat(const QuantBatch& b, int64_t s) {
  int t = 0;
  while (t + 1 < b.n && s >= b.chunk_start[t + 1]) ++t;
  const QuantArgs& a = b.t[t];
  Mat m;
  m.t = t;
  m.s0 = b.chunk_start[t];
  m.s1 = b.chunk_start[t + 1];
  m.src = a.src;
  m.codes = a.codes;
  m.scales = a.scales;
  m.elems = a.elems;
  m.cols = a.cols;
  m.nct = a.nct;
  m.magic = a.cols_magic64;
  m.aligned32 = (reinterpret_cast<uintptr_t>(a.src) & 31u) == 0u;
  m.codes_bytes = a.codes_bytes;
  m.scales_bytes = a.scales_bytes;
  m.words = a.scale_words;
  return m;
}

template <int FMT, bool F32, int NV>
__global__ void __launch_bounds__(kSThreads, SCfg<F32, NV != kMx>::kCtasPerSm)
    stream_kernel(const __grid_constant__ QuantBatch batch) {
  __shared__ float2 nv_tab[NV != kMx ? kSWarps : 1][128];  // NVFP4: each warp's divisor table
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  launch_dependents();
  grid_dependency_wait();  // inputs and outputs may belong to the previous kernel until here

  const int64_t nsteps = batch.chunk_start[batch.n];
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kSWarps;
  auto step_of = [&](int64_t k) { return NV == kNvComputed ? nsteps - 1 - k : k; };
  uint32_t run_max = 0;  // NVFP4 given-scale mode: running max |x| (fp32 bits) of matrix mp
  NvCtx nv;
  Mat mf, mp;  // the matrix of the step being fetched, and of the step being quantized
  constexpr int kBytes = F32 ? 128 : 64;

  // load this lane's piece of global step s (zeros where the matrix has ended)
  auto fetch = [&](Piece<F32>& p, int64_t s) {
    if (s < mf.s0 || s >= mf.s1) mf = find_mat(batch, s);  // warp-uniform
    p.t = mf.t;
    p.f = (s - mf.s0) * 1024 + 32 * static_cast<int64_t>(lane);
    int64_t left = mf.elems - p.f;
    if (!in_bounds(p.f >= 0, batch.status)) left = 0;
    const uint8_t* src = mf.src + p.f * (F32 ? 4 : 2);
    if (left >= 32) {
      p.live = 32;
      if (mf.aligned32) {
#pragma unroll
        for (int i = 0; i < kBytes / 32; ++i) ld32(src + 32 * i, p.w + 8 * i);
      } else {
#pragma unroll
        for (int i = 0; i < kBytes / 16; ++i) ld16(src + 16 * i, p.w + 4 * i);
      }
    } else {
      p.live = left >= 16 ? 16 : 0;
#pragma unroll
      for (int i = 0; i < Piece<F32>::kWords; ++i) p.w[i] = 0u;
      if (p.live == 16) {
#pragma unroll
        for (int i = 0; i < kBytes / 32; ++i) ld16(src + 16 * i, p.w + 4 * i);
      }
    }
  };

  // quantize one fetched piece
  auto process = [&](Piece<F32>& p) {
    if (p.t != mp.t) {  // warp-uniform: a step lies in one matrix
      if constexpr (NV == kNvGiven) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) run_max = max(run_max, __shfl_xor_sync(0xFFFFFFFFu, run_max, o));
        if (mp.t >= 0 && lane == 0 && run_max != 0) atomicMax(&batch.t[mp.t].tail[1], run_max);
        run_max = 0;
      }
      mp = find_mat(batch, p.t == mf.t ? mf.s0 : batch.chunk_start[p.t]);
      if constexpr (NV != kMx) {
        const QuantArgs& a = batch.t[p.t];
        const float g = NV == kNvComputed ? __fdiv_rn(__uint_as_float(a.tail[1]), 2688.0f)  // amax / (6 * 448)
                                         : *a.g_in;
        nv = nv_context(g, nv_tab[NV != kMx ? warp : 0]);
      }
    }
    if constexpr (NV != kMx) {
      if (p.f == 0) {  // the matrix's first piece records g
        const QuantArgs& a = batch.t[p.t];
        a.tail[0] = __float_as_uint(nv.g);
        if constexpr (NV == kNvComputed) {
          if (a.g_out != nullptr) *a.g_out = nv.g;
        }
      }
    }
    const bool live = p.live != 0;  // lanes past the matrix's end still take part in the shuffles
    uint32_t w[FMT == BSQ_MXFP8 ? 8 : 4];
    uint32_t sb = 0;
    // the piece's values as fp32 (exact path): fp32 sources, and NVFP4 blocks whose quotient step is
    // not valid
    auto exact = [&]() {
      float x[32];
      if constexpr (F32) {
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(p.w[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          x[2 * i] = __uint_as_float(p.w[i] << 16);
          x[2 * i + 1] = __uint_as_float(p.w[i] & 0xFFFF0000u);
        }
      }
      if constexpr (F32 && NV == kNvGiven) run_max = max(run_max, __float_as_uint(abs_max<32>(x)));
      sb = quantize32<FMT>(x, nv, w);
    };
    if (live) {
      if constexpr (F32) {
        exact();
      } else if constexpr (FMT == BSQ_NVFP4) {
        if constexpr (NV == kNvGiven) run_max = max(run_max, __float_as_uint(bf16_block_amax<16>(p.w)));
        if (!nv_piece_bf16(p.w, nv, w, sb)) exact();
      } else {
        sb = mx_piece_bf16<FMT>(p.w, w);
      }
      // codes: the piece's 32 (E4M3) or 16 (e2m1; 8 if only the first NVFP4 block is present)
      // bytes at code byte f (E4M3) or f / 2, 16-byte aligned since f is a multiple of 32
      const int64_t cb = (FMT == BSQ_MXFP8) ? p.f : (p.f >> 1);
      const int64_t cn = (FMT == BSQ_MXFP8) ? 32 : p.live / 2;
      if (in_bounds(cb >= 0 && cb + cn <= mp.codes_bytes, batch.status)) {
        if constexpr (FMT == BSQ_MXFP8) {
          uint4* dst = reinterpret_cast<uint4*>(mp.codes + cb);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        } else if (p.live == 32) {
          *reinterpret_cast<uint4*>(mp.codes + cb) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
          *reinterpret_cast<uint2*>(mp.codes + cb) = make_uint2(w[0], w[1]);
        }
      }
    }
    // scale bytes at their places in the tiled layout (rows and columns below 2^31)
    if (FMT == BSQ_NVFP4 && mp.words) {
      // cols a multiple of 64: the 4 scale bytes of each aligned 4-column group of a row are the
      // two blocks of an even lane and of the next lane, whose 32-bit word the even lane stores
      // (one store where there were four byte stores into the same word; measured on GB300 the
      // same for MXFP4 / MXFP8 with 4-lane groups, so those keep their byte stores)
      const uint32_t v = sb & 0xFFFFu;
      const uint32_t word = v | (__shfl_down_sync(0xFFFFFFFFu, v, 1) << 16);
      if (live && (lane & 1u) == 0u) {
        const int64_t row64 = div_cols(p.f, mp.cols, mp.magic);
        const uint32_t r = static_cast<uint32_t>(row64);
        const uint32_t sc = static_cast<uint32_t>(p.f - row64 * mp.cols) >> 4;
        const uint64_t tile = static_cast<uint64_t>(r >> 7) * static_cast<uint64_t>(mp.nct) + (sc >> 2);
        const uint64_t so = tile * 512 + (((r & 31u) << 4) | (((r >> 5) & 3u) << 2));
        if (in_bounds(so + 4 <= static_cast<uint64_t>(mp.scales_bytes), batch.status))
          *reinterpret_cast<uint32_t*>(mp.scales + so) = word;
      }
    } else if (live) {
      // byte stores (the padding columns of the last 4-column group are zeroed after the loop)
      const int64_t row64 = div_cols(p.f, mp.cols, mp.magic);
      const uint32_t row = static_cast<uint32_t>(row64);
      const uint32_t col = static_cast<uint32_t>(p.f - row64 * mp.cols);
      constexpr int kBlocks = FMT == BSQ_NVFP4 ? 2 : 1;
#pragma unroll
      for (int h = 0; h < kBlocks; ++h) {
        if (h == 1 && p.live != 32) break;
        uint32_t r = row, c = col + 16u * h;
        if (FMT == BSQ_NVFP4 && c >= static_cast<uint32_t>(mp.cols)) {  // cols % 32 == 16: the next row
          c -= static_cast<uint32_t>(mp.cols);
          ++r;
        }
        const uint32_t sc = c >> (FMT == BSQ_NVFP4 ? 4 : 5);
        const uint64_t tile = static_cast<uint64_t>(r >> 7) * static_cast<uint64_t>(mp.nct) + (sc >> 2);
        const uint64_t so = tile * 512 + (((r & 31u) << 4) | (((r >> 5) & 3u) << 2) | (sc & 3u));
        if (in_bounds(so < static_cast<uint64_t>(mp.scales_bytes), batch.status))
          mp.scales[so] = static_cast<uint8_t>(sb >> (8 * h));
      }
    }
  };

  Piece<F32> pa, pb;
  int64_t k = static_cast<int64_t>(blockIdx.x) * kSWarps + warp;
  if constexpr (SCfg<F32, NV != kMx>::kPrefetch) {
    // two piece buffers, alternating: the next step's loads are in flight while this one is
    // quantized
    if (k < nsteps) fetch(pa, step_of(k));
    while (k < nsteps) {
      if (k + nw < nsteps) fetch(pb, step_of(k + nw));
      process(pa);
      k += nw;
      if (k >= nsteps) break;
      if (k + nw < nsteps) fetch(pa, step_of(k + nw));
      process(pb);
      k += nw;
    }
  } else {
    // one buffer: the loads of other warps cover this warp's quantization
    for (; k < nsteps; k += nw) {
      fetch(pa, step_of(k));
      process(pa);
    }
  }
  if constexpr (NV == kNvGiven) {
    // the last matrix's share of |x| maxima -> its tail word 1
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) run_max = max(run_max, __shfl_xor_sync(0xFFFFFFFFu, run_max, o));
    if (mp.t >= 0 && lane == 0 && run_max != 0) atomicMax(&batch.t[mp.t].tail[1], run_max);
  }
  // padding of the tiled scales reads 0: every word of the padding rows of each matrix's last row
  // tile, and the bytes past the last scale column in each row's last 4-column group (byte
  // stores: the row's real scale bytes in the same word are written by other lanes)
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kSThreads + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * kSThreads;
  for (int m = 0; m < batch.n; ++m) {
    const QuantArgs& a = batch.t[m];
    const int64_t pad_rows = (128 - a.rows % 128) % 128;
    const int64_t words = pad_rows * a.nct;
    for (int64_t wd = tid; wd < words; wd += nthr) {
      const int64_t r = a.rows + wd / a.nct, tc = wd % a.nct;
      const int64_t so = scale_word_offset(r, 4 * tc, a.nct);
      if (in_bounds(so + 4 <= a.scales_bytes, batch.status)) *reinterpret_cast<uint32_t*>(a.scales + so) = 0u;
    }
    const int64_t pad_cols = 4 * a.nct - a.nsc;
    for (int64_t i = tid; i < a.rows * pad_cols; i += nthr) {
      const int64_t r = i / pad_cols, c = a.nsc + i % pad_cols;
      const int64_t so = scale_word_offset(r, c, a.nct) + (c & 3);
      if (in_bounds(so < a.scales_bytes, batch.status)) a.scales[so] = 0;
    }
  }
}

// ---------------------------------------------------------------------------- LayerNorm rows
// Statistics of a row of at most 1024 elements held in registers, 32 per lane (zeros in lanes
// past the row's end, act = false there): mean = sum / n and var = sum (x - mean)^2 / n in fp32
// (two passes, each lane's four running sums of every fourth element, then a butterfly warp
// sum), rstd = 1 / sqrt(var + eps). Every warp of the row gets the same values.
__device__ __forceinline__ void ln_row_stats(const float (&x)[32], bool act, int n, float eps, float& mean,
                                             float& rstd) {
  float p4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int i = 0; i < 32; ++i) p4[i & 3] += x[i];
  float acc_s = (p4[0] + p4[1]) + (p4[2] + p4[3]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc_s += __shfl_xor_sync(0xFFFFFFFFu, acc_s, o);
  mean = __fdiv_rn(acc_s, static_cast<float>(n));
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
  const float var = __fdiv_rn(acc_s, static_cast<float>(n));
  rstd = __fdiv_rn(1.0f, __fsqrt_rn(var + eps));
}

// y = (x - mean) * rstd * gamma + beta for the 32 elements of row `row` at column cc (x holds the
// source values; each step rounded in fp32), then their MX block: codes and scale byte (the
// padding columns of the row's last 4-column scale group are zeroed by the lane of the row's last
// block).
template <int FMT>
__device__ __forceinline__ void ln_finish(const QuantArgs& a, int* status, uint32_t row, int cc, float (&x)[32],
                                          float mean, float rstd) {
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
  const uint32_t sb = quantize32<FMT>(x, NvCtx(), w);
  const uint64_t cb = (FMT == BSQ_MXFP8) ? e : (e >> 1);
  if (in_bounds(cb + (FMT == BSQ_MXFP8 ? 32 : 16) <= static_cast<uint64_t>(a.codes_bytes), status)) {
    if constexpr (FMT == BSQ_MXFP8) {
      uint4* dst = reinterpret_cast<uint4*>(a.codes + e);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
      *reinterpret_cast<uint4*>(a.codes + (e >> 1)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  const uint32_t sc = static_cast<uint32_t>(cc) >> 5;
  const uint64_t so = static_cast<uint64_t>((row >> 7) * static_cast<uint32_t>(a.nct) + (sc >> 2)) * 512 +
                      (((row & 31u) << 4) | (((row >> 5) & 3u) << 2) | (sc & 3u));
  if (in_bounds(so + (4 - (sc & 3u)) <= static_cast<uint64_t>(a.scales_bytes), status)) {
    uint8_t* sp = a.scales + so;
    *sp = static_cast<uint8_t>(sb);
    if (sc + 1 == static_cast<uint32_t>(a.nsc)) {
      for (uint32_t j = (sc & 3u) + 1; j < 4; ++j) sp[j - (sc & 3u)] = 0;
    }
  }
}

// ---------------------------------------------------------------------------- LayerNorm, streaming
// LayerNorm + MX quantization of bf16 rows of at most 1024 elements (ViT-B's 768 and ViT-L's 1024
// channels): one row per warp step, lane l holding columns [32 l, 32 l + 32) in registers -- loaded
// straight from global memory -- for both statistics passes, the affine step and the quantization
// (ln_row_stats, ln_finish: the arithmetic of the shared-memory kernel below, so both give the
// same bytes). No shared memory, no barriers: 32 warps per SM, each with its own row, hide the
// latency of a row's loads and two warp reductions. Measured on GB300 (bf16 51200 x 1024 -> MXFP4,
// L2 flushed): 43 us, against 55 us for the shared-memory kernel; 44.6 us with 3 CTAs per SM and
// 50.2 us with the next row prefetched into registers at 3 CTAs (its 80 registers spill).
template <int FMT>
__global__ void __launch_bounds__(kSThreads, 4) ln_stream_kernel(const __grid_constant__ QuantBatch batch) {
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  launch_dependents();
  grid_dependency_wait();  // inputs and outputs may belong to the previous kernel until here
  const QuantArgs& a = batch.t[0];
  const int nci = static_cast<int>(a.cols);
  const int cc = static_cast<int>(lane) * kLaneElems;
  const bool act = cc < nci;
  const bool aligned32 = (reinterpret_cast<uintptr_t>(a.src) & 31u) == 0u;
  const int64_t nw = static_cast<int64_t>(gridDim.x) * kSWarps;
  // this lane's 16 words (32 bf16) of row r (zeros past the row's end or past the last row)
  auto fetch = [&](uint32_t (&w)[16], int64_t r) {
    const int64_t off = r * a.cols + cc;
    if (act && r < a.rows && in_bounds(off >= 0 && off + 32 <= a.elems, batch.status)) {
      const uint8_t* src = a.src + off * 2;
      if (aligned32) {
        ld32(src, w);
        ld32(src + 32, w + 8);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) ld16(src + 16 * i, w + 4 * i);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = 0u;
    }
  };
  auto process = [&](const uint32_t (&w)[16], int64_t r) {
    float x[32];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    float mean, rstd;
    ln_row_stats(x, act, nci, a.eps, mean, rstd);
    if (act) ln_finish<FMT>(a, batch.status, static_cast<uint32_t>(r), cc, x, mean, rstd);
  };
  uint32_t w[16];
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kSWarps + warp; r < a.rows; r += nw) {
    fetch(w, r);
    process(w, r);
  }
  // padding of the tiled scales reads 0: every word of the padding rows of the last row tile (the
  // padding columns of each row's last group are zeroed by ln_finish)
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kSThreads + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * kSThreads;
  const int64_t pad_rows = (128 - a.rows % 128) % 128;
  for (int64_t wd = tid; wd < pad_rows * a.nct; wd += nthr) {
    const int64_t pr = a.rows + wd / a.nct, tc = wd % a.nct;
    const int64_t so = scale_word_offset(pr, 4 * tc, a.nct);
    if (in_bounds(so + 4 <= a.scales_bytes, batch.status)) *reinterpret_cast<uint32_t*>(a.scales + so) = 0u;
  }
}

// ---------------------------------------------------------------------------- LayerNorm kernel
// LayerNorm + MX quantization (MXFP8, MXFP4): the source is cut into chunks of whole rows (at
// most 16 KB), each brought into shared memory by one 1-D TMA bulk copy; a producer thread keeps a
// ring of kRing chunk buffers in flight and each consumer warp owns whole rows of a chunk, dealt
// round-robin over the CTA's chunks: the row's mean and rstd (fp32, two passes over the row -- in
// registers for rows of at most 1024 elements, else in shared memory -- with butterfly warp sums),
// then y = (x - mean) * rstd * gamma + beta and the quantization of the row, 32 columns per lane,
// with no barrier between the warps.
template <int FMT, bool F32>
__global__ void __launch_bounds__(QCfg::kThreads, QCfg::kCtasPerSm)
    layernorm_kernel(const __grid_constant__ QuantBatch batch) {
  constexpr int kThreads = QCfg::kThreads;
  constexpr int kRing = QCfg::kRing;
  constexpr int kConsumerWarps = QCfg::kConsumerWarps;
  constexpr int kEsize = F32 ? 4 : 2;
  extern __shared__ uint8_t q_smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(q_smem_raw) + 127) & ~uintptr_t(127));
  __shared__ uint64_t full_bar[kRing], empty_bar[kRing];
  __shared__ int abort_flag;
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const QuantArgs& a = batch.t[0];

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

  const int64_t nchunks = batch.chunk_start[1];
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t armed = 0;  // chunks loaded so far (ring order from stage 0)
      for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
        if (armed == batch.stall_after) break;  // injected stall: no more loads, none announced
        if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, &abort_flag, batch.status, batch.wait_ns)) break;
        const int64_t r0 = c * a.rows_per_chunk;
        const int64_t nr = min(a.rows_per_chunk, a.rows - r0);
        // a skipped (out-of-range) chunk still completes its stage, with no bytes
        const bool ok = in_bounds(r0 >= 0 && nr > 0 && nr * a.cols * kEsize <= kChunkMax && (r0 + nr) <= a.rows,
                                  batch.status);
        const uint32_t bytes = ok ? static_cast<uint32_t>(nr * a.cols * kEsize) : 0u;
        mbar_arrive_expect_tx(&full_bar[stage], bytes);
        if (ok) bulk_load(ring + stage * kChunkMax, a.src + r0 * a.cols * kEsize, bytes, &full_bar[stage]);
        ++armed;
        if (++stage == kRing) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // nothing this CTA loads may still be in flight when it exits
      wait_armed_stages(full_bar, kRing, armed, batch.status, batch.wait_ns);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const NvCtx nv;  // unused by the MX formats
    // rows are dealt round-robin over the concatenation of the CTA's chunks, so that a chunk whose
    // row count is not a multiple of the warp count does not give the same warps an extra row
    // every time; `lead`: this warp's first row in the current chunk
    uint32_t lead = warp - 1;
    int stage = 0;
    uint32_t phase = 0;
    const int nci = static_cast<int>(a.cols);
    const int pieces = nci * kEsize / 16;  // 16-byte pieces of a row
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
      if (!mbar_wait_bounded_warp(&full_bar[stage], phase, &abort_flag, batch.status, batch.wait_ns)) break;
      const int64_t r0 = c * a.rows_per_chunk;
      const int64_t nr = min(a.rows_per_chunk, a.rows - r0);
      const uint8_t* buf = ring + stage * kChunkMax;
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
        auto finish = [&](int cc, float (&x)[32], float mean, float rstd) {
          ln_finish<FMT>(a, batch.status, row, cc, x, mean, rstd);
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
          float mean, rstd;
          ln_row_stats(x, act, nci, a.eps, mean, rstd);
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
    }
  }

  // scale bytes of the padding rows of the last row tile read 0
  const int64_t pad_rows = (128 - a.rows % 128) % 128;
  const int64_t words = pad_rows * a.nct;
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; w < words;
       w += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int64_t r = a.rows + w / a.nct, tc = w % a.nct;
    const int64_t so = scale_word_offset(r, 4 * tc, a.nct);
    if (in_bounds(so + 4 <= a.scales_bytes, batch.status)) *reinterpret_cast<uint32_t*>(a.scales + so) = 0u;
  }
}

// Tensor amax (NVFP4 computed-scale mode) of every matrix of a list: max |x| over each tensor,
// NaN skipped like the block maxima -> atomicMax on the fp32 bits at its `out` (non-negative
// floats order like their bit patterns). The CTAs stride over each matrix in turn, so one launch
// serves a whole batch. Reads use the default cache policy so that the quantize pass that
// follows finds the most recently read lines in L2.
struct AmaxList {
  const uint4* src[kMaxBatch];
  int64_t nvec[kMaxBatch];  // 16-byte vectors of each source
  uint32_t* out[kMaxBatch];
  int n;
};

template <bool F32>
__global__ void __launch_bounds__(kAmaxThreads) amax_kernel(const __grid_constant__ AmaxList list) {
  constexpr int kU = 4;
  __shared__ float red[kAmaxThreads / 32];
  launch_dependents();
  grid_dependency_wait();  // the sources and the zeroed tails may belong to earlier work until here
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kAmaxThreads + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * kAmaxThreads;
  for (int t = 0; t < list.n; ++t) {
    const uint4* src = list.src[t];
    const int64_t nvec = list.nvec[t];
    float m = 0.0f;
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
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      float b = 0.0f;
      for (int i = 0; i < kAmaxThreads / 32; ++i) b = fmaxf(b, red[i]);
      if (b != 0.0f) atomicMax(list.out[t], __float_as_uint(b));
    }
    __syncthreads();  // red[] is reused by the next matrix
  }
}

// Launch with programmatic dependent launch where `pdl` is set: the kernel may then be launched
// while the previous kernel in the stream finishes; every kernel here waits for it
// (grid_dependency_wait) before touching memory, so the flag changes timing, not results.
template <typename... Args>
cudaError_t launch_pdl(void (*kernel)(Args...), int grid, int threads, int smem, cudaStream_t stream, bool pdl,
                       const Args&... args) {
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The streaming kernel takes programmatic dependent launch only right after the batch's own amax
// pass. After other kernels (a GEMM in a layer sequence) its early-launched CTAs measured slower on
// GB300: graph-replayed with the L2 flushed, the ViT-L MLP step at M = 51200 (MXFP4 + NVFP4) took
// 695.9 us with it on for every quantizer launch and 685.7 us with it off, the ViT-L MXFP8 layers
// at M = 7168 131.1 against 127.0 us; the NVFP4 ones at M = 7168 kept it after their amax pass
// (157.2 us with it off there too, against 154.5 us).
template <int FMT, bool F32, int NV>
cudaError_t launch_stream(const QuantBatch& b, int num_sms, cudaStream_t stream) {
  const int64_t ctas = ceil_div(b.chunk_start[b.n], kSWarps);
  const int grid =
      static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(ctas, SCfg<F32, NV != kMx>::kCtasPerSm * num_sms)));
  return launch_pdl(stream_kernel<FMT, F32, NV>, grid, kSThreads, 0, stream, NV == kNvComputed, b);
}

template <int FMT, bool F32>
cudaError_t launch_ln(const QuantBatch& b, int grid, cudaStream_t stream, int device) {
  static PerDevice<cudaError_t> setup;  // the shared-memory opt-in holds per device
  const cudaError_t attr = setup.run(device, [] {
    return cudaFuncSetAttribute(layernorm_kernel<FMT, F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, QCfg::kSmem);
  });
  if (attr != cudaSuccess) return attr;
  return launch_pdl(layernorm_kernel<FMT, F32>, grid, QCfg::kThreads, QCfg::kSmem, stream, true, b);
}

template <int FMT>
cudaError_t launch_ln_stream(const QuantBatch& b, int num_sms, cudaStream_t stream) {
  const int64_t ctas = ceil_div(b.t[0].rows, kSWarps);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(ctas, 4 * static_cast<int64_t>(num_sms))));
  return launch_pdl(ln_stream_kernel<FMT>, grid, kSThreads, 0, stream, true, b);
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

int launch_amax(const void* const* srcs, const int64_t* elems, uint32_t* const* outs, int n, bool src_f32,
                cudaStream_t stream, const DeviceInfo& dev) {
  if (n < 1 || n > kMaxBatch) return BSQ_ERR_ARG;
  AmaxList l{};
  l.n = n;
  int64_t most = 0;
  for (int i = 0; i < n; ++i) {
    l.src[i] = static_cast<const uint4*>(srcs[i]);
    l.nvec[i] = elems[i] * (src_f32 ? 4 : 2) / 16;
    l.out[i] = outs[i];
    most = std::max(most, l.nvec[i]);
  }
  const int agrid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(ceil_div(most, kAmaxThreads * 4), dev.num_sms * 8)));
  const cudaError_t e = src_f32 ? launch_pdl(amax_kernel<true>, agrid, kAmaxThreads, 0, stream, true, l)
                                : launch_pdl(amax_kernel<false>, agrid, kAmaxThreads, 0, stream, true, l);
  return e == cudaSuccess ? BSQ_OK : BSQ_ERR_LAUNCH;
}

// Per-matrix arguments of a batch.
void fill_args(QuantArgs& a, int fmt, const QuantItem& it) {
  a.src = static_cast<const uint8_t*>(it.src);
  a.rows = it.rows;
  a.cols = it.cols;
  a.elems = it.rows * it.cols;
  a.codes = static_cast<uint8_t*>(it.codes);
  a.scales = static_cast<uint8_t*>(it.scales);
  a.nsc = it.cols / block_size(fmt);
  a.nct = ceil_div(a.nsc, 4);
  a.cols_magic = static_cast<uint32_t>((uint64_t{1} << 32) / static_cast<uint64_t>(it.cols) + 1);
  a.cols_magic64 = ~uint64_t{0} / static_cast<uint64_t>(it.cols);
  a.codes_bytes = fmt == BSQ_MXFP8 ? a.elems : a.elems / 2;
  a.scales_bytes = scales_body_bytes(fmt, it.rows, it.cols);
  a.scale_words = fmt == BSQ_NVFP4 && it.cols % 64 == 0;
  if (fmt == BSQ_NVFP4) {
    a.tail = reinterpret_cast<uint32_t*>(a.scales + scales_body_bytes(fmt, it.rows, it.cols));
    a.g_in = it.global_scale;
    a.g_out = it.global_scale;
  }
}

int launch_quantize_batch(int fmt, bool src_f32, bool global_given, int count, const QuantItem* items,
                          cudaStream_t stream, const DeviceInfo& dev) {
  if (count < 1 || count > kMaxBatch) return BSQ_ERR_ARG;
  QuantBatch b{};
  b.n = count;
  b.status = dev.status;
  b.chunk_start[0] = 0;
  for (int i = 0; i < count; ++i) {  // warp steps of 1024 elements, concatenated
    fill_args(b.t[i], fmt, items[i]);
    b.chunk_start[i + 1] = b.chunk_start[i] + ceil_div(b.t[i].elems, 32 * kLaneElems);
  }

  cudaError_t err = cudaSuccess;
  if (fmt == BSQ_NVFP4) {
    const void* srcs[kMaxBatch];
    int64_t elems[kMaxBatch];
    uint32_t* outs[kMaxBatch];
    for (int i = 0; i < count; ++i) {
      const QuantArgs& a = b.t[i];
      if (cudaMemsetAsync(a.tail, 0, 16, stream) != cudaSuccess) return BSQ_ERR_LAUNCH;
      srcs[i] = a.src;
      elems[i] = a.elems;
      outs[i] = a.tail + 1;
    }
    // one amax launch for the whole batch
    if (!global_given && launch_amax(srcs, elems, outs, count, src_f32, stream, dev) != BSQ_OK) return BSQ_ERR_LAUNCH;
    if (!global_given) {
      err = src_f32 ? launch_stream<BSQ_NVFP4, true, kNvComputed>(b, dev.num_sms, stream)
                    : launch_stream<BSQ_NVFP4, false, kNvComputed>(b, dev.num_sms, stream);
    } else {
      err = src_f32 ? launch_stream<BSQ_NVFP4, true, kNvGiven>(b, dev.num_sms, stream)
                    : launch_stream<BSQ_NVFP4, false, kNvGiven>(b, dev.num_sms, stream);
    }
  } else if (fmt == BSQ_MXFP8) {
    err = src_f32 ? launch_stream<BSQ_MXFP8, true, kMx>(b, dev.num_sms, stream)
                  : launch_stream<BSQ_MXFP8, false, kMx>(b, dev.num_sms, stream);
  } else {
    err = src_f32 ? launch_stream<BSQ_MXFP4, true, kMx>(b, dev.num_sms, stream)
                  : launch_stream<BSQ_MXFP4, false, kMx>(b, dev.num_sms, stream);
  }
  return err == cudaSuccess ? BSQ_OK : BSQ_ERR_LAUNCH;
}

int launch_layernorm_quantize(int fmt, bool src_f32, const QuantItem& item, const uint16_t* gamma,
                              const uint16_t* beta, float eps, cudaStream_t stream, const DeviceInfo& dev) {
  const int64_t esize = src_f32 ? 4 : 2;
  const int64_t row_bytes = item.cols * esize;
  if (row_bytes > kChunkMax) return BSQ_ERR_SHAPE;  // whole rows only
  QuantBatch b{};
  b.n = 1;
  b.status = dev.status;
  QuantArgs& a = b.t[0];
  fill_args(a, fmt, item);
  a.gamma = gamma;
  a.beta = beta;
  a.eps = eps;
  if (!src_f32 && item.cols <= 32 * kLaneElems) {
    // bf16 rows of at most 1024 elements: the streaming kernel (it waits on no barrier, so an
    // injected stall has nothing to act on and stays armed for the shared-memory kernel)
    const cudaError_t err = fmt == BSQ_MXFP8 ? launch_ln_stream<BSQ_MXFP8>(b, dev.num_sms, stream)
                                             : launch_ln_stream<BSQ_MXFP4>(b, dev.num_sms, stream);
    return err == cudaSuccess ? BSQ_OK : BSQ_ERR_LAUNCH;
  }
  const StallInjection inj = take_stall(BSQ_KERNEL_LAYERNORM);
  b.stall_after = inj.after;
  b.wait_ns = inj.limit_ns;
  // chunks of whole rows: at most one ring buffer, and small enough that every SM gets a few
  const int64_t target = std::max<int64_t>(
      kChunkMin, std::min<int64_t>(kChunkMax, a.elems * esize / (4 * QCfg::kCtasPerSm * static_cast<int64_t>(dev.num_sms))));
  a.rows_per_chunk = std::max<int64_t>(1, std::min<int64_t>(target / row_bytes, kLnMaxRows));
  b.chunk_start[0] = 0;
  b.chunk_start[1] = ceil_div(a.rows, a.rows_per_chunk);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(b.chunk_start[1], QCfg::kCtasPerSm * dev.num_sms)));
  cudaError_t err;
  if (fmt == BSQ_MXFP8) {
    err = src_f32 ? launch_ln<BSQ_MXFP8, true>(b, grid, stream, dev.device) : launch_ln<BSQ_MXFP8, false>(b, grid, stream, dev.device);
  } else {
    err = src_f32 ? launch_ln<BSQ_MXFP4, true>(b, grid, stream, dev.device) : launch_ln<BSQ_MXFP4, false>(b, grid, stream, dev.device);
  }
  return err == cudaSuccess ? BSQ_OK : BSQ_ERR_LAUNCH;
}

}  // namespace bsq
