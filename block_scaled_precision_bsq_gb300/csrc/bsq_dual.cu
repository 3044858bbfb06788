// bsq_dual.cu -- dual-layout MX quantization for the backward GEMMs: one R x C bf16 / fp32
// matrix gives both its row-wise operand (quantized along C, R x C) and its column-wise one
// (quantized along R, stored transposed as C x R), each with codes and tiled scales, in one pass
// over the source. With stochastic rounding the element rounding is the gradient form: the
// magnitude steps up from the grid point below iff frac(|v| / spacing) > u, u = h 2^-16 with h
// 16 bits of Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as
// 1, 2, 3", SC'11) keyed by the seed, one call per 8 elements counting over the element's index
// in its layout.
//
// Why dual: dgrad (dX = dY W) contracts over N and wgrad (dW = dY^T X) over M, so the backward
// pass needs dY quantized along both of its dimensions, W along N and X along M ("lightly-train
// - DINOv3 + EoMT on RTX 5090" README, section 4.3, the quantized training stack). Reading the
// source once and writing both layouts costs 2 + 2 bytes per bf16 element (MXFP8) against 2 x
// (2 + 1) for two quantizer calls over the source and its transpose.
//
// Work mapping (two CTAs per SM, persistent over tiles). A tile is 128 columns x kRows rows
// (128 for bf16, 64 for fp32: 32 KB), loaded by one 2-D TMA copy into a 3-deep ring; tiles past
// the matrix edge read zeros. Every tile covers exactly one 512-byte scale tile of the row
// layout and one (bf16) or half of one (fp32) of the column layout, so the kernel writes every
// scale byte, padding included (zero blocks give scale byte 0), and no buffer needs clearing.
//   row pass     each lane takes 32 consecutive elements of a row -- one MX block, two NVFP4
//                blocks -- so block maxima need no shuffle; four lanes cover a 128-column row,
//                whose scale bytes are OR-ed into 32-bit words of the tiled layout by one or
//                two shuffles. (With 16-byte pieces per lane and shuffles for the maxima the
//                pass took ~12.6 instructions per element.)
//   column pass  each thread takes one column and 64 / 32 rows of the tile: the warp reads 32
//                consecutive columns of one row per load (conflict-free), the thread reduces
//                its 32-row blocks alone and puts each block's codes into a shared-memory
//                staging tile laid out as the transposed operand's 128 rows (one per source
//                column), swizzled so that 8 lanes on 8 rows hit 8 different bank groups; one
//                2-D TMA store per tile then writes the staging tile as whole lines. Direct
//                stores from this layout touch 32 lines per warp instruction and were the
//                kernel's top stall (measured on GB300).
// The staging tile is reused once the previous tile's store has read it (bulk wait_group.read
// by the issuing thread before a named barrier of the consumer warps); that barrier also
// reduces the consumers' full-barrier outcomes, so a timeout sends every consumer warp out of
// the loop together.
//
// Stochastic rounding runs on the fp32 bits of v (exact): for a normal target binade it adds
// the complement of the random bits, aligned below the kept mantissa, and truncates, which
// rounds up exactly when frac(q) > u; a target in the element format's subnormal range takes
// the fixed-point form (ceil(q 2^16) + 2^16 - 1 - h) >> 16.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "bsq_device.cuh"
#include "bsq_internal.h"

namespace bsq {
namespace {

constexpr int kDCols = 128;          // tile columns
constexpr int kDTileBytes = 32768;   // one tile of source
constexpr int kDStages = 3;
constexpr int kDConsumerWarps = 8;   // warps 1..8; warp 0 lane 0 is the TMA producer
constexpr int kDThreads = 32 * (kDConsumerWarps + 1);
constexpr int kDCtasPerSm = 2;
constexpr int kDStageBytes = 16384;  // transposed codes of one tile (at most 128 x 128 bytes)
// dynamic shared memory: staging tile (1024-byte aligned for the swizzled TMA store), input
// ring, barriers; nothing static, so that two CTAs fit on an SM
constexpr int kDRingOff = kDStageBytes;
constexpr int kDBarOff = kDRingOff + kDStages * kDTileBytes;
constexpr int kDTabOff = kDBarOff + 128;  // NVFP4: reciprocals of the 128 block divisors
constexpr int kDSmem = kDTabOff + 512;
static_assert(kDCtasPerSm * (kDSmem + 1024) <= 233472, "two CTAs per SM, each with 1 KB reserved");

struct DualArgs {
  int64_t rows, cols;  // R, C
  uint8_t* row_codes;
  uint8_t* row_scales;
  uint8_t* col_codes;
  uint8_t* col_scales;
  int64_t tiles_c;  // 128-column tiles
  int64_t ntiles;
  int64_t nct_row;  // 512-byte scale tiles per 128-row group, row layout: ceil(C / (4 * block))
  int64_t nct_col;  // same for the column layout (C rows, R / block scale columns): ceil(R / (4 * block))
  uint32_t seed_lo, seed_hi;
  // Philox round keys, computed on the host: keys[2i] = seed_lo + i * 0x9E3779B9, keys[2i + 1] =
  // seed_hi + i * 0xBB67AE85 (kernel parameters, so every round XORs a constant-bank operand)
  uint32_t keys[20];
  // NVFP4: the per-tensor scale g, shared by both layouts; {g, amax} tails after each scale body
  uint32_t* row_tail;
  uint32_t* col_tail;
  const float* g_in;  // given mode (else g = amax / 2688 from row_tail[1], put there beforehand)
  float* g_out;       // computed mode: receives g (nullable)
  int* status;
  int64_t stall_after;  // injected stall (tests): the producer stops after this many tiles; -1 = none
  uint64_t wait_ns;     // limit of every bounded wait
  int64_t codes_bytes;  // size of each layout's code buffer (index checks)
  int64_t row_scales_bytes, col_scales_bytes;  // tiled scale bodies of the two layouts
};

// Philox4x32-10 of the SC'11 paper: ten rounds of two 32 x 32 -> 64-bit products mixed into
// the other two counter words and the round key (the key bumped by the Weyl constants after every
// round: the caller's precomputed keys[2i], keys[2i + 1]).
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               const uint32_t* keys) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c0;  // one widening multiply each
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c2;
    c0 = static_cast<uint32_t>(p1 >> 32) ^ c1 ^ keys[2 * i];
    c1 = static_cast<uint32_t>(p1);
    c2 = static_cast<uint32_t>(p0 >> 32) ^ c3 ^ keys[2 * i + 1];
    c3 = static_cast<uint32_t>(p0);
  }
  return make_uint4(c0, c1, c2, c3);
}

// The random bits h (u = h 2^-16) of elements 8g .. 8g+7 of a layout (0 = row, 1 = column):
// element 8g + j takes the 16-bit half j mod 2 (low first) of Philox word j / 2 at counter g;
// lo holds elements 8g .. 8g+3, hi elements 8g+4 .. 8g+7.
__device__ __forceinline__ void sr_words8(uint64_t g, uint32_t layout, const DualArgs& a, uint4& lo, uint4& hi) {
  const uint4 w = philox4x32_10(static_cast<uint32_t>(g), static_cast<uint32_t>(g >> 32), layout, 0u, a.keys);
  lo = make_uint4(w.x & 0xFFFFu, w.x >> 16, w.y & 0xFFFFu, w.y >> 16);
  hi = make_uint4(w.z & 0xFFFFu, w.z >> 16, w.w & 0xFFFFu, w.w >> 16);
}

// Block scale byte of the MX rule: floor(log2(amax)) - emax, clamped at -127, plus 127.
template <int FMT>
__device__ __forceinline__ uint32_t mx_scale_byte(float amax) {
  constexpr uint32_t kEmax = (FMT == BSQ_MXFP8) ? 8u : 2u;
  const uint32_t ef = __float_as_uint(amax) >> 23;
  return ef > kEmax ? ef - kEmax : 0u;
}

// 2^(127 - sbyte) = 1 / scale, exact.
__device__ __forceinline__ float mx_inv_scale(uint32_t sbyte) { return __uint_as_float((254u - sbyte) << 23); }

// Stochastic rounding of y = x / scale (exact in fp32 unless it fell below fp32's range) to an
// E4M3 (MXFP8) or e2m1 code with the element's 16 random bits h: q = |y| / spacing at y's
// binade (the subnormal spacing below the smallest normal), magnitude floor(q) + (frac(q) > u)
// with u = h 2^-16, saturating at the largest finite value. Exact.
template <int FMT>
__device__ __forceinline__ uint32_t sr_code(float y, float x, uint32_t h) {
  constexpr uint32_t kM = (FMT == BSQ_MXFP8) ? 3u : 1u;         // mantissa bits
  constexpr uint32_t D = 23u - kM;                              // fp32 mantissa bits below the kept ones
  constexpr uint32_t kEminB = (FMT == BSQ_MXFP8) ? 121u : 127u;  // biased exponent of the lowest normal binade
  constexpr uint32_t kMaxCode = (FMT == BSQ_MXFP8) ? 0x7Eu : 0x7u;
  constexpr uint32_t kSign = (FMT == BSQ_MXFP8) ? 7u : 3u;
  const uint32_t yb = __float_as_uint(y);
  const uint32_t b = yb & 0x7FFFFFFFu;
  uint32_t mag;
  // normal target binade: q's fraction is the low D mantissa bits t, and u in units of 2^-D is
  // h 2^(D - 16): up iff t > h 2^(D - 16), i.e. iff t + (2^D - 1 - h 2^(D - 16)) carries into the
  // kept bits; the carry may move to the next binade, which is the next grid point. The exponent
  // re-bias folds into the same add.
  auto normal_mag = [&]() { return (b + ((1u << D) - 1u - ((kEminB - 1u) << 23)) - (h << (D - 16u))) >> D; };
  // subnormal target: q = |y| / 2^-S (S = 9 for E4M3, 1 for e2m1) < 2^kM, and frac(q) > u iff
  // ceil(frac(q) 2^16) > h, so floor(q) + (frac(q) > u) =
  // (ceil(q 2^16) + 2^16 - 1 - h) >> 16. ceil(|y| 2^(S + 16)) is a round-up add of 2^23 to the
  // exact product (below 2^(kM + 16), fp32 denormals included), read off the sum's bits. A y
  // that underflowed to 0 from x != 0 is a positive value below every step: ceiling 1.
  auto subnormal_mag = [&]() {
    constexpr float kScale = (FMT == BSQ_MXFP8) ? 33554432.0f : 131072.0f;  // 2^25, 2^17
    uint32_t c = __float_as_uint(__fadd_ru(__fmul_rn(__uint_as_float(b), kScale), 8388608.0f)) - 0x4B000000u;
    // (NVFP4 passes the quotient itself as x, so there b == 0 implies x == 0)
    if constexpr (FMT != BSQ_NVFP4) {
      if (b == 0u && x != 0.0f) c = 1u;
    }
    return (c + 0xFFFFu - h) >> 16;
  };
  if constexpr (FMT == BSQ_MXFP8) {
    // E4M3: values in the subnormal range are rare (a block's maximum sits 2^14 above it), so the
    // branch is almost always warp-uniform
    if (b < (kEminB << 23)) mag = subnormal_mag();
    else mag = normal_mag();
  } else {
    // e2m1: |v| < 1 (the format's subnormal range) is common, so both forms are computed and
    // selected instead of diverging
    const uint32_t mn = normal_mag(), ms = subnormal_mag();
    mag = b >= (kEminB << 23) ? mn : ms;
  }
  // from the largest finite value up the magnitude is at least kMaxCode; below it, at most
  mag = min(mag, kMaxCode);
  return ((yb >> 31) << kSign) | mag;
}

// The value a code encodes, x / scale: MX x * (1 / scale) (exact), NVFP4 fp32(x / fp32(s g)), the
// IEEE quotient -- by markstein_quotient with the block's reciprocal r where that is valid for the
// whole block (kQuick), else by division.
template <int FMT, bool kQuick>
__device__ __forceinline__ float scaled(float x, float f, float r) {
  if constexpr (FMT == BSQ_NVFP4) return kQuick ? markstein_quotient(x, f, r) : __fdiv_rn(x, f);
  else return x * f;
}

// Round-to-nearest-even codes of n (a multiple of 4, at most 8 for e2m1) consecutive elements
// x[0..n) with the block factor f, packed: E4M3 one byte each (element i in byte i % 4 of
// w[i / 4]), e2m1 one nibble each (element i in bits 4i of w[0]).
template <int FMT, int N, bool kQuick>
__device__ __forceinline__ void rne_codes(const float* x, float f, float r, uint32_t* w) {
  if constexpr (FMT == BSQ_MXFP8) {
#pragma unroll
    for (int j = 0; j < N / 4; ++j)
      w[j] = cvt_e4m3x4(x[4 * j] * f, x[4 * j + 1] * f, x[4 * j + 2] * f, x[4 * j + 3] * f);
  } else if constexpr (N == 8 && FMT == BSQ_NVFP4 && kQuick) {
    // markstein_quotient on packed pairs with the reciprocal negated: q0' = x (-r) = -q0,
    // t = q0' f + x (the exact remainder x - q0 f), y = t (-r) + q0' = -(q0 + t r), the negated
    // IEEE quotient; one XOR per eight codes flips the signs back, signed zeros included
    const uint64_t f2v = f2_splat(f), nr2 = f2_splat(-r);
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      const uint64_t x2 = f2(x[i], x[i + 1]);
      const uint64_t q0 = f2_mul(x2, nr2);
      f2_split(f2_fma(f2_fma(q0, f2v, x2), nr2, q0), y[i], y[i + 1]);
    }
    w[0] = cvt_e2m1x8(y) ^ 0x88888888u;
  } else if constexpr (N == 8) {
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = scaled<FMT, kQuick>(x[i], f, r);
    w[0] = cvt_e2m1x8(y);
  } else {
    w[0] = cvt_e2m1x2(scaled<FMT, kQuick>(x[0], f, r), scaled<FMT, kQuick>(x[1], f, r)) |
           (cvt_e2m1x2(scaled<FMT, kQuick>(x[2], f, r), scaled<FMT, kQuick>(x[3], f, r)) << 8);
  }
}

// Stochastic codes of the four elements x[0..4) with the block factor f and the random bits q
// (element i takes q's component i, 16 bits), packed as rne_codes packs four: E4M3 one word,
// e2m1 the low 16 bits.
// MX passes x for sr_code's underflow test (the MX value x / scale is exact unless it leaves
// fp32's range); NVFP4 rounds the fp32 quotient itself, so the quotient stands in for x.
// E4M3 tests the range once per four elements: when all four scaled values lie in the normal
// range (all but ~1 % of groups: the subnormal range sits 2^14 below a block's maximum), each
// code is sr_code's normal-range carry form without a branch per element; otherwise sr_code.
template <int FMT, bool kQuick>
__device__ __forceinline__ uint32_t sr_codes4(const float* x, float f, float r, uint4 q) {
  constexpr int kBits = (FMT == BSQ_MXFP8) ? 8 : 4;
  const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
  uint32_t w = 0;
  if constexpr (FMT == BSQ_MXFP8) {
    float y[4];
    uint32_t bmin = 0xFFFFFFFFu;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      y[i] = scaled<FMT, kQuick>(x[i], f, r);
      bmin = min(bmin, __float_as_uint(y[i]) & 0x7FFFFFFFu);
    }
    if (bmin >= (121u << 23)) {  // 2^-6, the smallest normal E4M3 magnitude
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t yb = __float_as_uint(y[i]);
        const uint32_t b = yb & 0x7FFFFFFFu;
        const uint32_t mag = min((b + ((1u << 20) - 1u - (120u << 23)) - (qq[i] << 4)) >> 20, 0x7Eu);
        w |= (((yb >> 31) << 7) | mag) << (8 * i);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) w |= sr_code<FMT>(y[i], x[i], qq[i]) << (8 * i);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float y = scaled<FMT, kQuick>(x[i], f, r);
      w |= sr_code<FMT>(y, FMT == BSQ_NVFP4 ? y : x[i], qq[i]) << (kBits * i);
    }
  }
  return w;
}

// Codes of a zero NVFP4 block scale: zeros carrying the sign of each element (n <= 8).
template <int N>
__device__ __forceinline__ uint32_t sign_codes(const float* x) {
  uint32_t w = 0;
#pragma unroll
  for (int i = 0; i < N; ++i) w |= (__float_as_uint(x[i]) >> 31) << (4 * i + 3);
  return w;
}

// Codes of one block of BS elements xb (MX 32, NVFP4 16) with the block factor f (and NVFP4's
// reciprocal r), packed into wb as rne_codes / sr_codes4 pack them: round to nearest even, or
// stochastic with the random words of element group g0 (8 elements per group) in `layout`.
template <int FMT, bool SR, bool kQuick>
__device__ __forceinline__ void block_codes(const float* xb, float f, float r, uint64_t g0, uint32_t layout,
                                            const DualArgs& a, uint32_t* wb) {
  constexpr bool kFp8 = (FMT == BSQ_MXFP8);
  constexpr int BS = (FMT == BSQ_NVFP4) ? 16 : 32;
  if constexpr (SR) {
#pragma unroll
    for (int go = 0; go < BS / 8; ++go) {
      uint4 rlo, rhi;
      sr_words8(g0 + go, layout, a, rlo, rhi);
      const uint32_t v0 = sr_codes4<FMT, kQuick>(xb + 8 * go, f, r, rlo);
      const uint32_t v1 = sr_codes4<FMT, kQuick>(xb + 8 * go + 4, f, r, rhi);
      if constexpr (kFp8) {
        wb[2 * go] = v0;
        wb[2 * go + 1] = v1;
      } else {
        wb[go] = v0 | (v1 << 16);
      }
    }
  } else {
    constexpr int kWords = BS * (kFp8 ? 8 : 4) / 32;
#pragma unroll
    for (int j = 0; j < kWords; ++j) rne_codes<FMT, kFp8 ? 4 : 8, kQuick>(xb + (kFp8 ? 4 : 8) * j, f, r, wb + j);
  }
}

// NVFP4 divisors of the tensor: g, 6 g, its reciprocal (NaN where markstein_quotient is not valid
// for 6 g) and the reciprocal of fp32(s g) for every E4M3 scale code s (NaN for s = 0 and where the
// quotient step is not valid for that divisor), in shared memory.
struct NvScales {
  float g, six_g, r6;
  const float* rtab;
};

// Block scale from the block maximum: MX the UE8M0 byte and 1 / scale; NVFP4 the E4M3 code of
// fp32(amax / fp32(6 g)) and fp32(s g) (0 when s is 0: the block's codes are signed zeros), with r
// the reciprocal of fp32(s g) and `quick` true when markstein_quotient gives every element's IEEE
// quotient (scaled<FMT, true>).
template <int FMT>
__device__ __forceinline__ uint32_t block_scale(float amax, const NvScales& nv, float& f, float& r, bool& quick) {
  if constexpr (FMT == BSQ_NVFP4) {
    uint32_t sc = 0;
    if (nv.g != 0.0f) {
      float qs;
      if (__fmul_rn(amax, nv.r6) < 0x1p100f) qs = markstein_quotient(amax, nv.six_g, nv.r6);
      else qs = __fdiv_rn(amax, nv.six_g);
      sc = cvt_e4m3x2(qs, 0.0f) & 0xFFu;
    }
    f = __fmul_rn(e4m3_to_f32(sc), nv.g);
    r = nv.rtab[sc];
    quick = __fmul_rn(amax, r) < 0x1p100f;
    return sc;
  } else {
    const uint32_t sb = mx_scale_byte<FMT>(amax);
    f = mx_inv_scale(sb);
    r = 0.0f;
    quick = true;
    return sb;
  }
}

// Named barriers of the consumer warps (ids 1 and 2; 0 is __syncthreads).
__device__ __forceinline__ bool consumers_and_sync(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(p)), "n"(32 * kDConsumerWarps)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(32 * kDConsumerWarps) : "memory");
}

// Byte offset in the staging tile of logical byte `b` of row `row` (rows of S bytes), with the
// TMA swizzle of an S-byte box row: 16-byte chunk bits [4, 4 + log2(S / 16)) XOR-ed with the
// address bits from 7 up (the staging tile is 1024-byte aligned).
template <int S>
__device__ __forceinline__ uint32_t staging_offset(uint32_t row, uint32_t b) {
  constexpr uint32_t kMask = S / 16 - 1;  // 7 (128 B), 3 (64 B), 1 (32 B)
  const uint32_t off = row * S + b;
  return off ^ (((off >> 7) & kMask) << 4);
}

template <int FMT, bool F32, bool SR>
__global__ void __launch_bounds__(kDThreads, kDCtasPerSm)
    dual_kernel(const __grid_constant__ CUtensorMap src_map, const __grid_constant__ CUtensorMap col_map,
                const DualArgs a) {
  constexpr bool kNv = (FMT == BSQ_NVFP4);
  constexpr bool kFp8 = (FMT == BSQ_MXFP8);
  constexpr int BS = kNv ? 16 : 32;                        // block size
  constexpr int kEsize = F32 ? 4 : 2;
  constexpr int kRows = kDTileBytes / (kDCols * kEsize);  // 128 bf16, 64 fp32
  constexpr int kRowSteps = kRows / 8 / kDConsumerWarps;  // row-pass steps per warp (8 rows each)
  constexpr int kColUnits = kRows / 32 / 2;  // column-pass 32-row units per thread (2 bf16, 1 fp32)
  constexpr int kUnitScales = 32 / BS;       // scale bytes of a 32-row unit
  constexpr int kUnitCodeBytes = kFp8 ? 32 : 16;           // codes of a 32-element unit
  constexpr int S = kRows * kUnitCodeBytes / 32;           // staging row: the tile's rows of one column
  extern __shared__ __align__(1024) uint8_t d_smem[];
  uint8_t* staging = d_smem;
  uint8_t* ring = d_smem + kDRingOff;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(d_smem + kDBarOff);
  uint64_t* empty_bar = full_bar + kDStages;
  int* abort_flag = reinterpret_cast<int*>(empty_bar + kDStages);
  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;

  // the swizzled staging tile needs a 1024-byte aligned address (uniform: every thread leaves)
  if (smem_u32(d_smem) & 1023u) {
    if (threadIdx.x == 0) atomicCAS(a.status, 0, BSQ_ERR_LAUNCH);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kDStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kDConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  launch_dependents();
  grid_dependency_wait();  // the source and outputs may belong to the previous kernel until here

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&src_map);
      int stage = 0;
      uint32_t phase = 0;
      int64_t armed = 0;  // tiles loaded so far (ring order from stage 0)
      for (int64_t t = blockIdx.x; t < a.ntiles; t += gridDim.x) {
        if (armed == a.stall_after) break;  // injected stall: no more loads, none announced
        if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, a.status, a.wait_ns)) break;
        const int64_t ti = t / a.tiles_c, tj = t - ti * a.tiles_c;
        mbar_arrive_expect_tx(&full_bar[stage], kDTileBytes);
        tma_load_2d(ring + stage * kDTileBytes, &src_map, &full_bar[stage], static_cast<int32_t>(tj * kDCols),
                    static_cast<int32_t>(ti * kRows));
        ++armed;
        if (++stage == kDStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // nothing this CTA loads may still be in flight when it exits
      wait_armed_stages(full_bar, kDStages, armed, a.status, a.wait_ns);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cw = static_cast<int>(warp) - 1;
  const int ct = static_cast<int>(threadIdx.x) - 32;  // 0 .. 255
  const bool issuer = ct == 0;                         // issues the staging tile's TMA stores
  if (issuer) prefetch_tmap(&col_map);
  const int64_t R = a.rows, C = a.cols;
  // NVFP4 per-tensor scale (both layouts): given, or amax / 2688 with amax in the row tail
  float* nv_rtab = reinterpret_cast<float*>(d_smem + kDTabOff);
  NvScales nv{0.0f, 0.0f, 0.0f, nv_rtab};
  if constexpr (kNv) {
    const float g = a.g_in != nullptr ? *a.g_in : __fdiv_rn(__uint_as_float(a.row_tail[1]), 2688.0f);
    nv.g = g;
    nv.six_g = __fmul_rn(6.0f, g);
    const float r6 = __frcp_rn(nv.six_g);
    nv.r6 = markstein_ok(nv.six_g, r6, 0.0f) ? r6 : __uint_as_float(0x7FC00000u);
    if (ct < 128) {  // the block divisors' reciprocals, one scale code per thread
      const float d = __fmul_rn(e4m3_to_f32(static_cast<uint32_t>(ct)), g);
      const float r = __frcp_rn(d);
      nv_rtab[ct] = (ct != 0 && markstein_ok(d, r, 0.0f)) ? r : __uint_as_float(0x7FC00000u);
    }
    consumers_sync();
    if (blockIdx.x == 0 && ct == 0) {
      a.row_tail[0] = __float_as_uint(g);
      a.col_tail[0] = __float_as_uint(g);
      if (a.g_in == nullptr) {
        a.col_tail[1] = a.row_tail[1];
        if (a.g_out != nullptr) *a.g_out = g;
      }
    }
  }
  uint32_t run_max = 0;  // NVFP4 given mode: this thread's largest |x| (fp32 bits) for the tails
  bool stored = false;
  int stage = 0;
  uint32_t phase = 0;
  for (int64_t t = blockIdx.x; t < a.ntiles; t += gridDim.x) {
    const bool ok = mbar_wait_bounded_warp(&full_bar[stage], phase, abort_flag, a.status, a.wait_ns);
    const int64_t ti = t / a.tiles_c, tj = t - ti * a.tiles_c;
    const int64_t r0 = ti * kRows, c0 = tj * kDCols;
    const uint8_t* tile = ring + stage * kDTileBytes;

    // ---- row pass: each lane one 32-element piece of a row (one MX block, two NVFP4 blocks),
    // four lanes per 128-column row, 8 rows per warp step
    if (ok) {
#pragma unroll 1
      for (int s = 0; s < kRowSteps; ++s) {
        const int rr = (s * kDConsumerWarps + cw) * 8 + static_cast<int>(lane >> 2);
        const int cc = static_cast<int>(lane & 3u) * 32;
        float x[32];
        const uint4* src = reinterpret_cast<const uint4*>(tile + (rr * kDCols + cc) * kEsize);
        if constexpr (F32) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 v = src[i];
            x[4 * i] = __uint_as_float(v.x);
            x[4 * i + 1] = __uint_as_float(v.y);
            x[4 * i + 2] = __uint_as_float(v.z);
            x[4 * i + 3] = __uint_as_float(v.w);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 v = src[i];
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              x[8 * i + 2 * k] = __uint_as_float(wv[k] << 16);
              x[8 * i + 2 * k + 1] = __uint_as_float(wv[k] & 0xFFFF0000u);
            }
          }
        }
        const int64_t r = r0 + rr, c = c0 + cc;
        constexpr int kBlocks = 32 / BS;               // 1 (MX) or 2 (NVFP4)
        constexpr int kWords = kFp8 ? 8 : 4;           // code words of the piece
        constexpr int kBlockWords = kWords / kBlocks;  // code words of one block
        uint32_t w[kWords];
        uint32_t sbytes = 0;
        const uint64_t g0 = (static_cast<uint64_t>(r) * static_cast<uint64_t>(C) + static_cast<uint64_t>(c)) >> 3;
#pragma unroll
        for (int h = 0; h < kBlocks; ++h) {
          const float* xb = x + h * BS;
          float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int k = 0; k < BS; ++k) m[k & 3] = fmaxf(m[k & 3], fabsf(xb[k]));
          const float amax = fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
          if constexpr (kNv) run_max = max(run_max, __float_as_uint(amax));
          float bf, br;
          bool quick;
          sbytes |= block_scale<FMT>(amax, nv, bf, br, quick) << (8 * h);
          uint32_t* wb = w + h * kBlockWords;
          if (kNv && bf == 0.0f) {
            wb[0] = sign_codes<8>(xb);
            wb[1] = sign_codes<8>(xb + 8);
          } else if (!kNv || quick) {
            block_codes<FMT, SR, true>(xb, bf, br, g0 + h * (BS / 8), 0u, a, wb);
          } else {
            block_codes<FMT, SR, false>(xb, bf, br, g0 + h * (BS / 8), 0u, a, wb);
          }
        }
        if (r < R && c < C &&
            in_bounds((kFp8 ? r * C + c + 32 : (r * C + c) / 2 + 16) <= a.codes_bytes, a.status)) {
          const int64_t idx = r * C + c;
          if constexpr (kFp8) {
            uint4* dst = reinterpret_cast<uint4*>(a.row_codes + idx);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          } else {
            *reinterpret_cast<uint4*>(a.row_codes + idx / 2) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        // the row's scale bytes -> 32-bit words of the tiled layout: MX one word (lane b of the
        // row holds byte b), NVFP4 two words (lanes 2k and 2k + 1 hold word k)
        uint32_t sw;
        if constexpr (kNv) {
          sw = sbytes << (16 * (lane & 1u));
          sw |= __shfl_xor_sync(0xFFFFFFFFu, sw, 1);
        } else {
          sw = sbytes << (8 * (lane & 3u));
          sw |= __shfl_xor_sync(0xFFFFFFFFu, sw, 1);
          sw |= __shfl_xor_sync(0xFFFFFFFFu, sw, 2);
        }
        const int64_t grp = c / (4 * BS);  // 4-scale-column group of the row layout
        if ((lane & (kNv ? 1u : 3u)) == 0 && grp < a.nct_row) {
          const int64_t off = ((r >> 7) * a.nct_row + grp) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
          if (in_bounds(off + 4 <= a.row_scales_bytes, a.status)) *reinterpret_cast<uint32_t*>(a.row_scales + off) = sw;
        }
      }
    }

    // the previous tile's store has read the staging tile; every consumer saw its full barrier
    if (issuer && stored) bulk_wait_group_read<0>();
    if (!consumers_and_sync(ok)) break;

    // ---- column pass: one column, kColUnits units of 32 rows per thread
    {
      const int cc = ct & (kDCols - 1);
      const int gh = ct >> 7;
      const int64_t c = c0 + cc;
      uint32_t sbytes = 0;
#pragma unroll 1
      for (int bb = 0; bb < kColUnits; ++bb) {
        const int rb = (gh * kColUnits + bb) * 32;
        float x[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          if constexpr (F32) {
            x[k] = *reinterpret_cast<const float*>(tile + ((rb + k) * kDCols + cc) * 4);
          } else {
            x[k] = __uint_as_float(
                static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(tile + ((rb + k) * kDCols + cc) * 2)) << 16);
          }
        }
        uint32_t w[kFp8 ? 8 : 4];
        const uint64_t g0 = (static_cast<uint64_t>(c) * static_cast<uint64_t>(R) + static_cast<uint64_t>(r0 + rb)) >> 3;
#pragma unroll
        for (int h = 0; h < kUnitScales; ++h) {  // the unit's blocks: 1 (MX) or 2 (NVFP4) of BS rows
          const float* xb = x + h * BS;
          float m[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            m[i] = 0.0f;
#pragma unroll
            for (int k = i; k < BS; k += 4) m[i] = fmaxf(m[i], fabsf(xb[k]));
          }
          const float amax = fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
          float bf, br;
          bool quick;
          const uint32_t sbyte = block_scale<FMT>(amax, nv, bf, br, quick);
          sbytes |= sbyte << (8 * (bb * kUnitScales + h));
          constexpr int kWords = BS * (kFp8 ? 8 : 4) / 32;  // code words of one block
          uint32_t* wb = w + h * kWords;
          if (kNv && bf == 0.0f) {
            wb[0] = sign_codes<8>(xb);
            wb[1] = sign_codes<8>(xb + 8);
          } else if (!kNv || quick) {
            block_codes<FMT, SR, true>(xb, bf, br, g0 + h * (BS / 8), 1u, a, wb);
          } else {
            block_codes<FMT, SR, false>(xb, bf, br, g0 + h * (BS / 8), 1u, a, wb);
          }
        }
        // codes -> staging row cc, bytes [rb * kUnitCodeBytes / 32, + kUnitCodeBytes)
        const uint32_t b0 = static_cast<uint32_t>(rb * kUnitCodeBytes / 32);
        *reinterpret_cast<uint4*>(staging + staging_offset<S>(cc, b0)) = make_uint4(w[0], w[1], w[2], w[3]);
        if constexpr (kFp8)
          *reinterpret_cast<uint4*>(staging + staging_offset<S>(cc, b0 + 16)) = make_uint4(w[4], w[5], w[6], w[7]);
      }
      // scale bytes of column c: row c of the column layout, scale columns from rt / BS on
      const int64_t rt = r0 + gh * kColUnits * 32;
      const int64_t grp = rt / (4 * BS);
      constexpr int kBytes = kColUnits * kUnitScales;  // 1, 2 or 4, never crossing a word
      if (grp < a.nct_col) {
        const int64_t off =
            (tj * a.nct_col + grp) * 512 + (cc & 31) * 16 + ((cc >> 5) & 3) * 4 + (rt / BS) % 4;
        if (in_bounds(off + kBytes <= a.col_scales_bytes, a.status)) {
          if constexpr (kBytes == 4) *reinterpret_cast<uint32_t*>(a.col_scales + off) = sbytes;
          else if constexpr (kBytes == 2) *reinterpret_cast<uint16_t*>(a.col_scales + off) = static_cast<uint16_t>(sbytes);
          else a.col_scales[off] = static_cast<uint8_t>(sbytes);
        }
      }
    }

    // every read of the tile is done: release it to the producer
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[stage]);
    // staging complete and visible to the async proxy -> one TMA store of the transposed codes
    // (rows of the column layout beyond C and bytes beyond R are clipped by the tensor map)
    fence_proxy_async_smem();
    consumers_sync();
    if (issuer && r0 < R) {
      tma_store_2d(&col_map, staging, static_cast<int32_t>(r0 * kUnitCodeBytes / 32), static_cast<int32_t>(c0));
      bulk_commit_group();
      stored = true;
    }
    if (++stage == kDStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
  if constexpr (kNv) {
    if (a.g_in != nullptr) {  // given mode: this tensor's amax into both tails
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) run_max = max(run_max, __shfl_xor_sync(0xFFFFFFFFu, run_max, o));
      if (lane == 0 && run_max != 0) {
        atomicMax(&a.row_tail[1], run_max);
        atomicMax(&a.col_tail[1], run_max);
      }
    }
  }
  if (issuer && stored) bulk_wait_group0();  // the last stores have completed
}

template <int FMT, bool F32, bool SR>
cudaError_t launch_d(const CUtensorMap& src_map, const CUtensorMap& col_map, const DualArgs& a, int grid,
                     cudaStream_t stream, int device) {
  static PerDevice<cudaError_t> setup;  // the shared-memory opt-in holds per device
  const cudaError_t attr = setup.run(device, [] {
    return cudaFuncSetAttribute(dual_kernel<FMT, F32, SR>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDSmem);
  });
  if (attr != cudaSuccess) return attr;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDThreads);
  cfg.dynamicSmemBytes = kDSmem;
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dual_kernel<FMT, F32, SR>, src_map, col_map, a);
}

template <int FMT>
cudaError_t launch_d_fmt(bool f32, bool sr, const CUtensorMap& src_map, const CUtensorMap& col_map,
                         const DualArgs& a, int grid, cudaStream_t stream, int device) {
  if (f32) {
    return sr ? launch_d<FMT, true, true>(src_map, col_map, a, grid, stream, device)
              : launch_d<FMT, true, false>(src_map, col_map, a, grid, stream, device);
  }
  return sr ? launch_d<FMT, false, true>(src_map, col_map, a, grid, stream, device)
            : launch_d<FMT, false, false>(src_map, col_map, a, grid, stream, device);
}

}  // namespace

int launch_quantize_dual(int fmt, bool src_f32, bool stochastic, bool global_given, uint64_t seed, const void* src,
                         int64_t rows, int64_t cols, void* row_codes, void* row_scales, void* col_codes,
                         void* col_scales, float* global_scale, cudaStream_t stream, const DeviceInfo& dev) {
  const int64_t esize = src_f32 ? 4 : 2;
  const int64_t tile_rows = kDTileBytes / (kDCols * esize);
  const int64_t bs = block_size(fmt);
  DualArgs a{};
  a.rows = rows;
  a.cols = cols;
  a.row_codes = static_cast<uint8_t*>(row_codes);
  a.row_scales = static_cast<uint8_t*>(row_scales);
  a.col_codes = static_cast<uint8_t*>(col_codes);
  a.col_scales = static_cast<uint8_t*>(col_scales);
  a.tiles_c = ceil_div(cols, kDCols);
  // row tiles cover the rows padded to 128, so that every scale byte of both layouts is written
  a.ntiles = (ceil_div(rows, 128) * 128 / tile_rows) * a.tiles_c;
  a.nct_row = ceil_div(cols, 4 * bs);
  a.nct_col = ceil_div(rows, 4 * bs);
  a.codes_bytes = fmt == BSQ_MXFP8 ? rows * cols : rows * cols / 2;
  a.row_scales_bytes = scales_body_bytes(fmt, rows, cols);
  a.col_scales_bytes = scales_body_bytes(fmt, cols, rows);
  a.seed_lo = static_cast<uint32_t>(seed);
  a.seed_hi = static_cast<uint32_t>(seed >> 32);
  for (int i = 0; i < 10; ++i) {
    a.keys[2 * i] = a.seed_lo + static_cast<uint32_t>(i) * 0x9E3779B9u;
    a.keys[2 * i + 1] = a.seed_hi + static_cast<uint32_t>(i) * 0xBB67AE85u;
  }
  a.status = dev.status;
  const StallInjection inj = take_stall(BSQ_KERNEL_DUAL);
  a.stall_after = inj.after;
  a.wait_ns = inj.limit_ns;
  if (fmt == BSQ_NVFP4) {
    a.row_tail = reinterpret_cast<uint32_t*>(a.row_scales + scales_body_bytes(fmt, rows, cols));
    a.col_tail = reinterpret_cast<uint32_t*>(a.col_scales + scales_body_bytes(fmt, cols, rows));
    a.g_in = global_given ? global_scale : nullptr;
    a.g_out = global_given ? nullptr : global_scale;
    if (cudaMemsetAsync(a.row_tail, 0, 16, stream) != cudaSuccess) return BSQ_ERR_LAUNCH;
    if (cudaMemsetAsync(a.col_tail, 0, 16, stream) != cudaSuccess) return BSQ_ERR_LAUNCH;
    const int64_t elems = rows * cols;
    uint32_t* amax_out = a.row_tail + 1;
    if (!global_given && launch_amax(&src, &elems, &amax_out, 1, src_f32, stream, dev) != BSQ_OK)
      return BSQ_ERR_LAUNCH;
  }
  CUtensorMap map, col_map;
  if (!make_map_2d(&map, src_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, src,
                   static_cast<uint64_t>(cols), static_cast<uint64_t>(rows), static_cast<uint64_t>(cols * esize), kDCols,
                   static_cast<uint32_t>(tile_rows), CU_TENSOR_MAP_SWIZZLE_NONE))
    return BSQ_ERR_LAUNCH;
  // the column-layout codes as `cols` rows of R code bytes (MXFP8) or R / 2 (4-bit); a box is
  // one tile's staging: 128 rows of tile_rows codes
  const int64_t code_row = fmt == BSQ_MXFP8 ? rows : rows / 2;
  const uint32_t box_inner = static_cast<uint32_t>(fmt == BSQ_MXFP8 ? tile_rows : tile_rows / 2);
  const CUtensorMapSwizzle sw = box_inner == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : box_inner == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                  : CU_TENSOR_MAP_SWIZZLE_32B;
  if (!make_map_2d(&col_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, col_codes, static_cast<uint64_t>(code_row),
                   static_cast<uint64_t>(cols), static_cast<uint64_t>(code_row), box_inner, kDCols, sw))
    return BSQ_ERR_LAUNCH;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(a.ntiles, kDCtasPerSm * dev.num_sms)));
  cudaError_t err;
  if (fmt == BSQ_MXFP8) err = launch_d_fmt<BSQ_MXFP8>(src_f32, stochastic, map, col_map, a, grid, stream, dev.device);
  else if (fmt == BSQ_MXFP4) err = launch_d_fmt<BSQ_MXFP4>(src_f32, stochastic, map, col_map, a, grid, stream, dev.device);
  else err = launch_d_fmt<BSQ_NVFP4>(src_f32, stochastic, map, col_map, a, grid, stream, dev.device);
  return err == cudaSuccess ? BSQ_OK : BSQ_ERR_LAUNCH;
}

}  // namespace bsq
