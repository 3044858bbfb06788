// bsq_gemm.cu -- block-scaled GEMM on the 5th-generation tensor cores (tcgen05, sm_103a):
//   out[m, n] = bf16_rn(alpha * sum_k Ahat[m, k] * Bhat[n, k] + bias[n])
// for MXFP8 (kind::mxf8f6f4, UE8M0 scale per 32 K), NVFP4 (kind::mxf4nvf4, E4M3 scale per
// 16 K, alpha = g_A * g_B) and MXFP4 (kind::mxf4, UE8M0 scale per 32 K). The formats are the
// ones of the "lightly-train - DINOv3 + EoMT on RTX 5090" README, section 2; the README's
// kernels are sm_120 mma.sync designs, this one is written for tcgen05 + TMEM + TMA.
//
// Design (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0      TMA producer: A tile 128 rows x 128 bytes, B tile 256 rows x 128 bytes
//               (128-byte swizzle, K-major), plus the tile's scale-factor atoms (512-byte
//               blocks already in the tcgen05 layout) by bulk copy, into a kStages ring.
//   warp 1      TMEM owner and MMA issuer: per stage it copies the scale atoms smem -> TMEM
//               (tcgen05.cp 32x128b.warpx4, one TMEM slot per ring stage) and issues four
//               block-scaled MMAs of M=128, N=256 into one fp32 accumulator (256 columns);
//               tcgen05.commit frees the stage and, after the last K step, signals the tile.
//   warps 2..9  epilogue: warp w reads TMEM lanes 32*(w%4).. (its quadrant), columns
//               128*((w-2)/4).. (its half); it drains its 32 x 128 accumulator block to
//               registers, releases the accumulator to the MMA warp at once, then applies
//               alpha and bias, rounds to bf16 and writes 32 x 32 chunks through a
//               64-byte-swizzled staging buffer with TMA stores.
// Every mbarrier wait is bounded (%globaltimer); on a timeout the kernel records
// BSQ_ERR_TIMEOUT in the device status word, all roles leave their loops, the MMA warp
// waits for its own outstanding tensor-core work and TMEM is released before exit.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "bsq_device.cuh"
#include "bsq_internal.h"

namespace bsq {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int kRowBytes = 128;  // K bytes per stage and row: one 128-byte swizzle span
constexpr int kNumEpiWarps = 8;
constexpr int kAccCols = BN;     // fp32 accumulator columns in TMEM
constexpr uint32_t kTmemCols = 512;
constexpr int kABytes = BM * kRowBytes;  // 16 KB
constexpr int kBBytes = BN * kRowBytes;  // 32 KB
constexpr int kEpiChunkBytes = 32 * 32 * 2;

template <int FMT>
struct Cfg;
template <>
struct Cfg<BSQ_MXFP8> {  // 128 K per stage = 4 MMAs of K 32; 4 UE8M0 scales per row per stage
  static constexpr int kStages = 4, kKElems = 128, kAtoms = 1, kSfCols = 16, kSfWarps = 1;
};
template <>
struct Cfg<BSQ_NVFP4> {  // 256 K per stage = 4 MMAs of K 64; 16 E4M3 scales per row per stage
  static constexpr int kStages = 3, kKElems = 256, kAtoms = 4, kSfCols = 64, kSfWarps = 2;
};
template <>
struct Cfg<BSQ_MXFP4> {  // 256 K per stage = 4 MMAs of K 64; 8 UE8M0 scales per row per stage
  static constexpr int kStages = 4, kKElems = 256, kAtoms = 2, kSfCols = 32, kSfWarps = 1;
};

// Warp roles: 0 TMA producer, 1 MMA issuer, 2 .. 1 + kSfWarps scale-factor copiers, then
// kNumEpiWarps epilogue warps.
template <int FMT>
__host__ __device__ constexpr int first_epi_warp() {
  return 2 + Cfg<FMT>::kSfWarps;
}
template <int FMT>
__host__ __device__ constexpr int threads_of() {
  return (first_epi_warp<FMT>() + kNumEpiWarps) * 32;
}

template <int FMT>
struct Smem {
  static constexpr int S = Cfg<FMT>::kStages;
  static constexpr int kSfaBytes = Cfg<FMT>::kAtoms * 512;
  static constexpr int kSfbBytes = 2 * Cfg<FMT>::kAtoms * 512;
  static constexpr int a_off = 0;
  static constexpr int b_off = a_off + S * kABytes;
  static constexpr int sfa_off = b_off + S * kBBytes;
  static constexpr int sfb_off = sfa_off + S * kSfaBytes;
  static constexpr int epi_off = ((sfb_off + S * kSfbBytes) + 1023) / 1024 * 1024;
  static constexpr int bias_off = epi_off + kNumEpiWarps * kEpiChunkBytes;
  static constexpr int bar_off = bias_off + kNumEpiWarps * 128 * 4;
  static constexpr int kNumBars = 3 * S + 4;
  static constexpr int misc_off = bar_off + kNumBars * 8;
  static constexpr int total = misc_off + 16;
  static constexpr int alloc = total + 1024;  // slack for aligning the base to 1024
};
static_assert(Smem<BSQ_MXFP8>::alloc <= 232448, "MXFP8 shared memory budget");
static_assert(Smem<BSQ_NVFP4>::alloc <= 232448, "NVFP4 shared memory budget");
static_assert(Smem<BSQ_MXFP4>::alloc <= 232448, "MXFP4 shared memory budget");
static_assert(kAccCols + Cfg<BSQ_MXFP8>::kStages * Cfg<BSQ_MXFP8>::kSfCols <= 512, "TMEM budget");
static_assert(kAccCols + Cfg<BSQ_NVFP4>::kStages * Cfg<BSQ_NVFP4>::kSfCols <= 512, "TMEM budget");
static_assert(kAccCols + Cfg<BSQ_MXFP4>::kStages * Cfg<BSQ_MXFP4>::kSfCols <= 512, "TMEM budget");

// Instruction descriptor of a block-scaled MMA (kinds mxf8f6f4 / mxf4 / mxf4nvf4):
// bits 4-5 scale-factor B id, 7-9 A type, 10-12 B type, 15/16 A/B major (0 = K-major),
// 17-22 N >> 3, 23 scale type (1 = UE8M0, 0 = UE4M3), 27-28 M >> 7, 29-30 scale-factor A id.
// Element types: E4M3 = 0 under mxf8f6f4, E2M1 = 1 under mxf4 / mxf4nvf4.
template <int FMT>
__host__ __device__ constexpr uint32_t make_idesc(uint32_t sf_id) {
  const uint32_t t = (FMT == BSQ_MXFP8) ? 0u : 1u;
  const uint32_t ue8m0 = (FMT == BSQ_NVFP4) ? 0u : 1u;
  return (sf_id << 4) | (t << 7) | (t << 10) | (static_cast<uint32_t>(BN >> 3) << 17) | (ue8m0 << 23) |
         (static_cast<uint32_t>(BM >> 7) << 27) | (sf_id << 29);
}

struct GemmArgs {
  const uint8_t* sfa;
  const uint8_t* sfb;
  const uint16_t* bias;  // nullable
  const float* ga;       // NVFP4: per-tensor scales in the scale tails
  const float* gb;
  int M, N, K;
  int tiles_n, num_tiles, nk;
  int sf_nct;          // 4-column scale tiles per row (K / block / 4)
  int sfb_row_tiles;   // ceil(N / 128)
  int* status;
};

template <int FMT>
__global__ void __launch_bounds__(threads_of<FMT>(), 1)
    gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                const __grid_constant__ CUtensorMap mapOut, const GemmArgs args) {
  using C = Cfg<FMT>;
  using L = Smem<FMT>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bar_off);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + S;
  uint64_t* sf_ready = bars + 2 * S;
  uint64_t* tmem_full = bars + 3 * S;
  uint64_t* tmem_empty = bars + 3 * S + 1;
  uint64_t* drain_bar = bars + 3 * S + 2;     // MMA issuer's outstanding work
  uint64_t* sf_drain_bar = bars + 3 * S + 3;  // scale-factor copiers' outstanding work
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
      mbar_init(&sf_ready[s], C::kSfWarps);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, kNumEpiWarps);
    mbar_init(drain_bar, 1);
    mbar_init(sf_drain_bar, C::kSfWarps);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&mapA);
    prefetch_tmap(&mapB);
    prefetch_tmap(&mapOut);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < args.num_tiles && ok; tile += gridDim.x) {
      const int m_blk = tile / args.tiles_n, n_blk = tile % args.tiles_n;
      for (int kb = 0; kb < args.nk; ++kb) {
        if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, args.status)) {
          ok = false;
          break;
        }
        const bool hi_ok = (2 * n_blk + 1) < args.sfb_row_tiles;
        const uint32_t bytes = kABytes + kBBytes + L::kSfaBytes + (hi_ok ? 2 : 1) * (L::kSfaBytes);
        mbar_arrive_expect_tx(&full_bar[stage], bytes);
        tma_load_2d(smem + L::a_off + stage * kABytes, &mapA, &full_bar[stage], kb * kRowBytes, m_blk * BM);
        tma_load_2d(smem + L::b_off + stage * kBBytes, &mapB, &full_bar[stage], kb * kRowBytes, n_blk * BN);
        const int64_t atom_a = static_cast<int64_t>(m_blk) * args.sf_nct + static_cast<int64_t>(kb) * C::kAtoms;
        bulk_load(smem + L::sfa_off + stage * L::kSfaBytes, args.sfa + atom_a * 512, L::kSfaBytes, &full_bar[stage]);
        for (int h = 0; h < (hi_ok ? 2 : 1); ++h) {
          const int64_t atom_b =
              static_cast<int64_t>(2 * n_blk + h) * args.sf_nct + static_cast<int64_t>(kb) * C::kAtoms;
          bulk_load(smem + L::sfb_off + stage * L::kSfbBytes + h * L::kSfaBytes, args.sfb + atom_b * 512,
                    L::kSfaBytes, &full_bar[stage]);
        }
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------------ MMA issuer
    // Every tcgen05 instruction and every mbarrier wait costs the issuing thread a few dozen
    // cycles; one MMA of 128 x 256 takes 128 tensor cycles. The issuer therefore does only the
    // waits, the four MMAs and the commit of each stage (the scale-factor copies run on their
    // own warps), with descriptors precomputed so that each MMA is a couple of adds.
    int stage = 0;
    uint32_t phase = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    const uint64_t adesc0 = smem_desc(smem_u32(smem + L::a_off), 16, 1024, kSwizzle128B);
    const uint64_t bdesc0 = smem_desc(smem_u32(smem + L::b_off), 16, 1024, kSwizzle128B);
    for (int tile = blockIdx.x; tile < args.num_tiles && ok; tile += gridDim.x) {
      // wait until the epilogue has drained the accumulator of the previous tile
      if (!mbar_wait_bounded(tmem_empty, acc_phase ^ 1u, abort_flag, args.status)) break;
      acc_phase ^= 1u;
      tc_fence_after();
      for (int kb = 0; kb < args.nk; ++kb) {
        // operands landed (full) and this stage's scale factors are in TMEM (sf_ready)
        if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag, args.status) ||
            !mbar_wait_bounded(&sf_ready[stage], phase, abort_flag, args.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sfa_t = tmem_base + kAccCols + stage * C::kSfCols;
        const uint32_t sfb_t = sfa_t + 4 * C::kAtoms;
        // start-address field of the descriptors is in 16-byte units (stays below 2^14)
        const uint64_t adesc = adesc0 + static_cast<uint64_t>((stage * kABytes) >> 4);
        const uint64_t bdesc = bdesc0 + static_cast<uint64_t>((stage * kBBytes) >> 4);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t sfa = sfa_t, sfb = sfb_t, id = 0;
          if constexpr (FMT == BSQ_MXFP8) {
            id = k;  // byte k of each 32-bit scale cell: K block k of this stage
          } else if constexpr (FMT == BSQ_NVFP4) {
            sfa += 4 * k;  // one atom (4 scales of 16 K) per MMA
            sfb += 8 * k;
          } else {
            sfa += 4 * (k >> 1);  // two scales of 32 K per MMA: bytes {0,1} or {2,3}
            sfb += 8 * (k >> 1);
            id = 2 * (k & 1);
          }
          tc_mma_block_scaled<FMT>(tmem_base, adesc + 2 * k, bdesc + 2 * k, make_idesc<FMT>(id), sfa, sfb,
                                   (kb | k) != 0 ? 1u : 0u);
        }
        tc_commit(&empty_bar[stage]);  // the stage is free once these MMAs have read it
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) tc_commit(tmem_full);  // accumulator complete
    }
    // every tensor-core operation of this thread must finish before TMEM is released
    tc_commit(drain_bar);
    mbar_wait_bounded(drain_bar, 0, nullptr, args.status);
  } else if (warp >= 2 && warp < first_epi_warp<FMT>()) {
    // ------------------------------------------------------------------ scale-factor copiers
    // Each of the kSfWarps warps copies its share of the stage's 512-byte scale atoms from
    // shared memory into the stage's TMEM slot, then commits onto sf_ready[stage] (count
    // kSfWarps): the commit arrives once the copies are done.
    if (lane == 0) {
      constexpr int kCps = 3 * C::kAtoms;  // A atoms, then B atoms (two 128-row halves each)
      constexpr int kPer = kCps / C::kSfWarps;
      static_assert(kCps % C::kSfWarps == 0, "scale copies split evenly");
      const int first = (warp - 2) * kPer;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < args.num_tiles && ok; tile += gridDim.x) {
        for (int kb = 0; kb < args.nk; ++kb) {
          if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa_t = tmem_base + kAccCols + stage * C::kSfCols;
          const uint32_t sfb_t = sfa_t + 4 * C::kAtoms;
          const uint32_t sfa_s = smem_u32(smem + L::sfa_off + stage * L::kSfaBytes);
          const uint32_t sfb_s = smem_u32(smem + L::sfb_off + stage * L::kSfbBytes);
#pragma unroll
          for (int c = 0; c < kPer; ++c) {
            const int i = first + c;
            if (i < C::kAtoms) {
              tc_cp_32x128b_warpx4(sfa_t + 4 * i, smem_desc(sfa_s + 512 * i, 128, 128, kSwizzleNone));
            } else {
              const int j = i - C::kAtoms, at = j >> 1, h = j & 1;
              tc_cp_32x128b_warpx4(sfb_t + 8 * at + 4 * h,
                                   smem_desc(sfb_s + h * L::kSfaBytes + 512 * at, 128, 128, kSwizzleNone));
            }
          }
          tc_commit(&sf_ready[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // the copies must be finished before TMEM is released
      tc_commit(sf_drain_bar);
      mbar_wait_bounded(sf_drain_bar, 0, nullptr, args.status);
    }
  } else if (warp >= first_epi_warp<FMT>()) {
    // ------------------------------------------------------------------ epilogue
    const uint32_t e = warp - first_epi_warp<FMT>();  // 0..7
    const uint32_t quad = warp & 3u;                  // TMEM lane quadrant this warp may access
    const uint32_t half = e >> 2;
    uint8_t* stage_buf = smem + L::epi_off + e * kEpiChunkBytes;
    float* bias_s = reinterpret_cast<float*>(smem + L::bias_off) + e * 128;
    float alpha = 1.0f;
    if constexpr (FMT == BSQ_NVFP4) alpha = __fmul_rn(*args.ga, *args.gb);
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < args.num_tiles; tile += gridDim.x) {
      const int m_blk = tile / args.tiles_n, n_blk = tile % args.tiles_n;
      const int n0 = n_blk * BN + half * 128;
      const int m0 = m_blk * BM + quad * 32;
      // bias of this warp's 128 columns (zero past N or without bias)
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int n = n0 + 4 * lane + i;
        bias_s[4 * lane + i] =
            (args.bias != nullptr && n < args.N) ? __uint_as_float(static_cast<uint32_t>(args.bias[n]) << 16) : 0.0f;
      }
      __syncwarp();
      if (!mbar_wait_bounded(tmem_full, acc_phase, abort_flag, args.status)) break;
      acc_phase ^= 1u;
      tc_fence_after();
      uint32_t acc[4][32];
      const uint32_t taddr = tmem_base + ((quad * 32u) << 16) + half * 128u;
#pragma unroll
      for (int j = 0; j < 4; ++j) tmem_ld_32x32b_x32(taddr + 32u * j, acc[j]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmem_empty);  // accumulator may be overwritten now

#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (lane == 0) bulk_wait_group_read0();  // staging buffer free again
        __syncwarp();
        uint32_t packed[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float b0 = bias_s[32 * j + 2 * c], b1 = bias_s[32 * j + 2 * c + 1];
          float v0 = __uint_as_float(acc[j][2 * c]), v1 = __uint_as_float(acc[j][2 * c + 1]);
          if constexpr (FMT == BSQ_NVFP4) {
            v0 = __fmaf_rn(v0, alpha, b0);
            v1 = __fmaf_rn(v1, alpha, b1);
          } else {
            v0 = __fadd_rn(v0, b0);
            v1 = __fadd_rn(v1, b1);
          }
          __nv_bfloat162 p = __floats2bfloat162_rn(v0, v1);
          packed[c] = *reinterpret_cast<uint32_t*>(&p);
        }
        // row `lane` of the 32 x 32 chunk, 64 bytes, 16-byte pieces swizzled (64-byte mode)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t phys = (static_cast<uint32_t>(q) ^ ((lane >> 1) & 3u)) << 4;
          *reinterpret_cast<uint4*>(stage_buf + lane * 64 + phys) =
              make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int x = n0 + 32 * j;
        if (lane == 0 && x < args.N && m0 < args.M) {
          tma_store_2d(&mapOut, stage_buf, x, m0);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT>
int run_gemm(const void* A, const void* A_scales, const void* B, const void* B_scales, const void* bias, void* out,
             int64_t M, int64_t N, int64_t K, cudaStream_t stream, const DeviceInfo& dev) {
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(gemm_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<FMT>::alloc);
  });
  if (attr_err != cudaSuccess) return BSQ_ERR_LAUNCH;

  const uint64_t kbytes = (FMT == BSQ_MXFP8) ? static_cast<uint64_t>(K) : static_cast<uint64_t>(K) / 2;
  CUtensorMap mA, mB, mOut;
  if (!make_map_2d(&mA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, kbytes, M, kbytes, kRowBytes, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&mB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, kbytes, N, kbytes, kRowBytes, BN,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&mOut, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out, N, M, static_cast<uint64_t>(N) * 2, 32, 32,
                   CU_TENSOR_MAP_SWIZZLE_64B))
    return BSQ_ERR_LAUNCH;

  GemmArgs a{};
  a.sfa = static_cast<const uint8_t*>(A_scales);
  a.sfb = static_cast<const uint8_t*>(B_scales);
  a.bias = static_cast<const uint16_t*>(bias);
  a.ga = reinterpret_cast<const float*>(a.sfa + scales_body_bytes(FMT, M, K));
  a.gb = reinterpret_cast<const float*>(a.sfb + scales_body_bytes(FMT, N, K));
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  const int tiles_m = static_cast<int>(ceil_div(M, BM));
  a.tiles_n = static_cast<int>(ceil_div(N, BN));
  a.num_tiles = tiles_m * a.tiles_n;
  a.nk = static_cast<int>(K / Cfg<FMT>::kKElems);
  a.sf_nct = static_cast<int>(K / block_size(FMT) / 4);
  a.sfb_row_tiles = static_cast<int>(ceil_div(N, 128));
  a.status = dev.status;
  const int grid = std::min(a.num_tiles, dev.num_sms);
  gemm_kernel<FMT><<<grid, threads_of<FMT>(), Smem<FMT>::alloc, stream>>>(mA, mB, mOut, a);
  return cudaGetLastError() == cudaSuccess ? BSQ_OK : BSQ_ERR_LAUNCH;
}

}  // namespace

int launch_gemm(int fmt, const void* A, const void* A_scales, const void* B, const void* B_scales, const void* bias,
                void* out, int64_t M, int64_t N, int64_t K, cudaStream_t stream, const DeviceInfo& dev) {
  switch (fmt) {
    case BSQ_MXFP8:
      return run_gemm<BSQ_MXFP8>(A, A_scales, B, B_scales, bias, out, M, N, K, stream, dev);
    case BSQ_NVFP4:
      return run_gemm<BSQ_NVFP4>(A, A_scales, B, B_scales, bias, out, M, N, K, stream, dev);
    case BSQ_MXFP4:
      return run_gemm<BSQ_MXFP4>(A, A_scales, B, B_scales, bias, out, M, N, K, stream, dev);
    default:
      return BSQ_ERR_ARG;
  }
}

}  // namespace bsq
