// bsq_gemm.cu -- block-scaled GEMM on the 5th-generation tensor cores (tcgen05, sm_103a):
//   out[m, n] = bf16_rn(alpha * sum_k Ahat[m, k] * Bhat[n, k] + bias[n])
// for MXFP8 (kind::mxf8f6f4, UE8M0 scale per 32 K), NVFP4 (kind::mxf4nvf4, E4M3 scale per
// 16 K, alpha = g_A * g_B) and MXFP4 (kind::mxf4, UE8M0 scale per 32 K). The formats are the
// ones of the "lightly-train - DINOv3 + EoMT on RTX 5090" README, section 2; the README's
// kernels are sm_120 mma.sync designs, this one is written for tcgen05 + TMEM + TMA.
//
// Why 2-SM tiles. A stage of a 128 x 256 single-CTA tile brings 48 KB into one SM's shared
// memory for 512 tensor cycles of work, and TMA fills one SM's shared memory at ~84 bytes per
// cycle (measured on GB300), so a single CTA cannot feed its tensor core. The 2-SM MMA
// (.cta_group::2) computes a 256 x 256 tile on a pair of SMs with each SM holding only its 128
// rows of A and its 128-row half of B: 32 KB per stage per SM for the same 512 cycles.
//
// Design (a (2,1,1) cluster per SM pair, persistent over 256 x 256 tiles; rank 0 = leader):
//   warp 0      (both CTAs) TMA producer: per stage one 128-byte K chunk of the CTA's A rows
//               and of its half of the B rows (128-byte swizzle, K-major), the CTA's A scale
//               atoms and all B scale atoms of the tile, into a kStages ring. Every copy is a
//               tensor copy in its .cta_group::2 form, completing on the LEADER's full[]
//               barrier, which expects the bytes of both CTAs: the leader learns that the
//               whole stage landed without any relay between the CTAs.
//   warp 1      leader: TMEM owner and MMA issuer. The whole warp runs the loop (operands
//               stay warp-uniform) and one elected lane issues, per stage, the scale-factor
//               copies into the stage's TMEM slot of both CTAs (tcgen05.cp.cta_group::2: each
//               CTA's TMEM gets its own shared-memory atoms), the four MMAs
//               (tcgen05.mma.cta_group::2, M=256 N=256) and one commit multicast to both
//               CTAs' empty[] barriers; one commit per tile to both CTAs' tmem_full.
//   warps 2..9  (both CTAs) epilogue: drain the CTA's 128 x 256 fp32 accumulator, alpha +
//               bias, bf16, swizzled staging, TMA store; tell the leader (tmem_empty, 16
//               arrivals) as soon as the accumulator has been read.
// Measured on GB300 (clock64 instrumentation): each tcgen05 instruction costs the issuing
// thread a few dozen cycles, so the issue loop holds nothing else; in one thread the tensor
// pipe keeps copies and MMAs in order, so a stage's scales need no extra barrier.
// Every mbarrier wait is bounded (%globaltimer); on a timeout the kernel records
// BSQ_ERR_TIMEOUT in the device status word, the roles leave their loops, outstanding
// tensor-core work is waited for and TMEM is released after a final cluster barrier.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "bsq_device.cuh"
#include "bsq_internal.h"

namespace bsq {
namespace {

constexpr int BM = 128;           // rows of A per CTA (256 per pair)
constexpr int BN = 256;           // columns of the output tile (both CTAs)
constexpr int BNH = BN / 2;       // rows of B held per CTA
constexpr int kChunkBytes = 128;  // K bytes per stage: one 128-byte swizzle span per row
constexpr int kMmasPerStage = 4;  // 32 K bytes per MMA
constexpr int kFirstEpiWarp = 2;
constexpr int kAccCols = BN;  // fp32 accumulator columns in TMEM
constexpr uint32_t kTmemCols = 512;

// Epilogue modes. kEpiBf16: out = bf16(v), v = alpha * acc + bias. kEpiGeluBf16: out =
// bf16(GELU(v)) (the "fc1 + GELU" epilogue every stack of the "lightly-train - DINOv3 + EoMT on
// RTX 5090" README fuses, section 4.3). kEpiGeluMxfp8 / kEpiGeluMxfp4: GELU(v) quantized along
// the output row straight into MX codes and tiled scales, the fc2 operand (the MXFP8 stack's
// fc1 epilogue, same section); bytes laid out as bsq_quantize writes them. kEpiConvT /
// kEpiConvTGelu: the head's kernel-2 stride-2 transposed convolution (same README section: the
// ScaleBlocks' ConvT, then GELU): column n = (2 dy + dx) C_out + co of output row (b, h, w) is
// stored at pixel (b, 2h + dy, 2w + dx), channel co, of the NHWC output, with bias[co].
// kEpiF32Partial: split-K -- K is cut into `splits` equal ranges of stages, the work units are
// (tile, range) pairs, and each unit stores its raw fp32 accumulator (no alpha, no bias) into
// slice `range` of an fp32 workspace of splits x M x N; splitk_finalize_kernel sums the slices.
// For shapes with fewer tiles than SM pairs and a long K (the weight gradient dW = dY^T X:
// M, N the weight's shape, K the token count), where one unit per tile leaves SMs idle.
enum EpiMode {
  kEpiBf16 = 0,
  kEpiGeluBf16 = 1,
  kEpiGeluMxfp8 = 2,
  kEpiGeluMxfp4 = 3,
  kEpiConvT = 4,
  kEpiConvTGelu = 5,
  kEpiF32Partial = 6
};

// Epilogue warps per CTA, by epilogue mode. The GELU epilogues are bound by their arithmetic
// (about 10 instructions per value) and run 16 warps, four per TMEM lane quadrant, of 64 columns
// each; the others are bound by their store phase, where more warps (and so more TMA stores in
// flight beside the operand loads) made the kernel slower, and run 8 warps of 128 columns.
// Measured on GB300, L2 flushed, M = 51200, K = 1024, N = 4096: fc1 with GELU into MXFP4 codes
// 188 -> 164 us with 16 warps; the plain NVFP4 fc1 96 -> 117 us with 16.
template <int EPI>
struct Epi {
  static constexpr bool kGelu =
      EPI == kEpiGeluBf16 || EPI == kEpiGeluMxfp8 || EPI == kEpiGeluMxfp4 || EPI == kEpiConvTGelu;
  static constexpr int kWarps = kGelu ? 16 : 8;
  static constexpr int kWarpCols = 4 * BN / kWarps;
  static constexpr int kAccRegs = kWarpCols / 32;  // 32-column TMEM loads per warp
  static constexpr int kThreads = (kFirstEpiWarp + kWarps) * 32;
};

// Per format: kStages stages in the ring, kAtoms 512-byte scale atoms per 128 rows per stage
// (4 scale columns of 128 rows each), kEpiCols output columns per epilogue store chunk and
// kEpiBufs staging buffers per epilogue warp (stores in flight per warp). A
// stage's scale slot in TMEM takes 4 columns per A atom and 8 per B atom (two 128-row halves).
// One staging buffer: the output's stores and the operand loads share the SMs' path to L2, and
// with two buffers the faster store stream starves the operand feed (measured on GB300, FP4 at
// M = 51200, K = 1024, N = 4096: 96 -> 112 us).
template <int FMT>
struct Cfg;
template <>
struct Cfg<BSQ_MXFP8> {  // 128 K per stage = 4 MMAs of K 32, one UE8M0 scale each
  static constexpr int kStages = 6, kAtoms = 1, kEpiCols = 32, kEpiBufs = 1;
};
template <>
struct Cfg<BSQ_NVFP4> {  // 256 K per stage = 4 MMAs of K 64, four E4M3 scales (one atom) each
  static constexpr int kStages = 5, kAtoms = 4, kEpiCols = 32, kEpiBufs = 1;
};
template <>
struct Cfg<BSQ_MXFP4> {  // 256 K per stage = 4 MMAs of K 64, two UE8M0 scales each
  // 5 stages leave room for 32-column store chunks: at K = 1024 (2048 MMA cycles per tile) the
  // epilogue's store round trips bound the tile, and halving their number beats a sixth stage
  static constexpr int kStages = 5, kAtoms = 2, kEpiCols = 32, kEpiBufs = 1;
};
template <int FMT>
__host__ __device__ constexpr int sf_cols() {
  return 12 * Cfg<FMT>::kAtoms;
}
// Pipeline stages of a (format, epilogue) kernel: MXFP8 with 16 epilogue warps takes 5, the
// staging buffers of the 8 extra warps not fitting beside a sixth.
template <int FMT, int EPI>
__host__ __device__ constexpr int stages() {
  return (FMT == BSQ_MXFP8 && Epi<EPI>::kWarps == 16) ? 5 : Cfg<FMT>::kStages;
}

template <int FMT, int EPI>
struct Smem {
  static constexpr int S = stages<FMT, EPI>();
  static constexpr int kABytes = BM * kChunkBytes;   // own 128 rows of A
  static constexpr int kBBytes = BNH * kChunkBytes;  // own 128-row half of B
  static constexpr int kSfaBytes = Cfg<FMT>::kAtoms * 512;      // this CTA's 128 A rows
  static constexpr int kSfbBytes = 2 * Cfg<FMT>::kAtoms * 512;  // all 256 B rows of the tile
  static constexpr int kEpiChunkBytes = 32 * Cfg<FMT>::kEpiCols * 2;
  static constexpr int a_off = 0;
  static constexpr int b_off = a_off + S * kABytes;
  static constexpr int sfa_off = b_off + S * kBBytes;
  static constexpr int sfb_off = sfa_off + S * kSfaBytes;
  static constexpr int epi_off = ((sfb_off + S * kSfbBytes) + 1023) / 1024 * 1024;
  static constexpr int bias_off = epi_off + Epi<EPI>::kWarps * Cfg<FMT>::kEpiBufs * kEpiChunkBytes;
  static constexpr int bar_off = bias_off + Epi<EPI>::kWarps * Epi<EPI>::kWarpCols * 4;
  static constexpr int kNumBars = 2 * S + 3;
  static constexpr int misc_off = bar_off + kNumBars * 8;
  static constexpr int total = misc_off + 16;
  static constexpr int alloc = total;  // the dynamic region is 1024-byte aligned (checked at kernel start)
};

// Instruction descriptor of a block-scaled MMA (kinds mxf8f6f4 / mxf4 / mxf4nvf4):
// bits 4-5 scale-factor B id, 7-9 A type, 10-12 B type, 15/16 A/B major (0 = K-major),
// 17-22 N >> 3, 23 scale type (1 = UE8M0, 0 = UE4M3), 27-28 M >> 7, 29-30 scale-factor A id.
// Element types: E4M3 = 0 under mxf8f6f4, E2M1 = 1 under mxf4 / mxf4nvf4. M = 256 (the pair).
template <int FMT>
__host__ __device__ constexpr uint32_t make_idesc(uint32_t sf_id) {
  const uint32_t t = (FMT == BSQ_MXFP8) ? 0u : 1u;
  const uint32_t ue8m0 = (FMT == BSQ_NVFP4) ? 0u : 1u;
  return (sf_id << 4) | (t << 7) | (t << 10) | (static_cast<uint32_t>(BN >> 3) << 17) | (ue8m0 << 23) |
         (static_cast<uint32_t>((2 * BM) >> 7) << 27) | (sf_id << 29);
}


// 3-D tile store (coordinates innermost first).
__device__ __forceinline__ void tma_store_3d(const void* tmap, const void* smem_src, int32_t c0, int32_t c1,
                                             int32_t c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}


// GELU(v) = v Phi(v) (the erf form) with Phi(v) = 1 - erfc(z) / 2 for v >= 0 and erfc(z) / 2
// for v < 0, z = |v| / sqrt 2 (no cancellation in the negative tail), and erfc from
// Abramowitz & Stegun, Handbook of Mathematical Functions, formula 7.1.26:
//   erfc(z) = (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-z^2) + err, t = 1 / (1 + p z),
//   |err| <= 1.5e-7,
// here for two values at once: one reciprocal and one exp2 per value on the special-function
// unit, the multiplies and FMAs in packed form (the coefficients carry the factor 1/2 of
// erfc(z) / 2, an exact scaling at every Horner step), about 10 instructions per value -- the
// GELU epilogues are bound by instruction issue, and the scalar form took 17 (bit-identical
// results; 8-11 % faster GEMMs with a GELU epilogue). Measured in fp32 against the exact
// function: |GELU_kernel(v) - GELU(v)| <= 1e-7 |v| + 2^-21 |GELU(v)| (plus about one ulp from
// the hardware reciprocal and exp2).
__device__ __forceinline__ void gelu_erf2(float& a, float& b) {
  const uint64_t z = f2(fabsf(a) * 0.7071067811865476f, fabsf(b) * 0.7071067811865476f);
  float xa, xb, ta, tb;
  f2_split(f2_fma(f2_splat(0.3275911f), z, f2_splat(1.0f)), xa, xb);
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(ta) : "f"(xa));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(tb) : "f"(xb));
  const uint64_t t = f2(ta, tb);
  uint64_t poly = f2_fma(f2_splat(0.5f * 1.061405429f), t, f2_splat(0.5f * -1.453152027f));
  poly = f2_fma(poly, t, f2_splat(0.5f * 1.421413741f));
  poly = f2_fma(poly, t, f2_splat(0.5f * -0.284496736f));
  poly = f2_fma(poly, t, f2_splat(0.5f * 0.254829592f));
  float la, lb, ea, eb;
  f2_split(f2_mul(f2_mul(z, z), f2_splat(-1.4426950408889634f)), la, lb);
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ea) : "f"(la));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(eb) : "f"(lb));
  const uint64_t h = f2_mul(f2_mul(poly, t), f2(ea, eb));  // erfc(z) / 2
  float ha, hb, ca, cb;
  f2_split(h, ha, hb);
  f2_split(f2_fma(h, f2_splat(-1.0f), f2_splat(1.0f)), ca, cb);  // 1 - h
  f2_split(f2_mul(f2(a, b), f2(a >= 0.0f ? ca : ha, b >= 0.0f ? cb : hb)), a, b);
}

struct GemmArgs {
  const uint16_t* bias;  // nullable
  uint8_t* qscales;      // quantized epilogues: tiled scales of the M x N output
  int q_nct;             // quantized epilogues: 4-column scale tiles per output row (N / 128, rounded up)
  const float* ga;       // NVFP4: per-tensor scales in the scale tails
  const float* gb;
  int M, N;
  int tiles_n, num_pairs;
  int splits, num_units;  // split-K ranges (1 outside kEpiF32Partial); work units = num_pairs * splits
  int nk;  // stages per tile: K bytes / 128
  int cv_c, cv_w;  // ConvT epilogues: output channels C_out, input width W
  int* status;
  int64_t stall_after;  // injected stall (tests): producers stop after this many stages; -1 = none
  uint64_t wait_ns;     // limit of every bounded wait
  int64_t qscales_bytes;  // size of the quantized epilogues' tiled scale body (index checks)
  int bias_len;           // bias values: N, or C_out for the transposed convolutions
};

template <int FMT, int EPI>
__global__ void __launch_bounds__(Epi<EPI>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                const __grid_constant__ CUtensorMap mapSfa, const __grid_constant__ CUtensorMap mapSfb,
                const __grid_constant__ CUtensorMap mapOut, const GemmArgs args) {
  using C = Cfg<FMT>;
  using L = Smem<FMT, EPI>;
  constexpr int S = stages<FMT, EPI>();
  constexpr int kNumEpiWarps = Epi<EPI>::kWarps;
  constexpr int kWarpCols = Epi<EPI>::kWarpCols;
  constexpr int kAccRegs = Epi<EPI>::kAccRegs;
  static_assert(L::alloc <= 232448, "shared memory budget");
  static_assert(kAccCols + S * sf_cols<FMT>() <= 512, "TMEM budget");
  extern __shared__ __align__(1024) uint8_t smem[];
  // the 128-byte swizzled operand tiles need a 1024-byte aligned base (uniform: every thread of
  // both CTAs leaves before touching a barrier)
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicCAS(args.status, 0, BSQ_ERR_LAUNCH);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bar_off);
  uint64_t* full_bar = bars;                // leader: both CTAs' operands of a stage landed
  uint64_t* empty_bar = bars + S;           // the pair's MMAs are done with a stage
  uint64_t* tmem_full = bars + 2 * S;       // the accumulator of a tile is complete
  uint64_t* tmem_empty = bars + 2 * S + 1;  // leader: both CTAs drained their accumulator
  uint64_t* drain_bar = bars + 2 * S + 2;   // leader: MMA issuer's outstanding work
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::misc_off + 4);

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t rank = cluster_rank();
  const bool leader = (rank == 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, 2 * kNumEpiWarps);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&mapA);
    prefetch_tmap(&mapB);
    prefetch_tmap(&mapSfa);
    prefetch_tmap(&mapSfb);
    prefetch_tmap(&mapOut);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, kTmemCols);  // one warp in each CTA, collectively
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // barriers of both CTAs initialised before any remote arrival
  tc_fence_after();
  launch_dependents();
  grid_dependency_wait();  // the operands (and the output buffer) may belong to the previous kernel until here
  const uint32_t tmem_base = *tmem_holder;
  const int first_pair = static_cast<int>(cluster_id_x());
  const int pair_stride = static_cast<int>(num_clusters_x());
  // The producer and the MMA issuer address shared memory through a copy of its base that the
  // compiler cannot fold into constant offsets; the epilogue keeps the folded base. Measured on
  // GB300 (graph-replayed, L2 flushed), each choice is the faster one for its roles: the copy in
  // the two issue loops took ViT-B fc1 MXFP8 from 29.1 to 28.1 us and the MXFP4 fc2 at M = 51200
  // from 71.5 to 70.2 us; the copy in the epilogue as well cost the FP4 fc1 at M = 51200 3 us.
  uint8_t* smem_issue;
  asm volatile("mov.b64 %0, %1;" : "=l"(smem_issue) : "l"(smem));

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    uint8_t* const smem = smem_issue;  // shadows the array: addresses from the runtime base
    uint64_t* const full_bar = reinterpret_cast<uint64_t*>(smem + L::bar_off);
    uint64_t* const empty_bar = full_bar + S;
    // Boxes reaching past M, N or the scale atoms are zero-filled by TMA and still deliver
    // their full byte count, so every stage of every CTA brings exactly kStageBytes.
    constexpr uint32_t kStageBytes = L::kABytes + L::kBBytes + L::kSfaBytes + L::kSfbBytes;
    // every row block of A (codes and scales) is read by tiles_n tiles and every column block of
    // B by all row blocks: keep the operands in L2 ahead of the output lines the epilogue streams
    // through it (measured: 4-6 % faster on the ViT shapes than default caching)
    const uint64_t keep = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int64_t armed = 0;  // stages armed so far (ring order from stage 0)
    // The loop, instantiated twice: the injected stall (tests) is compared only in the copy that
    // runs when one is armed (the compare in every stage measured ~1 us per launch on GB300).
    auto produce = [&](auto stall) {
      for (int u = first_pair; u < args.num_units && ok; u += pair_stride) {
        const int split = u / args.num_pairs, pt = u - split * args.num_pairs;
        const int m_blk = 2 * (pt / args.tiles_n) + static_cast<int>(rank);
        const int n_blk = pt % args.tiles_n;
        const int kb1 = (split + 1) * args.nk / args.splits;
        for (int kb = split * args.nk / args.splits; kb < kb1; ++kb) {
          if constexpr (decltype(stall)::value) {
            if (armed == args.stall_after) {  // injected stall: no more loads, none announced
              ok = false;
              break;
            }
          }
          if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, args.status, args.wait_ns)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * kStageBytes);
          const uint32_t bar = smem_u32(&full_bar[stage]) & ~kClusterRankBit;  // the leader's full[stage]
          tma_load_2d_to_leader(smem + L::a_off + stage * L::kABytes, &mapA, bar, kb * kChunkBytes, m_blk * BM, keep);
          tma_load_2d_to_leader(smem + L::b_off + stage * L::kBBytes, &mapB, bar, kb * kChunkBytes,
                                n_blk * BN + static_cast<int>(rank) * BNH, keep);
          tma_load_3d_to_leader(smem + L::sfa_off + stage * L::kSfaBytes, &mapSfa, bar, 0, kb * C::kAtoms, m_blk,
                                keep);
          tma_load_3d_to_leader(smem + L::sfb_off + stage * L::kSfbBytes, &mapSfb, bar, 0, kb * C::kAtoms, 2 * n_blk,
                                keep);
          ++armed;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    };
    if (args.stall_after < 0) produce(std::false_type{});
    else produce(std::true_type{});
    // both CTAs' loads complete on the leader's full barriers: the leader waits for every stage
    // it armed, and neither CTA passes the final cluster barrier before that
    if (leader) wait_armed_stages(full_bar, S, armed, args.status, args.wait_ns);
  } else if (warp == 1 && leader) {
    // ------------------------------------------------------------------ MMA issuer (leader)
    uint8_t* const smem = smem_issue;  // shadows the array: addresses from the runtime base
    uint64_t* const full_bar = reinterpret_cast<uint64_t*>(smem + L::bar_off);
    uint64_t* const empty_bar = full_bar + S;
    uint64_t* const tmem_full = full_bar + 2 * S;
    uint64_t* const tmem_empty = full_bar + 2 * S + 1;
    uint64_t* const drain_bar = full_bar + 2 * S + 2;
    const bool issuer = elect_one_sync();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    const uint32_t a_s0 = smem_u32(smem + L::a_off);
    const uint32_t b_s0 = smem_u32(smem + L::b_off);
    const uint32_t sfa_s0 = smem_u32(smem + L::sfa_off);
    const uint32_t sfb_s0 = smem_u32(smem + L::sfb_off);
    const uint32_t sf_t0 = tmem_base + kAccCols;
    for (int u = first_pair; u < args.num_units && ok; u += pair_stride) {
      const int split = u / args.num_pairs;
      const int kb0 = split * args.nk / args.splits, kb1 = (split + 1) * args.nk / args.splits;
      // wait until both CTAs' epilogues have drained the accumulator of the previous tile
      if (!mbar_wait_bounded_warp(tmem_empty, acc_phase ^ 1u, abort_flag, args.status, args.wait_ns)) break;
      acc_phase ^= 1u;
      tc_fence_after();
      for (int kb = kb0; kb < kb1; ++kb) {
        // both CTAs' operands of the stage landed
        if (!mbar_wait_bounded_warp(&full_bar[stage], phase, abort_flag, args.status, args.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sfa_t = sf_t0 + stage * sf_cols<FMT>();
        const uint32_t sfb_t = sfa_t + 4 * C::kAtoms;
        const uint32_t sfa_s = sfa_s0 + stage * L::kSfaBytes;
        const uint32_t sfb_s = sfb_s0 + stage * L::kSfbBytes;
        const uint64_t adesc = smem_desc(a_s0 + stage * L::kABytes, 16, 1024, kSwizzle128B);
        const uint64_t bdesc = smem_desc(b_s0 + stage * L::kBBytes, 16, 1024, kSwizzle128B);
        if (issuer) {
          // scale atoms into the stage's TMEM slot of both CTAs (A atoms, then the B atoms of
          // the two 128-row halves); in this thread's order they land before the MMAs read them
#pragma unroll
          for (int i = 0; i < C::kAtoms; ++i)
            tc_cp_pair_32x128b_warpx4(sfa_t + 4 * i, smem_desc(sfa_s + 512 * i, 128, 128, kSwizzleNone));
#pragma unroll
          for (int i = 0; i < 2 * C::kAtoms; ++i) {
            const int at = i >> 1, h = i & 1;
            tc_cp_pair_32x128b_warpx4(sfb_t + 8 * at + 4 * h,
                                      smem_desc(sfb_s + h * L::kSfaBytes + 512 * at, 128, 128, kSwizzleNone));
          }
#pragma unroll
          for (int k = 0; k < kMmasPerStage; ++k) {
            // 32 bytes of K per MMA within the 128-byte swizzle span (descriptor start
            // addresses are in 16-byte units)
            uint32_t sfa = sfa_t, sfb = sfb_t, id = 0;
            if constexpr (FMT == BSQ_MXFP8) {
              id = k;  // one scale of 32 K per MMA: byte k of the stage's atom
            } else if constexpr (FMT == BSQ_NVFP4) {
              sfa += 4 * k;  // one atom (4 scales of 16 K) per MMA
              sfb += 8 * k;
            } else {
              sfa += 4 * (k >> 1);  // two scales of 32 K per MMA: bytes {0,1} or {2,3}
              sfb += 8 * (k >> 1);
              id = 2 * (k & 1);
            }
            tc_mma_pair<FMT>(tmem_base, adesc + 2 * k, bdesc + 2 * k, make_idesc<FMT>(id), sfa, sfb,
                             (k > 0 || kb > kb0) ? 1u : 0u);
          }
          tc_commit_pair_mc(&empty_bar[stage], 0x3);  // both CTAs' stage is free once these MMAs read it
        }
        __syncwarp();
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok && issuer) tc_commit_pair_mc(tmem_full, 0x3);  // both CTAs' accumulators complete
      __syncwarp();
    }
    // every tensor-core operation of the issuing lane must finish before TMEM is released
    if (issuer) tc_commit_pair(drain_bar);
    __syncwarp();
    mbar_wait_bounded(drain_bar, 0, nullptr, args.status, args.wait_ns);
  } else if (warp >= static_cast<uint32_t>(kFirstEpiWarp)) {
    // ------------------------------------------------------------------ epilogue (both CTAs)
    const uint32_t e = warp - kFirstEpiWarp;
    const uint32_t quad = warp & 3u;  // TMEM lane quadrant this warp may access
    const uint32_t cgrp = e >> 2;     // which kWarpCols of the tile's 256 columns
    constexpr int NB = C::kEpiBufs;
    uint8_t* stage_base = smem + L::epi_off + e * NB * L::kEpiChunkBytes;
    uint32_t nstores = 0;  // stores issued by this warp: staging buffer nstores % NB is next
    float* bias_s = reinterpret_cast<float*>(smem + L::bias_off) + e * kWarpCols;
    const uint32_t tmem_empty_leader = mapa_shared(smem_u32(tmem_empty), 0);
    float alpha = 1.0f;
    if constexpr (FMT == BSQ_NVFP4) alpha = __fmul_rn(*args.ga, *args.gb);
    // this lane's kAccRegs bias values (consecutive columns from kAccRegs lane of the warp's
    // kWarpCols, bf16 pairs) of unit u, zero past N or without bias. They are loaded at the top of
    // the unit, where their latency hides behind the wait for the unit's accumulator. Loading them
    // a unit ahead, during the store phase of the unit before, measured slower on GB300: NVFP4 fc1
    // at M = 51200 96.4 -> 100.3 us, the MXFP4 GELU-quantize fc1 188 -> 204 us.
    using BiasRegs = uint32_t[kAccRegs / 2];
    auto load_bias = [&](int u, BiasRegs& b) {
      const int pt = u % args.num_pairs;
      const int n = (pt % args.tiles_n) * BN + static_cast<int>(cgrp) * kWarpCols + kAccRegs * static_cast<int>(lane);
      const int bn = (EPI == kEpiConvT || EPI == kEpiConvTGelu) ? n % args.cv_c : n;  // ConvT: per channel
#pragma unroll
      for (int i = 0; i < kAccRegs / 2; ++i) b[i] = 0u;
      if (args.bias != nullptr && n < args.N && in_bounds(bn >= 0 && bn + kAccRegs <= args.bias_len, args.status)) {
#pragma unroll
        for (int i = 0; i < kAccRegs / 2; ++i) b[i] = reinterpret_cast<const uint32_t*>(args.bias + bn)[i];
      }
    };
    uint32_t acc_phase = 0;
    for (int u = first_pair; u < args.num_units; u += pair_stride) {
      const int split = u / args.num_pairs, pt = u - split * args.num_pairs;
      const int m_blk = 2 * (pt / args.tiles_n) + static_cast<int>(rank);
      const int n_blk = pt % args.tiles_n;
      const int n0 = n_blk * BN + static_cast<int>(cgrp) * kWarpCols;
      const int m0 = m_blk * BM + quad * 32;
      BiasRegs bias;
      load_bias(u, bias);
      __syncwarp();  // every lane is done reading the previous unit's bias
#pragma unroll
      for (int i = 0; i < kAccRegs / 2; ++i)
        *reinterpret_cast<uint64_t*>(&bias_s[kAccRegs * lane + 2 * i]) =
            f2(__uint_as_float(bias[i] << 16), __uint_as_float(bias[i] & 0xFFFF0000u));
      __syncwarp();
      if (!mbar_wait_bounded(tmem_full, acc_phase, abort_flag, args.status, args.wait_ns)) break;
      acc_phase ^= 1u;
      tc_fence_after();
      uint32_t acc[kAccRegs][32];
      const uint32_t taddr = tmem_base + ((quad * 32u) << 16) + cgrp * kWarpCols;
#pragma unroll
      for (int j = 0; j < kAccRegs; ++j) tmem_ld_32x32b_x32(taddr + 32u * j, acc[j]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(tmem_empty_leader);  // accumulator may be overwritten now

      // the epilogue values of columns c, c + 1 (c even), packed: alpha * acc + bias (and GELU)
      auto value2 = [&](int c, float& lo, float& hi) {
        const uint64_t a2 = f2(__uint_as_float(acc[c >> 5][c & 31]), __uint_as_float(acc[c >> 5][(c + 1) & 31]));
        const uint64_t b2 = *reinterpret_cast<const uint64_t*>(&bias_s[c]);
        if constexpr (FMT == BSQ_NVFP4) {
          f2_split(f2_fma(a2, f2_splat(alpha), b2), lo, hi);
        } else {
          f2_split(f2_add(a2, b2), lo, hi);
        }
        if constexpr (EPI != kEpiBf16 && EPI != kEpiConvT) gelu_erf2(lo, hi);
      };
      // quantized epilogues: all kWarpCols values first (in place), one MX block per 32 columns
      // (the MX rule: exponent of the block's largest magnitude minus that of the element format's
      // top binade), the row's kAccRegs scale bytes stored in the tiled layout's 32-bit word of
      // four blocks, or half of it (zero for the padding rows of the tile)
      constexpr bool kQuant = (EPI == kEpiGeluMxfp8 || EPI == kEpiGeluMxfp4);
      float mul[kAccRegs];
      if constexpr (kQuant) {
#pragma unroll
        for (int c = 0; c < kWarpCols; c += 2) {
          float lo, hi;
          value2(c, lo, hi);
          acc[c >> 5][c & 31] = __float_as_uint(lo);
          acc[c >> 5][(c + 1) & 31] = __float_as_uint(hi);
        }
        constexpr uint32_t kEmax = (EPI == kEpiGeluMxfp8) ? 8u : 2u;
        uint32_t sword = 0;  // the row's scale bytes, block bk in byte bk
#pragma unroll
        for (int bk = 0; bk < kAccRegs; ++bk) {
          float amax = 0.0f;
#pragma unroll
          for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(__uint_as_float(acc[bk][i])));
          const uint32_t ef = __float_as_uint(amax) >> 23;
          const uint32_t sbyte = ef > kEmax ? ef - kEmax : 0u;
          mul[bk] = __uint_as_float((254u - sbyte) << 23);  // 2^(127 - sbyte), exact
          sword |= sbyte << (8 * bk);
        }
        // the words of the padded output tiles only: with an odd number of 128-row tiles the last
        // pair's second CTA computes a tile that lies wholly past them, and a word's second half
        // may lie wholly past N (padding blocks: zero)
        const uint32_t r = static_cast<uint32_t>(m0) + lane;
        if ((n0 >> 7) < args.q_nct && (r >> 7) < (static_cast<uint32_t>(args.M) + 127u) >> 7) {
          const uint64_t off = (static_cast<uint64_t>(r >> 7) * static_cast<uint64_t>(args.q_nct) +
                                static_cast<uint64_t>(n0 >> 7)) * 512 + (r & 31u) * 16 + ((r >> 5) & 3u) * 4 +
                               ((n0 >> 5) & 3);
          const uint32_t v = r < static_cast<uint32_t>(args.M) && n0 < args.N ? sword : 0u;
          if (in_bounds(off + kAccRegs <= static_cast<uint64_t>(args.qscales_bytes), args.status)) {
            if constexpr (kAccRegs == 4) *reinterpret_cast<uint32_t*>(args.qscales + off) = v;
            else *reinterpret_cast<uint16_t*>(args.qscales + off) = static_cast<uint16_t>(v);
          }
        }
      }

      // store: chunks of 32 rows x RB bytes through the staging buffer and TMA
      constexpr int kRowBytes = (EPI == kEpiF32Partial) ? 4 * kWarpCols
                                : (EPI == kEpiGeluMxfp8) ? kWarpCols
                                : (EPI == kEpiGeluMxfp4) ? kWarpCols / 2 : 2 * kWarpCols;
      constexpr int RB = kRowBytes < 64 ? kRowBytes : 64;  // bytes of a staged row: 64 or 32
      static_assert(32 * RB <= L::kEpiChunkBytes, "staging chunk");
      const int row_units = (EPI == kEpiGeluMxfp4) ? (args.N >> 1) : args.N;  // TMA x extent of a row
#pragma unroll
      for (int j = 0; j < kRowBytes / RB; ++j) {
        constexpr bool kBf16Out = (EPI == kEpiBf16 || EPI == kEpiGeluBf16 || EPI == kEpiConvT || EPI == kEpiConvTGelu);
        int x;  // first TMA x coordinate of the chunk (bf16 elements or code bytes)
        if constexpr (kBf16Out) x = n0 + (RB / 2) * j;
        else if constexpr (EPI == kEpiF32Partial) x = n0 + (RB / 4) * j;  // fp32 elements
        else if constexpr (EPI == kEpiGeluMxfp8) x = n0 + RB * j;
        else x = (n0 >> 1) + RB * j;
        if (x >= row_units || m0 >= args.M) break;  // nothing of this chunk is stored (warp-uniform)
        uint8_t* stage_buf = stage_base + (nstores % NB) * L::kEpiChunkBytes;
        uint32_t packed[RB / 4];
#pragma unroll
        for (int c = 0; c < RB / 4; ++c) {
          if constexpr (kBf16Out) {
            const int col = (RB / 2) * j + 2 * c;  // two bf16 per word
            float lo, hi;
            value2(col, lo, hi);
            __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
            packed[c] = *reinterpret_cast<uint32_t*>(&p);
          } else if constexpr (EPI == kEpiF32Partial) {
            const int col = (RB / 4) * j + c;  // the raw fp32 accumulator
            packed[c] = acc[col >> 5][col & 31];
          } else if constexpr (EPI == kEpiGeluMxfp8) {
            const int col = RB * j + 4 * c;  // four E4M3 codes per word, one block
            const float m = mul[col >> 5];
            packed[c] = cvt_e4m3x4(__uint_as_float(acc[col >> 5][col & 31]) * m,
                                   __uint_as_float(acc[col >> 5][(col + 1) & 31]) * m,
                                   __uint_as_float(acc[col >> 5][(col + 2) & 31]) * m,
                                   __uint_as_float(acc[col >> 5][(col + 3) & 31]) * m);
          } else {
            const int col = 2 * RB * j + 8 * c;  // eight e2m1 codes per word, one block
            const float m = mul[col >> 5];
            float y[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = __uint_as_float(acc[col >> 5][(col + i) & 31]) * m;
            packed[c] = cvt_e2m1x8(y);
          }
        }
        // the chunk's values are computed above while the store that last used this buffer may
        // still be reading it; wait for that read only now
        if (lane == 0) bulk_wait_group_read<NB - 1>();
        __syncwarp();
        // row `lane` of the 32 x RB chunk in 16-byte pieces; the TMA swizzle (64B or 32B mode)
        // XORs the piece index with address bits 7.. so that a quarter-warp hits distinct banks
#pragma unroll
        for (int q = 0; q < RB / 16; ++q) {
          const uint32_t sw = (RB == 64) ? ((lane >> 1) & 3u) : ((lane >> 2) & 1u);
          const uint32_t phys = (static_cast<uint32_t>(q) ^ sw) << 4;
          *reinterpret_cast<uint4*>(stage_buf + lane * RB + phys) =
              make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if constexpr (EPI == kEpiConvT || EPI == kEpiConvTGelu) {
            // the chunk's 32 output rows are tokens m0.. (whole image rows when W divides 32, a
            // 32-token piece of one image row when 32 divides W); its columns one tap (dy, dx)
            const int tap = x / args.cv_c, co = x - tap * args.cv_c;
            const int bh = m0 / args.cv_w, w0 = m0 - bh * args.cv_w;
            tma_store_5d(&mapOut, stage_buf, co, tap & 1, w0, tap >> 1, bh);
          } else if constexpr (EPI == kEpiF32Partial) {
            tma_store_3d(&mapOut, stage_buf, x, m0, split);  // slice `split` of the workspace
          } else {
            tma_store_2d(&mapOut, stage_buf, x, m0);
          }
          bulk_commit_group();
        }
        ++nstores;
      }
    }
    if (lane == 0) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while its peer may still touch its barriers or TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace

// ---------------------------------------------------------------------------- host side
// Tensor-map encoding, shared with the other translation units.
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

namespace {

// View of a tiled scale buffer as (128 words of a 512-byte atom, atoms of a row tile, row
// tiles); a box of (128, atoms, tiles) brings that many whole atoms in one copy.
bool make_map_scales(CUtensorMap* map, const void* base, uint64_t atoms_per_tile, uint64_t row_tiles,
                     uint32_t box_atoms, uint32_t box_tiles) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {128, atoms_per_tile, row_tiles};
  const cuuint64_t strides[2] = {512, atoms_per_tile * 512};
  const cuuint32_t box[3] = {128, box_atoms, box_tiles};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


// Launch as (2,1,1) clusters; with programmatic stream serialization the kernel may be
// launched while the previous kernel in the stream finishes (it waits for it before touching
// memory). `attr` holds two entries.
cudaLaunchConfig_t pair_launch_config(cudaLaunchAttribute* attr, int clusters, int threads, int smem,
                                      cudaStream_t stream) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

// NHWC output of a kernel-2 stride-2 transposed convolution as a 5-D tensor (channel co, dx, w,
// dy, b * H + h), one box = one epilogue chunk: EC channels of one tap for 32 tokens.
bool make_map_convt_out(CUtensorMap* map, void* out, int64_t cout, int64_t W, int64_t BH, uint32_t ec,
                        CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(cout), 2, static_cast<cuuint64_t>(W), 2,
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[4] = {static_cast<cuuint64_t>(cout) * 2, static_cast<cuuint64_t>(cout) * 4,
                                 static_cast<cuuint64_t>(W * cout) * 4, static_cast<cuuint64_t>(W * cout) * 8};
  const uint32_t wb = static_cast<uint32_t>(std::min<int64_t>(W, 32));
  const cuuint32_t box[5] = {ec, 1, wb, 1, 32 / wb};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, out, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The split-K workspace: `splits` slices of M x N fp32, row-major, as a 3-D tensor (n, m, slice);
// one box = one epilogue chunk of 16 columns x 32 rows (64-byte rows, 64-byte swizzle).
bool make_map_partial(CUtensorMap* map, void* ws, int64_t M, int64_t N, int splits) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(splits)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(N) * 4, static_cast<cuuint64_t>(M * N) * 4};
  const cuuint32_t box[3] = {16, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ws, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT, int EPI>
int run_gemm(const void* A, const void* A_scales, const void* B, const void* B_scales, const void* bias, void* out,
             void* out_scales, int64_t M, int64_t N, int64_t K, int64_t cv_w, int splits, cudaStream_t stream,
             const DeviceInfo& dev) {
  // per device: the shared-memory opt-in and the number of co-resident clusters (0 = unusable)
  static PerDevice<int> setup;
  const int max_clusters = setup.run(dev.device, [] {
    if (cudaFuncSetAttribute(gemm_kernel<FMT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<FMT, EPI>::alloc) !=
        cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cudaLaunchAttribute at[2];
    cudaLaunchConfig_t cfg = pair_launch_config(at, 1, Epi<EPI>::kThreads, Smem<FMT, EPI>::alloc, nullptr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_kernel<FMT, EPI>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return n;
  });
  if (max_clusters < 1) return BSQ_ERR_LAUNCH;

  const uint64_t kbytes = (FMT == BSQ_MXFP8) ? static_cast<uint64_t>(K) : static_cast<uint64_t>(K) / 2;
  CUtensorMap mA, mB, mSfa, mSfb, mOut;
  constexpr int EC = Cfg<FMT>::kEpiCols;
  const CUtensorMapSwizzle osw = EC == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  bool ok_out;
  if constexpr (EPI == kEpiF32Partial) {
    static_assert(EC == 32, "fp32 partial chunks are 16 columns = 64-byte rows, the staging of 32 bf16 columns");
    ok_out = make_map_partial(&mOut, out, M, N, splits);
  } else if constexpr (EPI == kEpiConvT || EPI == kEpiConvTGelu) {
    ok_out = make_map_convt_out(&mOut, out, N / 4, cv_w, M / cv_w, EC, osw);
  } else if constexpr (EPI == kEpiBf16 || EPI == kEpiGeluBf16) {
    ok_out = make_map_2d(&mOut, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out, N, M, static_cast<uint64_t>(N) * 2, EC, 32, osw);
  } else {
    // code bytes of an output row: N (E4M3) or N / 2 (e2m1); staged rows of 64 bytes, or 32 (e2m1 codes of a
    // warp's 64 columns)
    const uint64_t rb = (EPI == kEpiGeluMxfp8) ? static_cast<uint64_t>(N) : static_cast<uint64_t>(N) / 2;
    ok_out = (EPI == kEpiGeluMxfp8 || Epi<EPI>::kWarpCols / 2 >= 64)
                 ? make_map_2d(&mOut, CU_TENSOR_MAP_DATA_TYPE_UINT8, out, rb, M, rb, 2 * EC, 32, osw)
                 : make_map_2d(&mOut, CU_TENSOR_MAP_DATA_TYPE_UINT8, out, rb, M, rb, 32, 32, CU_TENSOR_MAP_SWIZZLE_32B);
  }
  if (!ok_out ||
      !make_map_2d(&mA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, kbytes, M, kbytes, kChunkBytes, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&mB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, kbytes, N, kbytes, kChunkBytes, BNH, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_scales(&mSfa, A_scales, static_cast<uint64_t>(ceil_div(K / block_size(FMT), 4)),
                       static_cast<uint64_t>(ceil_div(M, 128)), Cfg<FMT>::kAtoms, 1) ||
      !make_map_scales(&mSfb, B_scales, static_cast<uint64_t>(ceil_div(K / block_size(FMT), 4)),
                       static_cast<uint64_t>(ceil_div(N, 128)), Cfg<FMT>::kAtoms, 2))
    return BSQ_ERR_LAUNCH;

  GemmArgs a{};
  a.bias = static_cast<const uint16_t*>(bias);
  a.qscales = static_cast<uint8_t*>(out_scales);
  a.q_nct = static_cast<int>(ceil_div(N / 32, 4));
  a.qscales_bytes = ceil_div(M, 128) * a.q_nct * 512;
  a.bias_len = static_cast<int>((EPI == kEpiConvT || EPI == kEpiConvTGelu) ? N / 4 : N);
  a.ga = reinterpret_cast<const float*>(static_cast<const uint8_t*>(A_scales) + scales_body_bytes(FMT, M, K));
  a.gb = reinterpret_cast<const float*>(static_cast<const uint8_t*>(B_scales) + scales_body_bytes(FMT, N, K));
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.tiles_n = static_cast<int>(ceil_div(N, BN));
  a.num_pairs = static_cast<int>(ceil_div(ceil_div(M, BM), 2)) * a.tiles_n;
  a.nk = static_cast<int>(kbytes / kChunkBytes);
  a.cv_c = static_cast<int>(N / 4);
  a.cv_w = static_cast<int>(cv_w);
  a.splits = (EPI == kEpiF32Partial) ? splits : 1;
  a.num_units = a.num_pairs * a.splits;
  a.status = dev.status;
  const StallInjection inj = take_stall(BSQ_KERNEL_GEMM);
  a.stall_after = inj.after;
  a.wait_ns = inj.limit_ns;
  const int clusters = std::min(a.num_units, std::min(max_clusters, dev.num_sms / 2));

  cudaLaunchAttribute at[2];
  cudaLaunchConfig_t cfg = pair_launch_config(at, clusters, Epi<EPI>::kThreads, Smem<FMT, EPI>::alloc, stream);
  if (cudaLaunchKernelEx(&cfg, gemm_kernel<FMT, EPI>, mA, mB, mSfa, mSfb, mOut, a) != cudaSuccess)
    return BSQ_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? BSQ_OK : BSQ_ERR_LAUNCH;
}

// out[m, n] = bf16(fmaf(sum_s ws[s][m][n], alpha, bias[n])): the split-K partial sums added in
// slice order, then the GEMM's own epilogue arithmetic (alpha = g_A g_B for NVFP4; for MX alpha
// is 1 and the fma is the plain add acc + bias). Eight consecutive columns per thread (N % 8 == 0).
__global__ void __launch_bounds__(256)
    splitk_finalize_kernel(const float* ws, int splits, int64_t mn, int N, const uint16_t* bias, const float* ga,
                           const float* gb, uint16_t* out) {
  grid_dependency_wait();  // the partial sums come from the previous kernel
  const float alpha = ga != nullptr ? __fmul_rn(*ga, *gb) : 1.0f;
  const int64_t n8 = mn / 8;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = i * 8;
    float v[8];
    {
      const float4* p = reinterpret_cast<const float4*>(ws + e);
      const float4 a = p[0], b = p[1];
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
    for (int sl = 1; sl < splits; ++sl) {
      const float4* p = reinterpret_cast<const float4*>(ws + sl * mn + e);
      const float4 a = p[0], b = p[1];
      const float t[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = __fadd_rn(v[k], t[k]);
    }
    const int n = static_cast<int>(e % N);
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float b0 = bias != nullptr ? __uint_as_float(static_cast<uint32_t>(bias[n + 2 * k]) << 16) : 0.0f;
      const float b1 = bias != nullptr ? __uint_as_float(static_cast<uint32_t>(bias[n + 2 * k + 1]) << 16) : 0.0f;
      __nv_bfloat162 h = __floats2bfloat162_rn(__fmaf_rn(v[2 * k], alpha, b0), __fmaf_rn(v[2 * k + 1], alpha, b1));
      w[k] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(out + e) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  launch_dependents();
}

template <int FMT>
int run_gemm_epi(int epi, const void* A, const void* A_scales, const void* B, const void* B_scales, const void* bias,
                 void* out, void* out_scales, int64_t M, int64_t N, int64_t K, int64_t cv_w, int splits,
                 cudaStream_t stream, const DeviceInfo& dev) {
#define BSQ_RUN(E) run_gemm<FMT, E>(A, A_scales, B, B_scales, bias, out, out_scales, M, N, K, cv_w, splits, stream, dev)
  switch (epi) {
    case kEpiBf16: return BSQ_RUN(kEpiBf16);
    case kEpiGeluBf16: return BSQ_RUN(kEpiGeluBf16);
    case kEpiGeluMxfp8: return BSQ_RUN(kEpiGeluMxfp8);
    case kEpiGeluMxfp4: return BSQ_RUN(kEpiGeluMxfp4);
    case kEpiConvT: return BSQ_RUN(kEpiConvT);
    case kEpiConvTGelu: return BSQ_RUN(kEpiConvTGelu);
    case kEpiF32Partial: return BSQ_RUN(kEpiF32Partial);
    default: return BSQ_ERR_ARG;
  }
#undef BSQ_RUN
}

}  // namespace

int launch_gemm(int fmt, int epi, const void* A, const void* A_scales, const void* B, const void* B_scales,
                const void* bias, void* out, void* out_scales, int64_t M, int64_t N, int64_t K, cudaStream_t stream,
                const DeviceInfo& dev, int64_t convt_w, int splits) {
  switch (fmt) {
    case BSQ_MXFP8:
      return run_gemm_epi<BSQ_MXFP8>(epi, A, A_scales, B, B_scales, bias, out, out_scales, M, N, K, convt_w, splits,
                                     stream, dev);
    case BSQ_NVFP4:
      return run_gemm_epi<BSQ_NVFP4>(epi, A, A_scales, B, B_scales, bias, out, out_scales, M, N, K, convt_w, splits,
                                     stream, dev);
    case BSQ_MXFP4:
      return run_gemm_epi<BSQ_MXFP4>(epi, A, A_scales, B, B_scales, bias, out, out_scales, M, N, K, convt_w, splits,
                                     stream, dev);
    default:
      return BSQ_ERR_ARG;
  }
}

int launch_splitk_finalize(int fmt, const float* ws, int splits, int64_t M, int64_t N, int64_t K, const void* bias,
                           const void* A_scales, const void* B_scales, void* out, cudaStream_t stream,
                           const DeviceInfo& dev) {
  const float* ga = nullptr;
  const float* gb = nullptr;
  if (fmt == BSQ_NVFP4) {
    ga = reinterpret_cast<const float*>(static_cast<const uint8_t*>(A_scales) + scales_body_bytes(fmt, M, K));
    gb = reinterpret_cast<const float*>(static_cast<const uint8_t*>(B_scales) + scales_body_bytes(fmt, N, K));
  }
  const int64_t n8 = M * N / 8;
  const int64_t blocks = std::min<int64_t>(ceil_div(n8, 256), static_cast<int64_t>(dev.num_sms) * 8);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(std::max<int64_t>(blocks, 1)));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, splitk_finalize_kernel, ws, splits, M * N, static_cast<int>(N),
                         static_cast<const uint16_t*>(bias), ga, gb, static_cast<uint16_t*>(out)) != cudaSuccess)
    return BSQ_ERR_LAUNCH;
  return cudaGetLastError() == cudaSuccess ? BSQ_OK : BSQ_ERR_LAUNCH;
}

}  // namespace bsq
