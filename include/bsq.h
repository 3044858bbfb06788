/*
 * bsq.h -- C ABI of libbsq.so: block-scaled low-precision quantization (MXFP8, NVFP4,
 * MXFP4) and the block-scaled GEMM with a fused bias + bf16 epilogue, for GB300 (sm_103a).
 *
 * The method: the linear layers of a ViT block (qkv, proj, fc1, fc2) run as block-scaled
 * low-precision GEMMs ("lightly-train - DINOv3 + EoMT on RTX 5090" README, section 2 number
 * formats table; sections 4.3 and 5.3 name the quantized GEMMs). A layer is two steps:
 *   1. per-block quantization of a bf16 (or fp32) matrix along its K dimension;
 *   2. out = bf16(alpha * sum_k Ahat[m,k] * Bhat[n,k] + bias[n]), fp32 accumulation.
 *
 * Conventions shared by every entry point
 *   - All buffer pointers are DEVICE pointers, 16-byte aligned, allocated by the caller;
 *     the library allocates no memory and keeps no per-call state. Its only state is one
 *     status word per device (see bsq_get_device_status) and a thread-local last error.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream) and
 *     returns without synchronising, except bsq_get_device_status.
 *   - Matrices are row-major. Quantized operands are "K-major": element (r, k) of a
 *     rows x cols matrix is at r * cols + k (the "TN" GEMM of section 5.5 of the README).
 *   - Return value 0 = enqueued; a negative BSQ_ERR_* = nothing was enqueued (argument
 *     errors) or the launch failed (BSQ_ERR_LAUNCH). Device-side failures (a bounded wait
 *     that gave up) are reported later through bsq_get_device_status.
 *   - Requires a compute capability 10.3 device (GB300); otherwise BSQ_ERR_ARCH.
 */
#ifndef BSQ_H
#define BSQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* bsq_stream_t; /* identical to cudaStream_t */

/* Formats (README section 2, number-format table):
 *   BSQ_MXFP8  E4M3 elements, one UE8M0 (power-of-two) scale per 1x32 block, 8.25 bits/value.
 *   BSQ_NVFP4  e2m1 elements (2 per byte), one E4M3 scale per 1x16 block and one fp32
 *              per-tensor scale g, 4.5 bits/value.
 *   BSQ_MXFP4  e2m1 elements, one UE8M0 scale per 1x32 block, 4.25 bits/value. */
typedef enum { BSQ_MXFP8 = 1, BSQ_NVFP4 = 2, BSQ_MXFP4 = 3 } bsq_format;

/* Flags OR-ed into bsq_quantize's first argument. */
#define BSQ_FMT_MASK 0xFF
#define BSQ_FLAG_SRC_F32 0x100      /* src holds fp32 values; default: bf16 */
#define BSQ_FLAG_GLOBAL_GIVEN 0x200 /* NVFP4: read g from *global_scale instead of computing it
                                       (a static or delayed per-tensor scale, README sections
                                       4.3 and 5.5) */
#define BSQ_FLAG_STOCHASTIC 0x400   /* bsq_quantize_dual: stochastic rounding of the elements */

/* Status codes. */
#define BSQ_OK 0
#define BSQ_ERR_ARG -1     /* null pointer, non-positive size, unknown format or flag */
#define BSQ_ERR_SHAPE -2   /* a size the format or the GEMM cannot tile (see each call) */
#define BSQ_ERR_ALIGN -3   /* a pointer is not 16-byte aligned */
#define BSQ_ERR_ARCH -4    /* no CUDA device, or not compute capability 10.3 */
#define BSQ_ERR_LAUNCH -5  /* the CUDA runtime reported an error at launch */
#define BSQ_ERR_TIMEOUT -6 /* a kernel's bounded wait gave up (device status only) */
#define BSQ_ERR_DEVICE_CHECK -7 /* checked build (libbsq_checked.so) only: a kernel's index check
                                   failed and the access was skipped (device status only) */

/*
 * bsq_codes_bytes: size of the element-code buffer of a rows x cols matrix.
 *   MXFP8: rows * cols bytes (one E4M3 code per byte).
 *   NVFP4, MXFP4: rows * cols / 2 bytes; element 2j in the low nibble of byte j, 2j+1 in
 *   the high nibble. Returns 0 for invalid arguments.
 * Source: the element widths of the README's section 2 number-format table (8-bit E4M3,
 * 4-bit e2m1). The nibble order is a convention: the pages are silent on it.
 */
size_t bsq_codes_bytes(int fmt, int64_t rows, int64_t cols);

/*
 * bsq_scales_bytes: size of the scale buffer of a rows x cols matrix.
 * Source: the block sizes and scale types of the README's section 2 number-format table
 * (one 8-bit scale per 1x32 block for MX, per 1x16 block for NVFP4). The tiled layout below
 * is a convention; the pages are silent on how scales are laid out in memory.
 * Block scales are stored in tiles of 128 rows x 4 scale columns (512 bytes): the scale of
 * row r and block column c lives in tile (r / 128) * ceil(nsc / 4) + c / 4 at byte
 * (r % 32) * 16 + ((r / 32) % 4) * 4 + c % 4, nsc = cols / block size. Rows are padded to
 * 128 and scale columns to 4; padding bytes are written as 0. This is the layout the
 * tensor cores' scale-factor copy consumes, so the GEMM reads it without reshuffling.
 * NVFP4 appends a 16-byte tail {g, amax, 0, 0} (fp32): the per-tensor scale used and the
 * amax of the quantized tensor (the source of a delayed scale for the next call).
 * Returns 0 for invalid arguments.
 */
size_t bsq_scales_bytes(int fmt, int64_t rows, int64_t cols);

/*
 * bsq_quantize: quantize a rows x cols matrix along cols (K) in 1x32 (MX) or 1x16 (NVFP4)
 * blocks.
 *   fmt_flags    bsq_format | BSQ_FLAG_* bits.
 *   src          rows x cols bf16 (default) or fp32 (BSQ_FLAG_SRC_F32) values, finite.
 *   codes        bsq_codes_bytes(fmt, rows, cols) bytes, written.
 *   scales       bsq_scales_bytes(fmt, rows, cols) bytes, written (including padding).
 *   global_scale NVFP4 only, one fp32 in device memory. Without BSQ_FLAG_GLOBAL_GIVEN it
 *                receives g = amax(|src|) / 2688 (may be NULL: g is also in the scale tail);
 *                with the flag it is read as g (must not be NULL). Ignored for MX formats.
 * Rules (README section 2; rounding to nearest even with saturation at the largest finite
 * value, 448 for E4M3 and 6 for e2m1):
 *   MX     per block e = floor(log2(amax)) - emax (emax 8 for E4M3, 2 for e2m1), clamped to
 *          [-127, 127], amax = 0 -> -127; scale byte e + 127; code = RNE_sat(x * 2^-e).
 *   NVFP4  s = E4M3 RNE_sat(bamax / (6 g)); code = e2m1 RNE_sat(x / (s g)), each step one
 *          IEEE fp32 operation; s = 0 gives zero codes carrying the sign of x.
 * Shapes: cols % 32 == 0 (MX) or cols % 16 == 0 (NVFP4), rows and cols below 2^31, else
 * BSQ_ERR_SHAPE; any rows >= 1.
 * Codes and scales are bit-exact functions of the input (no dependence on launch shape).
 */
int bsq_quantize(int fmt_flags, const void* src, int64_t rows, int64_t cols, void* codes, void* scales,
                 float* global_scale, bsq_stream_t stream);

/*
 * bsq_layernorm_quantize: the LayerNorm + quantization kernel of the README's MXFP8 stack
 * ("lightly-train - DINOv3 + EoMT on RTX 5090" README, section 4.3: LN and quantization merged
 * into one kernel). Per row r of a rows x cols matrix:
 *   y[r, c] = (x[r, c] - mean_r) / sqrt(var_r + eps) * gamma[c] + beta[c]
 * with mean_r and the biased variance var_r over the row, in fp32, then y (kept in fp32)
 * quantized along the row as bsq_quantize does: codes and tiled scales of an MX format.
 *   fmt_flags   BSQ_MXFP8 or BSQ_MXFP4, optionally | BSQ_FLAG_SRC_F32
 *   gamma_bf16, beta_bf16   cols bf16 values each, 16-byte aligned
 *   eps         >= 0
 * Codes and scales are the MX quantization of the kernel's fp32 y; a code differs from that of
 * the exact value only where the exact value lies within the fp32 rounding of the statistics
 * and the affine step of a rounding boundary.
 * Work mapping: bf16 rows of at most 1024 elements run one row per warp with the row in
 * registers; other rows are staged through shared memory. Both give the same bytes for the same
 * values.
 * Shapes: as bsq_quantize for MX, and a row of at most 16384 bytes (cols <= 8192 bf16 or 4096
 * fp32), else BSQ_ERR_SHAPE. Errors: BSQ_ERR_ARG for another format or flag, NULL gamma /
 * beta or a negative or non-finite eps; otherwise as bsq_quantize.
 */
int bsq_layernorm_quantize(int fmt_flags, const void* src, const void* gamma_bf16, const void* beta_bf16, float eps,
                           int64_t rows, int64_t cols, void* codes, void* scales, bsq_stream_t stream);

#define BSQ_MAX_BATCH 8
typedef struct {
  const void* src;     /* rows x cols bf16 or fp32 (per fmt_flags) */
  int64_t rows, cols;
  void* codes;         /* bsq_codes_bytes(fmt, rows, cols) bytes, written */
  void* scales;        /* bsq_scales_bytes(fmt, rows, cols) bytes, written */
  float* global_scale; /* NVFP4 only, as bsq_quantize's global_scale; NULL otherwise */
} bsq_quant_item;

/*
 * bsq_quantize_batch: bsq_quantize applied to `count` matrices (1 <= count <= BSQ_MAX_BATCH)
 * in one kernel launch, e.g. a layer's activations and weights together. Every item is
 * validated as in bsq_quantize (its own rows, cols, buffers; global_scale as bsq_quantize's
 * argument) and the whole batch shares fmt_flags (one format, one source type, one
 * NVFP4 scale mode). Results are identical, byte for byte, to `count` bsq_quantize calls.
 * `items` is a host array read during the call only. The batching is an engineering entry
 * point (fewer launches for small matrices); the method itself has no counterpart.
 * Errors: BSQ_ERR_ARG if count is out of range or items is NULL, otherwise the first error
 * any item would give bsq_quantize; nothing is enqueued on an argument error.
 */
int bsq_quantize_batch(int fmt_flags, int count, const bsq_quant_item* items, bsq_stream_t stream);

/*
 * bsq_quantize_dual: dual-layout quantization for the backward GEMMs ("lightly-train - DINOv3 +
 * EoMT on RTX 5090" README, section 4.3, the quantized training stacks: dgrad contracts dY
 * over N and wgrad over M, so dY is needed quantized along both of its dimensions, W along N
 * and X along M; the README's fused FP4 quantizer writes both layouts from one read). From one
 * rows x cols matrix X, in one pass over it:
 *   row_codes, row_scales  the operand bsq_quantize(fmt, X, rows, cols) writes (blocks along
 *                          cols), sized bsq_codes_bytes / bsq_scales_bytes(fmt, rows, cols);
 *   col_codes, col_scales  the operand of X^T (cols x rows, blocks along rows), as
 *                          bsq_quantize(fmt, X^T, cols, rows) would write it, sized
 *                          bsq_codes_bytes / bsq_scales_bytes(fmt, cols, rows).
 * All four are written, scale padding included.
 *   fmt_flags     BSQ_MXFP8, BSQ_MXFP4 or BSQ_NVFP4, | BSQ_FLAG_SRC_F32 (fp32 source, default
 *                 bf16), | BSQ_FLAG_STOCHASTIC, | BSQ_FLAG_GLOBAL_GIVEN (NVFP4 only).
 *   global_scale  NVFP4: one fp32 in device memory, as bsq_quantize's argument (receives the
 *                 computed g, may be NULL; or, with BSQ_FLAG_GLOBAL_GIVEN, supplies g). The one
 *                 g serves both layouts; both scale tails hold {g, amax of X}. Ignored for MX.
 * Block scales follow the rules of bsq_quantize. Without BSQ_FLAG_STOCHASTIC the elements
 * round to nearest even (seed ignored); both layouts are then byte-identical to the two
 * bsq_quantize calls (NVFP4 with the same g). With it (the gradient rounding of quantized
 * training), for v = the element's quotient (MX: x / scale, exact; NVFP4: fp32(x / fp32(s g))):
 * q = |v| / spacing, the spacing of the element format at |v|'s binade (its subnormal step
 * below the smallest normal); |code| = floor(q) + (frac(q) > u), saturating at the largest
 * finite value (448, 6); u = h * 2^-16 with h the 16-bit half i mod 2 (low half first) of word
 * (i mod 8) / 2 of Philox4x32-10 (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3",
 * SC'11) at counter {floor(i/8) low 32 bits, high 32 bits, layout, 0} and key {seed low 32 bits,
 * high 32 bits}; i = r * cols + c in the row layout (layout 0), c * rows + r in the column
 * layout (layout 1). E[code value] = v below saturation wherever frac(q) has at most 16 bits
 * (every bf16 X whose quotient lies in the format's normal range), otherwise within 2^-16 of a
 * spacing; the codes are a function of (X, seed) alone. An NVFP4 block whose
 * scale is 0 gives signed zero codes either way.
 * Shapes: rows % 32 == 0 and cols % 32 == 0, both below 2^31, else BSQ_ERR_SHAPE.
 * Errors: BSQ_ERR_ARG for an unknown format or flag, BSQ_FLAG_GLOBAL_GIVEN without NVFP4 or
 * without global_scale, a NULL buffer or a non-positive size; BSQ_ERR_ALIGN for a buffer not
 * 16-byte aligned or a global_scale not 4-byte aligned.
 */
int bsq_quantize_dual(int fmt_flags, const void* src, int64_t rows, int64_t cols, uint64_t seed, void* row_codes,
                      void* row_scales, void* col_codes, void* col_scales, float* global_scale, bsq_stream_t stream);

/*
 * bsq_delayed_global_scale: the delayed NVFP4 per-tensor scale of quantized training
 * ("lightly-train - DINOv3 + EoMT on RTX 5090" README, section 5.5: the amax found while a
 * tensor is quantized in one step, times a headroom factor, is the next step's scale, so no
 * step spends an extra pass over the tensor on its amax; the README's dY study settles on a
 * headroom of 32). Enqueues one thread computing
 *   *g_out = fp32(fp32(amax * headroom) / 2688)
 * with amax the tail word of prev_scales, an NVFP4 scale buffer of a rows x cols matrix
 * written by bsq_quantize / bsq_quantize_batch / bsq_quantize_dual (either layout's buffer:
 * both tails hold the same amax). Pass g_out to the next quantization of the tensor with
 * BSQ_FLAG_GLOBAL_GIVEN; that call records the new amax in its own tail. Reading the tail and
 * writing g_out are ordered on `stream` only, with no host synchronisation.
 *   prev_scales  bsq_scales_bytes(BSQ_NVFP4, rows, cols) bytes, 16-byte aligned
 *   headroom     finite, > 0
 *   g_out        one fp32 in device memory, 4-byte aligned
 * Errors: BSQ_ERR_ARG (NULL pointer, non-positive size, bad headroom), BSQ_ERR_SHAPE (cols % 16,
 * sizes >= 2^31), BSQ_ERR_ALIGN.
 */
int bsq_delayed_global_scale(const void* prev_scales, int64_t rows, int64_t cols, float headroom, float* g_out,
                             bsq_stream_t stream);

/*
 * bsq_gemm: out[m, n] = bf16_rn(alpha * sum_k Ahat[m,k] * Bhat[n,k] + bias[n]).
 * Source: "lightly-train - DINOv3 + EoMT on RTX 5090" README, section 2 (the block-scaled
 * MXFP8 / NVFP4 / MXFP4 GEMM formats and their tensor-core rates) and section 4.3 (qkv, proj,
 * fc1, fc2 of every block run as these GEMMs, bias fused into the epilogue). Ahat, Bhat are the
 * decoded operands: code value times its block scale (times g for NVFP4, folded into alpha).
 *   A, A_scales  M x K operand as written by bsq_quantize(fmt, ..., M, K, ...).
 *   B, B_scales  N x K operand (the nn.Linear weight layout) from bsq_quantize(fmt, ..., N, K, ...).
 *   bias_bf16    N bf16 values, or NULL for no bias.
 *   out_bf16     M x N bf16, row-major, written.
 *   alpha        1 for MX formats; g_A * g_B for NVFP4, read on the device from the two
 *                scale tails (no host synchronisation).
 * Products are accumulated in fp32 in the tensor cores (tcgen05 block-scaled MMA).
 * Shapes: K % 128 == 0 (MXFP8) or K % 256 == 0 (NVFP4, MXFP4); N % 8 == 0; M >= 1 (rows
 * past M are never written). Otherwise BSQ_ERR_SHAPE.
 */
int bsq_gemm(int fmt, const void* A, const void* A_scales, const void* B, const void* B_scales,
             const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K, bsq_stream_t stream);

/*
 * bsq_gemm_splitk: bsq_gemm's result computed with the K dimension cut into `splits` equal
 * ranges of K stages (128 K for MXFP8, 256 for NVFP4 / MXFP4), each (output tile, range) pair
 * one unit of work, for shapes with fewer 256 x 256 output tiles than the GPU has SM pairs and
 * a long K: the weight gradient dW = dY^T X of a linear layer ("lightly-train - DINOv3 + EoMT
 * on RTX 5090" README, section 4.3: the training stacks' wgrad GEMM; M, N the weight's shape, K
 * the token count) has 36 tiles for 76 SM pairs at ViT-B/16 fc1. The method has no split-K of
 * its own: this is an engineering entry point. Each unit stores its raw fp32 sum into slice r
 * of `workspace`; a second kernel adds the slices in order (deterministic) and applies alpha,
 * the bias and the bf16 rounding as bsq_gemm does. The fp32 sum therefore rounds in a different
 * order than bsq_gemm's (within the same tolerance).
 *   splits           1..8 and at most the number of K stages; 1 is bsq_gemm itself
 *   workspace        splits * M * N fp32 in device memory, 16-byte aligned, owned by the caller;
 *                    overwritten, no initial contents needed; unused when splits == 1
 *   workspace_bytes  its size, at least splits * M * N * 4 (else BSQ_ERR_ARG)
 * Other arguments, shapes and errors as bsq_gemm; two launches on `stream`.
 */
int bsq_gemm_splitk(int fmt, const void* A, const void* A_scales, const void* B, const void* B_scales,
                    const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K, int splits,
                    void* workspace, size_t workspace_bytes, bsq_stream_t stream);

/*
 * bsq_gemm_splitk_splits: the number of K ranges bsq_gemm_splitk should use on the current
 * device for an M x N x K product: floor(SM pairs / output tiles of 256 x 256), at most 8 and at
 * most K stages / 8 (each range keeps at least 8 stages of the operand pipeline), at least 1 --
 * 2 for ViT-B/16 fc1's weight gradient (36 tiles, 76 SM pairs), 1 for every forward GEMM of the
 * ViT shapes. Returns the count, or a negative error (BSQ_ERR_ARG for an unknown format or a
 * non-positive size, BSQ_ERR_ARCH without a usable device).
 */
int bsq_gemm_splitk_splits(int fmt, int64_t M, int64_t N, int64_t K);

/*
 * bsq_gemm_splitk_scratch: bsq_gemm_splitk with the workspace taken from a fixed 64 MiB device
 * array inside the library instead of a caller buffer, so that a call allocates nothing. The
 * pages describe no counterpart: an engineering entry point.
 *   - The array is placed with the library's device module, once per device; its address is
 *     looked up once per device. No call allocates or frees memory.
 *   - Limit: splits * M * N * 4 bytes <= 64 MiB; a larger request fails with BSQ_ERR_ARG, as
 *     bsq_gemm_splitk does with too small a workspace (splits == 1 needs none).
 *   - Nothing needs to start at zero: each call overwrites the part of the array it uses before
 *     reading it.
 *   - The array is shared by every caller in the process on that device: calls that can overlap
 *     in time (on different streams, or from different host threads) race on it; the caller
 *     orders them.
 * Other arguments, results and errors as bsq_gemm_splitk.
 */
int bsq_gemm_splitk_scratch(int fmt, const void* A, const void* A_scales, const void* B, const void* B_scales,
                            const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K, int splits,
                            bsq_stream_t stream);

/*
 * bsq_gemm_gelu: as bsq_gemm with out = bf16_rn(GELU(v)), v = alpha * sum_k Ahat Bhat + bias
 * in fp32, GELU the erf form 0.5 v (1 + erf(v / sqrt 2)) (the "fc1 + GELU" epilogue of every
 * stack in the "lightly-train - DINOv3 + EoMT on RTX 5090" README, section 4.3), evaluated in
 * fp32 with erfc from Abramowitz & Stegun formula 7.1.26: |error| <= 4e-7 |v| + 2^-20 |GELU|.
 * Arguments, shapes and errors as bsq_gemm.
 */
int bsq_gemm_gelu(int fmt, const void* A, const void* A_scales, const void* B, const void* B_scales,
                  const void* bias_bf16, void* out_bf16, int64_t M, int64_t N, int64_t K, bsq_stream_t stream);

/*
 * bsq_gemm_gelu_quantize: the producer-fused fc1 of the README's MXFP8 stack (section 4.3: the
 * fc1 epilogue quantizes the GELU output straight into fc2's operand). y = GELU(v) as in
 * bsq_gemm_gelu, kept in fp32, then quantized along each output row with the MX rule of
 * bsq_quantize into out_fmt (BSQ_MXFP8 or BSQ_MXFP4):
 *   out_codes   bsq_codes_bytes(out_fmt, M, N) bytes, written;
 *   out_scales  bsq_scales_bytes(out_fmt, M, N) bytes (tiled layout, padding zero), written.
 * The pair is exactly an M x N operand as bsq_quantize(out_fmt, y, M, N) lays it out, ready
 * as fc2's A. Codes and scales are the MX quantization of the kernel's fp32 y, which differs
 * from the exact value by the fp32 accumulation and GELU rounding; a code differs from the
 * exact value's code only where that value lies within this error of a rounding boundary.
 * Shapes: as bsq_gemm, and N % 32 == 0. Errors: as bsq_gemm; BSQ_ERR_ARG for another out_fmt
 * or a NULL out_scales; BSQ_ERR_ALIGN for an unaligned out_scales.
 */
int bsq_gemm_gelu_quantize(int fmt, const void* A, const void* A_scales, const void* B, const void* B_scales,
                           const void* bias_bf16, int out_fmt, void* out_codes, void* out_scales, int64_t M,
                           int64_t N, int64_t K, bsq_stream_t stream);

/*
 * bsq_convt2x2: the head's transposed convolution with kernel 2 and stride 2 as a block-scaled
 * GEMM ("lightly-train - DINOv3 + EoMT on RTX 5090" README, section 4.3: the head's two
 * ScaleBlocks (ConvT k2 s2 -> GELU -> depthwise 3x3 -> LN2D) upscale the patch grid, and ConvT1 /
 * ConvT2 are two of the six quantized GEMM classes). Kernel = stride = 2: every output pixel has
 * exactly one input pixel, so
 *   out[b, 2h + dy, 2w + dx, co] = bf16(alpha * sum_ci Ahat[(b, h, w), ci] * Bhat[(2 dy + dx) C_out + co, ci]
 *                                       + bias[co])        (GELU of it when gelu != 0)
 * is one GEMM with N = 4 C_out whose epilogue stores each output column at its output pixel.
 *   A, A_scales  the NHWC input, batch * H * W rows (tokens in (b, h, w) order) x C_in, as written
 *                by bsq_quantize(fmt, ..., batch * H * W, C_in, ...)
 *   B, B_scales  the weight as a 4 C_out x C_in operand: row (2 dy + dx) C_out + co holds tap
 *                (dy, dx) of output channel co, i.e. W_torch[ci, co, dy, dx] of a PyTorch
 *                ConvTranspose2d weight [C_in, C_out, 2, 2]
 *   bias_bf16    C_out bf16 values or NULL
 *   out_bf16     batch x 2H x 2W x C_out bf16 (NHWC), written
 *   alpha        as bsq_gemm (NVFP4: g_A * g_B from the scale tails)
 * GELU is the erf form evaluated as in bsq_gemm_gelu.
 * Shapes: C_in as bsq_gemm's K (multiple of 128 MXFP8, 256 FP4); C_out % 32 == 0; W divides 32
 * or 32 divides W (so that 32 consecutive tokens are whole image rows or part of one); batch *
 * H * W below 2^31. Otherwise BSQ_ERR_SHAPE. Errors: as bsq_gemm.
 */
int bsq_convt2x2(int fmt, const void* A, const void* A_scales, const void* B, const void* B_scales,
                 const void* bias_bf16, void* out_bf16, int64_t batch, int64_t H, int64_t W, int64_t C_in,
                 int64_t C_out, int gelu, bsq_stream_t stream);

/*
 * bsq_get_device_status: synchronise `stream`, then read and clear the current device's
 * status word. Returns BSQ_OK, BSQ_ERR_TIMEOUT (a kernel's bounded wait on an mbarrier
 * gave up; that kernel returned early and its outputs are incomplete), BSQ_ERR_DEVICE_CHECK (the
 * checked build only: a kernel computed an index outside one of its buffers and skipped that
 * access) or BSQ_ERR_LAUNCH (a CUDA error while synchronising).
 * The checked build, libbsq_checked.so, is the same library compiled with BSQ_DEVICE_CHECKS=1:
 * every global load or store whose address a kernel computes itself (not the tensor copies, which
 * the tensor maps bound) is tested against its buffer's size first. It is the stand-in for a
 * memory checker.
 */
int bsq_get_device_status(bsq_stream_t stream);

/*
 * bsq_selftest_timeout: enqueue a one-thread kernel that waits on an mbarrier nothing
 * arrives on, bounded by limit_ns nanoseconds of %globaltimer; it then records
 * BSQ_ERR_TIMEOUT in the device status word and returns. Exercises the failure path of
 * every bounded wait without faulting or hanging the GPU. limit_ns in [1e3, 1e10].
 */
int bsq_selftest_timeout(int64_t limit_ns, bsq_stream_t stream);

/*
 * bsq_selftest_device_check: enqueue a one-thread kernel whose single index check fails. The
 * checked build (libbsq_checked.so) records BSQ_ERR_DEVICE_CHECK in the device status word; the
 * normal build, whose checks compile to nothing, records nothing. Shows which build is loaded and
 * that its checks report through the status word without a trap.
 */
int bsq_selftest_device_check(bsq_stream_t stream);

/*
 * bsq_test_inject_stall: a test of the failure path of the kernels that wait on barriers, with no
 * GPU fault: arms a one-shot stall for the calling thread's next launch of one kernel class.
 *   kernel         BSQ_KERNEL_GEMM (every bsq_gemm* and bsq_convt2x2 launch), BSQ_KERNEL_DUAL
 *                  (bsq_quantize_dual) or BSQ_KERNEL_LAYERNORM (bsq_layernorm_quantize on fp32
 *                  sources or rows longer than 1024 elements: its shared-memory kernel; bf16 rows
 *                  of at most 1024 elements run a kernel that waits on no barrier, and the stall
 *                  stays armed past such a launch)
 *   after_stages   >= 0: the producers of that launch stop issuing loads -- and never announce the
 *                  missing bytes -- after this many pipeline stages per CTA, so a consumer waits for
 *                  a stage that never arrives; -1: disarm any stall armed on the calling thread
 *   wait_limit_ns  the limit of every bounded wait in that launch, in [1e3, 1e10] (the default
 *                  limit is 2 s)
 * The starved wait gives up after wait_limit_ns; the kernel then records BSQ_ERR_TIMEOUT in the
 * device status word, every role leaves its loop, the loads already issued are waited for (so
 * nothing is left in flight), tensor-core work drains, TMEM is released and the kernel returns.
 * The launch's outputs are incomplete; the next launch of the kernel runs normally. The method has
 * no counterpart: this exists for the tests. Errors: BSQ_ERR_ARG for an unknown kernel, after_stages
 * below -1 or a limit out of range.
 */
#define BSQ_KERNEL_GEMM 1
#define BSQ_KERNEL_DUAL 2
#define BSQ_KERNEL_LAYERNORM 3
int bsq_test_inject_stall(int kernel, int64_t after_stages, int64_t wait_limit_ns);

/* bsq_last_error: the calling thread's last non-zero return code (0 if none). */
int bsq_last_error(void);

/* bsq_strerror: a static string describing a status code. */
const char* bsq_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* BSQ_H */
