/*
 * bsq_oracle.c -- plain, slow CPU oracle for block-scaled quantization (MXFP8, NVFP4,
 * MXFP4) and the block-scaled GEMM with a bias epilogue.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark load this library. The product (libbsq.so and its Python binding) never
 * calls it, and it shares no source, header, table or helper with the CUDA path.
 *
 * Sources (page title, section):
 *   [LT]  "lightly-train - DINOv3 + EoMT inference and training optimisation on RTX 5090"
 *         README, section 2 (number-format table): MXFP8 = E4M3 elements + a UE8M0 scale per
 *         1x32 block (8.25 bits/value); NVFP4 = e2m1 elements + an E4M3 scale per 1x16
 *         block + an fp32 per-tensor scale (4.5 bits/value); MXFP4 = e2m1 + UE8M0 per 1x32
 *         (4.25 bits/value). Section 4.7: the fake-quant study rounds to nearest ("RN").
 *         Section 5.5: 4-bit operands are K-major, every GEMM is written "TN".
 *   [BF]  "2x, not 16x: the real ledger of BF16 mixed precision" blog, section 2 table
 *         (bf16 = 8 exponent / 7 mantissa bits) and section 5.4 (largest finite E4M3 = 448).
 *
 * The pages leave these steps open; the oracle takes the following readings:
 *   R1  Rounding of elements and E4M3 scales: round to nearest, ties to even, from the
 *       exact value; magnitudes at or above the largest finite value saturate to it
 *       (448 for E4M3, 6 for e2m1). A zero result keeps the sign of its input.
 *   R2  UE8M0 exponent of a 1x32 block: e = floor(log2(amax)) - emax_elem, emax_elem = 8
 *       (E4M3) or 2 (e2m1), clamped to [-127, 127]; amax = 0 gives e = -127. The scale byte
 *       is e + 127 and the element is RNE_sat(x * 2^-e). (The shared-exponent rule of the
 *       OCP microscaling formats.)
 *   R3  NVFP4 per-tensor scale g = fp32(amax_tensor / 2688), 2688 = 6 * 448. Per 1x16 block:
 *       s_code = E4M3 RNE_sat(fp32(bamax / fp32(6 * g))), s = decode(s_code); elements
 *       y = fp32(x / fp32(s * g)), code = e2m1 RNE_sat(y). Every step is one IEEE fp32
 *       operation rounded to nearest (no fused multiply-add). s = 0 (which includes g = 0)
 *       makes every code of the block a zero carrying the sign of its input. With a given
 *       per-tensor scale the same steps run from that g.
 *   R4  Packing: codes are row-major with K contiguous; e2m1 element 2j is the low nibble
 *       of byte j and element 2j+1 the high nibble.
 *   R5  Scale layout: tiles of 128 rows x 4 scale columns (512 bytes); tile index =
 *       (row / 128) * n_col_tiles + col / 4; inside a tile byte (row % 32) * 16 +
 *       ((row / 32) % 4) * 4 + col % 4. Padding rows/columns hold 0. For NVFP4 a 16-byte
 *       tail after the tiles holds {g, amax_tensor, 0, 0} as fp32.
 *   R6  GEMM: y[m,n] = alpha * sum_k Ahat[m,k] * Bhat[n,k] + bias[n] in fp64, kept unrounded;
 *       alpha = g_A * g_B for NVFP4 (the block-scaled sum is formed first), 1 otherwise.
 *   R7  Non-finite inputs are outside the contract; the quantizers reject them.
 *   R8  Producer-fused quantization of a fc1 output ([LT] section 4.3: the MXFP8 stack's fc1
 *       epilogue quantizes the GELU output straight into fc2's operand): the value
 *       quantized is GELU(alpha * acc + bias) with GELU in its exact erf form
 *       0.5 v (1 + erf(v / sqrt 2)), taken before any bf16 rounding, then the MX rule R2
 *       along the output row. Here y is the unrounded fp64 value of R6.
 *   R9  Producer-fused quantization of a LayerNorm output ([LT] section 4.3: the MXFP8 stack
 *       merges LN and quantization into one kernel): y = (x - mean) / sqrt(var + eps) * gamma
 *       + beta per row, mean and biased variance over the row (the usual LayerNorm), gamma and
 *       beta bf16, taken before any bf16 rounding, then the MX rule R2 along the row.
 *   R10 Dual-layout quantization for the backward GEMMs ([LT] section 4.3 / the training path
 *       of the pages: dgrad needs dY along N and W along N, wgrad dY and X along M): one
 *       matrix R x C gives the row-wise MX operand (along C, R x C) and the column-wise one
 *       stored transposed (C x R, quantized along R), each with the MX rule R2.
 *       Stochastic rounding (for gradients) replaces RNE in R1: with q = |v| / spacing (the
 *       element format's spacing at v's binade, subnormal spacing below the smallest normal),
 *       the magnitude rounds up iff frac(q) > u, u = h * 2^-16; |v| >= max still saturates.
 *       h is the 16-bit half (i mod 2: 0 = low, 1 = high) of word ((i mod 8) / 2) of
 *       Philox4x32-10 (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11) at
 *       counter (floor(i/8) low 32 bits, high 32 bits, layout, 0) and key (seed low, seed high),
 *       i the element's index in its layout's order (row layout r * C + c, column layout
 *       c * R + r), layout 0 = row, 1 = column. 16 bits exceed the fraction any bf16 value
 *       keeps below an E4M3 or e2m1 code of the normal range, so E[code] = v there exactly;
 *       for longer fractions (fp32 sources, NVFP4 quotients) the bias is below 2^-16 spacing.
 *   R11 Dual-layout NVFP4 (the pages' fused FP4 quantizer writes NVFP4 codes for both
 *       layouts; [LT] section 4.3 training stack P3, dY with stochastic rounding): one per-tensor
 *       g for the whole matrix (R3: fp32(amax / 2688), or a given g), shared by both layouts;
 *       each layout applies R3 along its rows (1x16 blocks). With stochastic rounding the
 *       element y = fp32(x / fp32(s g)) of R3 rounds by the rule of R10 (e2m1, the same Philox
 *       words and element indices); s = 0 still gives signed zero codes.
 *   R12 Delayed per-tensor scale ([LT] section 5.5: the amax found while quantizing a tensor
 *       in one step, times a headroom factor H, gives the next step's scale without an extra
 *       pass; H = 32 for dY): g_next = fp32(fp32(amax_prev * H) / 2688), amax_prev the amax
 *       recorded by the previous NVFP4 quantization of the tensor.
 *   R13 Head transposed convolutions ([LT] section 4.3: the head's two ScaleBlocks start with a
 *       ConvT of kernel 2 and stride 2 that doubles the patch grid, and both ConvTs are quantized
 *       GEMMs): out[b, 2h + dy, 2w + dx, co] = alpha * sum_ci A[(b, h, w), ci] * B[(2 dy + dx) *
 *       C_out + co, ci] + bias[co], optionally GELU (the ScaleBlock's next step), A the NHWC
 *       input as a (batch H W) x C_in operand, B the weight as a 4 C_out x C_in operand whose row
 *       (2 dy + dx) C_out + co holds the kernel tap (dy, dx) of output channel co. Kernel and
 *       stride 2 do not overlap, so every output pixel has exactly one input pixel.
 *
 * Pins (tests that tie this code to something other than itself) are in the test suite:
 * exhaustive decode tables against two independent float8/float4 libraries, encoders
 * against brute-force nearest search over every bf16 value, power-of-two / top-binade /
 * shift invariants of the UE8M0 rule, NVFP4 sign symmetry and a hand-derived block, the
 * GEMM against a library matmul on tiny cases and closed forms. The scale layout R5 is a
 * convention (not a value the method fixes); on the CPU it is held to bijectivity and
 * zero padding, and on the GPU the tensor cores' own reading of it pins it end to end.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fopenmp -fPIC -shared (no fast-math).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_MXFP8 1
#define ORC_NVFP4 2
#define ORC_MXFP4 3

#define ORC_OK 0
#define ORC_ERR_ARG -1
#define ORC_ERR_SHAPE -2
#define ORC_ERR_NONFINITE -3

int orc_version(void) { return 1; }

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------------------
 * Decoders (format definitions).
 * ---------------------------------------------------------------------------------- */

/* E4M3 ("FN": no infinities, only S.1111.111 is NaN): sign s, exponent field E (bias 7),
 * mantissa m. E = 0 is subnormal: m * 2^-9. Largest finite 0x7E = 1.75 * 2^8 = 448 [BF 5.4]. */
double orc_decode_e4m3(unsigned c) {
    unsigned s = (c >> 7) & 1u, E = (c >> 3) & 15u, m = c & 7u;
    double mag;
    if (E == 15u && m == 7u) return NAN;
    if (E == 0u) mag = ldexp((double)m, -9);
    else mag = ldexp(1.0 + (double)m / 8.0, (int)E - 7);
    return s ? -mag : mag;
}

/* e2m1: sign, 2-bit exponent (bias 1), 1-bit mantissa; E = 0 is subnormal m * 0.5.
 * Magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}. Only the low nibble of c is read. */
double orc_decode_e2m1(unsigned c) {
    unsigned s = (c >> 3) & 1u, E = (c >> 1) & 3u, m = c & 1u;
    double mag;
    if (E == 0u) mag = 0.5 * (double)m;
    else mag = ldexp(1.0 + (double)m / 2.0, (int)E - 1);
    return s ? -mag : mag;
}

/* UE8M0: a bare biased exponent, 2^(b - 127); 0xFF is NaN. */
double orc_decode_ue8m0(unsigned c) {
    c &= 0xFFu;
    if (c == 0xFFu) return NAN;
    return ldexp(1.0, (int)c - 127);
}

float orc_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ------------------------------------------------------------------------------------
 * Encoders: round to nearest, ties to even, saturating (reading R1).
 *
 * A format with `mbits` mantissa bits and smallest normal exponent `emin` spaces its
 * values 2^(E - mbits) apart inside the binade [2^E, 2^(E+1)) and 2^(emin - mbits) apart
 * below 2^emin (subnormals). With E = max(floor(log2 |v|), emin), q = |v| / 2^(E - mbits)
 * is exact in fp64 and the magnitude code is ((E - emin) << mbits) + RNE(q): the integer
 * q' = RNE(q) carries the code's last bit, so "ties to even" on q' is "ties to the even
 * code", and q' = 2^(mbits+1) rolls over into the next binade's first code.
 * ---------------------------------------------------------------------------------- */
static unsigned encode_rne_sat(double v, int mbits, int emin, double maxval, unsigned maxcode,
                               unsigned signbit_pos) {
    unsigned sign = signbit(v) ? 1u : 0u;
    double a = fabs(v);
    unsigned mag;
    if (a >= maxval) {
        mag = maxcode;
    } else {
        int ex = 0;
        int E;
        double q, r;
        if (a == 0.0) {
            E = emin;
        } else {
            (void)frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1 */
            E = ex - 1;
            if (E < emin) E = emin;
        }
        q = ldexp(a, mbits - E);    /* exact: scaling by a power of two */
        r = nearbyint(q);           /* default rounding mode: to nearest, ties to even */
        mag = ((unsigned)(E - emin) << mbits) + (unsigned)r;
        if (mag > maxcode) mag = maxcode; /* cannot trigger for a < maxval; kept as a guard */
    }
    return (sign << signbit_pos) | mag;
}

unsigned orc_encode_e4m3(double v) { return encode_rne_sat(v, 3, -6, 448.0, 0x7Eu, 7); }
unsigned orc_encode_e2m1(double v) { return encode_rne_sat(v, 1, 0, 6.0, 0x7u, 3); }

/* ------------------------------------------------------------------------------------
 * Scale layout (reading R5).
 * ---------------------------------------------------------------------------------- */
static int64_t block_size(int fmt) { return fmt == ORC_NVFP4 ? 16 : 32; }

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t orc_scale_tiled_offset(int64_t r, int64_t c, int64_t n_scale_cols) {
    int64_t n_col_tiles = ceil_div(n_scale_cols, 4);
    int64_t tile = (r / 128) * n_col_tiles + c / 4;
    return tile * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4);
}

int64_t orc_scales_tiled_bytes(int fmt, int64_t rows, int64_t cols) {
    int64_t nsc = cols / block_size(fmt);
    int64_t bytes = ceil_div(rows, 128) * ceil_div(nsc, 4) * 512;
    return fmt == ORC_NVFP4 ? bytes + 16 : bytes;
}

int64_t orc_codes_bytes(int fmt, int64_t rows, int64_t cols) {
    return fmt == ORC_MXFP8 ? rows * cols : rows * cols / 2;
}

/* Plain row-major scales (rows x n_scale_cols) -> tiled layout; pads are 0, NVFP4 tail set. */
int orc_tile_scales(int fmt, const uint8_t* plain, int64_t rows, int64_t cols, float g, float amax,
                    uint8_t* tiled) {
    int64_t nsc, bytes, r, c;
    if (!plain || !tiled || rows <= 0 || cols <= 0) return ORC_ERR_ARG;
    nsc = cols / block_size(fmt);
    bytes = orc_scales_tiled_bytes(fmt, rows, cols);
    memset(tiled, 0, (size_t)bytes);
    for (r = 0; r < rows; ++r)
        for (c = 0; c < nsc; ++c) tiled[orc_scale_tiled_offset(r, c, nsc)] = plain[r * nsc + c];
    if (fmt == ORC_NVFP4) {
        float tail[4] = {g, amax, 0.0f, 0.0f};
        memcpy(tiled + bytes - 16, tail, 16);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------------------
 * Quantizers.
 * ---------------------------------------------------------------------------------- */
static float load_src(const void* src, int src_f32, int64_t i) {
    if (src_f32) return ((const float*)src)[i];
    return orc_bf16_to_f32(((const uint16_t*)src)[i]);
}

static int check_finite(const void* src, int src_f32, int64_t n) {
    int64_t i;
    int bad = 0;
#pragma omp parallel for reduction(| : bad)
    for (i = 0; i < n; ++i) {
        float x = load_src(src, src_f32, i);
        if (!isfinite(x)) bad |= 1;
    }
    return bad ? ORC_ERR_NONFINITE : ORC_OK;
}

static void put_code(int fmt, uint8_t* codes, int64_t idx, unsigned code) {
    if (fmt == ORC_MXFP8) {
        codes[idx] = (uint8_t)code;
    } else { /* reading R4: even element in the low nibble */
        uint8_t* b = &codes[idx >> 1];
        if ((idx & 1) == 0) *b = (uint8_t)((*b & 0xF0u) | (code & 0xFu));
        else *b = (uint8_t)((*b & 0x0Fu) | ((code & 0xFu) << 4));
    }
}

/* MXFP8 / MXFP4 [LT section 2] with the shared-exponent rule R2.
 * src: rows x cols, bf16 bits (src_f32 = 0) or fp32. codes: MXFP8 rows*cols bytes, MXFP4
 * rows*cols/2 bytes. scales: plain row-major rows x (cols/32) UE8M0 bytes. */
int orc_quantize_mx(int fmt, const void* src, int src_f32, int64_t rows, int64_t cols,
                    uint8_t* codes, uint8_t* scales) {
    int64_t nsc, r;
    int emax_elem, st;
    if (!src || !codes || !scales || rows <= 0 || cols <= 0) return ORC_ERR_ARG;
    if (fmt != ORC_MXFP8 && fmt != ORC_MXFP4) return ORC_ERR_ARG;
    if (cols % 32) return ORC_ERR_SHAPE;
    st = check_finite(src, src_f32, rows * cols);
    if (st) return st;
    nsc = cols / 32;
    emax_elem = fmt == ORC_MXFP8 ? 8 : 2; /* exponent of the largest binade: 448 = 1.75*2^8, 6 = 1.5*2^2 */
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        int64_t b;
        for (b = 0; b < nsc; ++b) {
            int64_t k, base = r * cols + b * 32;
            double amax = 0.0;
            int e, ex;
            for (k = 0; k < 32; ++k) {
                double a = fabs((double)load_src(src, src_f32, base + k));
                if (a > amax) amax = a;
            }
            if (amax == 0.0) {
                e = -127;
            } else {
                (void)frexp(amax, &ex);
                e = (ex - 1) - emax_elem;
                if (e < -127) e = -127;
                if (e > 127) e = 127;
            }
            scales[r * nsc + b] = (uint8_t)(e + 127);
            for (k = 0; k < 32; ++k) {
                double v = ldexp((double)load_src(src, src_f32, base + k), -e); /* exact */
                unsigned code = fmt == ORC_MXFP8 ? orc_encode_e4m3(v) : orc_encode_e2m1(v);
                put_code(fmt, codes, base + k, code);
            }
        }
    }
    return ORC_OK;
}

float orc_tensor_amax(const void* src, int src_f32, int64_t n) {
    int64_t i;
    float amax = 0.0f;
#pragma omp parallel for reduction(max : amax)
    for (i = 0; i < n; ++i) {
        float a = fabsf(load_src(src, src_f32, i));
        if (a > amax) amax = a;
    }
    return amax;
}

/* NVFP4 [LT section 2] with the two-level scaling R3.
 * scales: plain row-major rows x (cols/16) E4M3 bytes. g_out / amax_out receive the
 * per-tensor scale used and the tensor's own amax. */
int orc_quantize_nvfp4(const void* src, int src_f32, int64_t rows, int64_t cols, int global_given,
                       float g_in, uint8_t* codes, uint8_t* scales, float* g_out, float* amax_out) {
    int64_t nsc, r;
    float amax, g, six_g;
    int st;
    if (!src || !codes || !scales || rows <= 0 || cols <= 0) return ORC_ERR_ARG;
    if (cols % 16) return ORC_ERR_SHAPE;
    st = check_finite(src, src_f32, rows * cols);
    if (st) return st;
    if (global_given && !(isfinite(g_in) && g_in >= 0.0f)) return ORC_ERR_ARG;
    nsc = cols / 16;
    amax = orc_tensor_amax(src, src_f32, rows * cols);
    g = global_given ? g_in : amax / 2688.0f; /* one fp32 division, 2688 = 6 * 448 */
    six_g = 6.0f * g;                          /* one fp32 multiplication */
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        int64_t b;
        for (b = 0; b < nsc; ++b) {
            int64_t k, base = r * cols + b * 16;
            float bamax = 0.0f, q, s, sg;
            unsigned s_code;
            for (k = 0; k < 16; ++k) {
                float a = fabsf(load_src(src, src_f32, base + k));
                if (a > bamax) bamax = a;
            }
            if (g == 0.0f) {
                s_code = 0;
            } else {
                q = bamax / six_g;                       /* fp32 division */
                s_code = orc_encode_e4m3((double)q) & 0x7Fu; /* q >= 0; a +0 code for q = 0 */
            }
            scales[r * nsc + b] = (uint8_t)s_code;
            s = (float)orc_decode_e4m3(s_code);          /* exact in fp32 */
            sg = s * g;                                  /* fp32 multiplication */
            for (k = 0; k < 16; ++k) {
                float x = load_src(src, src_f32, base + k);
                unsigned code;
                if (s == 0.0f) {
                    code = signbit(x) ? 0x8u : 0x0u;
                } else {
                    float y = x / sg;                    /* fp32 division */
                    code = orc_encode_e2m1((double)y);
                }
                put_code(ORC_NVFP4, codes, base + k, code);
            }
        }
    }
    if (g_out) *g_out = g;
    if (amax_out) *amax_out = amax;
    return ORC_OK;
}

/* ------------------------------------------------------------------------------------
 * Decode to fp64 (exact): MX x = code * 2^(byte - 127); NVFP4 x = code * s (the per-tensor
 * g is applied by the GEMM's alpha, reading R6). scales are plain row-major.
 * ---------------------------------------------------------------------------------- */
int orc_decode(int fmt, const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols,
               double* out) {
    int64_t bs, nsc, r;
    if (!codes || !scales || !out || rows <= 0 || cols <= 0) return ORC_ERR_ARG;
    bs = block_size(fmt);
    if (cols % bs) return ORC_ERR_SHAPE;
    nsc = cols / bs;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        int64_t k;
        for (k = 0; k < cols; ++k) {
            int64_t idx = r * cols + k;
            uint8_t sb = scales[r * nsc + k / bs];
            double v, s;
            if (fmt == ORC_MXFP8) v = orc_decode_e4m3(codes[idx]);
            else v = orc_decode_e2m1((idx & 1) ? (codes[idx >> 1] >> 4) : (codes[idx >> 1] & 0xFu));
            s = fmt == ORC_NVFP4 ? orc_decode_e4m3(sb) : orc_decode_ue8m0(sb);
            out[idx] = v * s;
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------------------
 * GEMM (reading R6), rows [row0, row1) of the output:
 *   out[m - row0, n] = alpha * sum_k A[m,k] * B[n,k] + bias[n]
 *   abs_out[m - row0, n] = |alpha| * sum_k |A[m,k] * B[n,k]|   (for the tolerance)
 * A: M x K, B: N x K (both K contiguous), fp64. bias: N bf16 bits or NULL.
 * ---------------------------------------------------------------------------------- */
int orc_gemm(const double* A, const double* B, const uint16_t* bias, int64_t M, int64_t N, int64_t K,
             double alpha, int64_t row0, int64_t row1, double* out, double* abs_out) {
    int64_t m;
    if (!A || !B || !out || M <= 0 || N <= 0 || K <= 0) return ORC_ERR_ARG;
    if (row0 < 0 || row1 > M || row0 >= row1) return ORC_ERR_ARG;
#pragma omp parallel for schedule(dynamic, 1)
    for (m = row0; m < row1; ++m) {
        const double* a = A + m * K;
        int64_t n;
        for (n = 0; n < N; ++n) {
            const double* b = B + n * K;
            double acc = 0.0, acc_abs = 0.0;
            int64_t k;
            for (k = 0; k < K; ++k) {
                double p = a[k] * b[k];
                acc += p;
                acc_abs += fabs(p);
            }
            out[(m - row0) * N + n] = alpha * acc + (bias ? (double)orc_bf16_to_f32(bias[n]) : 0.0);
            if (abs_out) abs_out[(m - row0) * N + n] = fabs(alpha) * acc_abs;
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------------------
 * Producer-fused quantization of a fc1 output for fc2 ("lightly-train - DINOv3 + EoMT on
 * RTX 5090" README, section 4.3: in the MXFP8 stack the fc1 epilogue quantizes the GELU
 * output directly into fc2's operand), reading R8.
 * ---------------------------------------------------------------------------------- */

/* out[i] = GELU(v[i]) = v * Phi(v) = 0.5 * v * (1 + erf(v / sqrt 2)), fp64, evaluated as
 * 0.5 * v * erfc(-v / sqrt 2) (libm erfc): the same function without the cancellation of
 * 1 + erf(.) for negative v, where GELU is tiny but not zero. */
int orc_gelu_erf(const double* v, double* out, int64_t n) {
    int64_t i;
    if (!v || !out || n < 0) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i) out[i] = 0.5 * v[i] * erfc(-v[i] / sqrt(2.0));
    return ORC_OK;
}

/* MX quantization (reading R2) of fp64 values: y rows x cols, cols % 32 == 0, finite.
 * codes: MXFP8 rows*cols bytes, MXFP4 rows*cols/2 bytes; scales: plain rows x (cols/32). */
int orc_quantize_mx_f64(int fmt, const double* y, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* scales) {
    int64_t nsc, r, i;
    int emax_elem;
    if (!y || !codes || !scales || rows <= 0 || cols <= 0) return ORC_ERR_ARG;
    if (fmt != ORC_MXFP8 && fmt != ORC_MXFP4) return ORC_ERR_ARG;
    if (cols % 32) return ORC_ERR_SHAPE;
    for (i = 0; i < rows * cols; ++i)
        if (!isfinite(y[i])) return ORC_ERR_NONFINITE;
    nsc = cols / 32;
    emax_elem = fmt == ORC_MXFP8 ? 8 : 2;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        int64_t b;
        for (b = 0; b < nsc; ++b) {
            int64_t k, base = r * cols + b * 32;
            double amax = 0.0;
            int e, ex;
            for (k = 0; k < 32; ++k) {
                double a = fabs(y[base + k]);
                if (a > amax) amax = a;
            }
            if (amax == 0.0) {
                e = -127;
            } else {
                (void)frexp(amax, &ex);
                e = (ex - 1) - emax_elem;
                if (e < -127) e = -127;
                if (e > 127) e = 127;
            }
            scales[r * nsc + b] = (uint8_t)(e + 127);
            for (k = 0; k < 32; ++k) {
                double v = ldexp(y[base + k], -e);
                unsigned code = fmt == ORC_MXFP8 ? orc_encode_e4m3(v) : orc_encode_e2m1(v);
                put_code(fmt, codes, base + k, code);
            }
        }
    }
    return ORC_OK;
}

/* Element encoders over an array: elem 0 = E4M3, 1 = e2m1 (one code per byte). */
int orc_encode_array(int elem, const double* v, int64_t n, uint8_t* out) {
    int64_t i;
    if (!v || !out || n < 0 || (elem != 0 && elem != 1)) return ORC_ERR_ARG;
    for (i = 0; i < n; ++i) out[i] = (uint8_t)(elem == 0 ? orc_encode_e4m3(v[i]) : orc_encode_e2m1(v[i]));
    return ORC_OK;
}

/* LayerNorm of each row of a bf16 / fp32 rows x cols matrix in fp64 (reading R9):
 * out[r, c] = (x[r, c] - mean_r) / sqrt(var_r + eps) * gamma[c] + beta[c], mean_r and the
 * biased variance var_r over the row; gamma, beta: cols bf16 bits. */
int orc_layernorm(const void* src, int src_f32, const uint16_t* gamma, const uint16_t* beta, double eps,
                  int64_t rows, int64_t cols, double* out) {
    int64_t r, st;
    if (!src || !gamma || !beta || !out || rows <= 0 || cols <= 0 || eps < 0.0) return ORC_ERR_ARG;
    st = check_finite(src, src_f32, rows * cols);
    if (st) return (int)st;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        double mean = 0.0, var = 0.0, rstd;
        int64_t c;
        for (c = 0; c < cols; ++c) mean += (double)load_src(src, src_f32, r * cols + c);
        mean /= (double)cols;
        for (c = 0; c < cols; ++c) {
            double d = (double)load_src(src, src_f32, r * cols + c) - mean;
            var += d * d;
        }
        var /= (double)cols;
        rstd = 1.0 / sqrt(var + eps);
        for (c = 0; c < cols; ++c)
            out[r * cols + c] = ((double)load_src(src, src_f32, r * cols + c) - mean) * rstd *
                                    (double)orc_bf16_to_f32(gamma[c]) + (double)orc_bf16_to_f32(beta[c]);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------------------
 * Dual-layout quantization with optional stochastic rounding (reading R10).
 * ---------------------------------------------------------------------------------- */

/* Philox4x32-10 (Salmon et al. SC'11): 10 rounds of the Philox S-box on a 4 x 32-bit counter
 * with a 2 x 32-bit key, the key bumped by the Weyl constants after every round. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3], k0 = key[0], k1 = key[1];
    int rnd;
    for (rnd = 0; rnd < 10; ++rnd) {
        uint64_t p0 = (uint64_t)0xD2511F53u * c0, p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0, hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        c0 = hi1 ^ c1 ^ k0;
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k1;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The uniform u = h * 2^-16 of element i of a layout (reading R10): h the 16-bit half
 * (i mod 2) of word ((i mod 8) / 2) of Philox4x32-10 at counter floor(i / 8). */
static double sr_u(uint64_t seed, int layout, uint64_t i) {
    uint32_t ctr[4], key[2], out[4], h;
    uint64_t g = i >> 3;
    ctr[0] = (uint32_t)g; ctr[1] = (uint32_t)(g >> 32); ctr[2] = (uint32_t)layout; ctr[3] = 0;
    key[0] = (uint32_t)seed; key[1] = (uint32_t)(seed >> 32);
    orc_philox4x32_10(ctr, key, out);
    h = (i & 1) ? out[(i & 7) >> 1] >> 16 : out[(i & 7) >> 1] & 0xFFFFu;
    return ldexp((double)h, -16);
}

/* Stochastic rounding of v to E4M3 (elem 0) or e2m1 (elem 1) with the uniform u in [0, 1):
 * the magnitude steps up iff frac(|v| / spacing) > u; saturating. */
static unsigned encode_sr(double v, int elem, double u) {
    const int mbits = elem == 0 ? 3 : 1, emin = elem == 0 ? -6 : 0;
    const double maxval = elem == 0 ? 448.0 : 6.0;
    const unsigned maxcode = elem == 0 ? 0x7Eu : 0x7u, signpos = elem == 0 ? 7u : 3u;
    unsigned sign = signbit(v) ? 1u : 0u, mag;
    double a = fabs(v);
    if (a >= maxval) {
        mag = maxcode;
    } else {
        int ex = 0, E;
        double q, fl;
        if (a == 0.0) {
            E = emin;
        } else {
            (void)frexp(a, &ex);
            E = ex - 1;
            if (E < emin) E = emin;
        }
        q = ldexp(a, mbits - E); /* exact */
        fl = floor(q);
        mag = ((unsigned)(E - emin) << mbits) + (unsigned)fl + ((q - fl) > u ? 1u : 0u);
        if (mag > maxcode) mag = maxcode;
    }
    return (sign << signpos) | mag;
}

int orc_encode_sr_array(int elem, const double* v, const double* u, int64_t n, uint8_t* out) {
    int64_t i;
    if (!v || !u || !out || n < 0 || (elem != 0 && elem != 1)) return ORC_ERR_ARG;
    for (i = 0; i < n; ++i) out[i] = (uint8_t)encode_sr(v[i], elem, u[i]);
    return ORC_OK;
}

/* One MX block of 32 values at stride `step` in `x` (fp64): scale byte (rule R2) and codes,
 * RNE or stochastic with the words of elements base_index + k (k = 0..31) of `layout`. */
static uint8_t mx_block(int fmt, const double* x, int64_t step, int sr, uint64_t seed, int layout,
                        uint64_t base_index, unsigned codes[32]) {
    const int emax_elem = fmt == ORC_MXFP8 ? 8 : 2, elem = fmt == ORC_MXFP8 ? 0 : 1;
    double amax = 0.0;
    int k, e, ex;
    for (k = 0; k < 32; ++k) {
        double a = fabs(x[k * step]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0) {
        e = -127;
    } else {
        (void)frexp(amax, &ex);
        e = (ex - 1) - emax_elem;
        if (e < -127) e = -127;
        if (e > 127) e = 127;
    }
    for (k = 0; k < 32; ++k) {
        double v = ldexp(x[k * step], -e);
        if (sr) {
            double u = sr_u(seed, layout, base_index + (uint64_t)k);
            codes[k] = encode_sr(v, elem, u);
        } else {
            codes[k] = elem == 0 ? orc_encode_e4m3(v) : orc_encode_e2m1(v);
        }
    }
    return (uint8_t)(e + 127);
}

/* Dual-layout MX quantization (reading R10) of a bf16 / fp32 R x C matrix (R % 32 == 0 and
 * C % 32 == 0): row codes R x C (MXFP8 bytes / MXFP4 nibbles) with plain row scales R x C/32,
 * column codes C x R (the transpose, quantized along R) with plain scales C x R/32. */
int orc_quantize_mx_dual(int fmt, const void* src, int src_f32, int64_t R, int64_t C, int sr, uint64_t seed,
                         uint8_t* row_codes, uint8_t* row_scales, uint8_t* col_codes, uint8_t* col_scales) {
    double* x;
    int64_t i, r, c;
    int st;
    if (!src || !row_codes || !row_scales || !col_codes || !col_scales || R <= 0 || C <= 0) return ORC_ERR_ARG;
    if (fmt != ORC_MXFP8 && fmt != ORC_MXFP4) return ORC_ERR_ARG;
    if (R % 32 || C % 32) return ORC_ERR_SHAPE;
    st = check_finite(src, src_f32, R * C);
    if (st) return st;
    x = (double*)malloc((size_t)(R * C) * sizeof(double));
    if (!x) return ORC_ERR_ARG;
    for (i = 0; i < R * C; ++i) x[i] = (double)load_src(src, src_f32, i);
#pragma omp parallel for schedule(static)
    for (r = 0; r < R; ++r) {
        int64_t b;
        unsigned codes[32];
        int k;
        for (b = 0; b < C / 32; ++b) {
            row_scales[r * (C / 32) + b] =
                mx_block(fmt, x + r * C + b * 32, 1, sr, seed, 0, (uint64_t)(r * C + b * 32), codes);
            for (k = 0; k < 32; ++k) put_code(fmt, row_codes, r * C + b * 32 + k, codes[k]);
        }
    }
#pragma omp parallel for schedule(static)
    for (c = 0; c < C; ++c) {
        int64_t b;
        unsigned codes[32];
        int k;
        for (b = 0; b < R / 32; ++b) {
            col_scales[c * (R / 32) + b] =
                mx_block(fmt, x + (b * 32) * C + c, C, sr, seed, 1, (uint64_t)(c * R + b * 32), codes);
            for (k = 0; k < 32; ++k) put_code(fmt, col_codes, c * R + b * 32 + k, codes[k]);
        }
    }
    free(x);
    return ORC_OK;
}

/* One NVFP4 block of 16 values at stride `step` of `x` (R3 with the shared g and 6 g): E4M3
 * scale code and e2m1 codes, round-to-nearest or stochastic with the words of elements
 * base_index + k of `layout` (R11). */
static uint8_t nv_block(const float* x, int64_t step, float g, float six_g, int sr, uint64_t seed, int layout,
                        uint64_t base_index, unsigned codes[16]) {
    float bamax = 0.0f, q, s, sg;
    unsigned s_code;
    int k;
    for (k = 0; k < 16; ++k) {
        float a = fabsf(x[k * step]);
        if (a > bamax) bamax = a;
    }
    if (g == 0.0f) {
        s_code = 0;
    } else {
        q = bamax / six_g;                           /* fp32 division */
        s_code = orc_encode_e4m3((double)q) & 0x7Fu;
    }
    s = (float)orc_decode_e4m3(s_code);              /* exact in fp32 */
    sg = s * g;                                      /* fp32 multiplication */
    for (k = 0; k < 16; ++k) {
        float xv = x[k * step];
        if (s == 0.0f) {
            codes[k] = signbit(xv) ? 0x8u : 0x0u;
        } else {
            float y = xv / sg;                       /* fp32 division */
            if (sr) {
                double u = sr_u(seed, layout, base_index + (uint64_t)k);
                codes[k] = encode_sr((double)y, 1, u);
            } else {
                codes[k] = orc_encode_e2m1((double)y);
            }
        }
    }
    return (uint8_t)s_code;
}

/* Dual-layout NVFP4 (reading R11) of a bf16 / fp32 R x C matrix (R % 16 == 0, C % 16 == 0):
 * row codes R x C with plain E4M3 scales R x C/16, column codes C x R (the transpose,
 * quantized along R) with plain scales C x R/16; g_out / amax_out receive the shared
 * per-tensor scale and the tensor's amax. */
int orc_quantize_nv_dual(const void* src, int src_f32, int64_t R, int64_t C, int global_given, float g_in, int sr,
                         uint64_t seed, uint8_t* row_codes, uint8_t* row_scales, uint8_t* col_codes,
                         uint8_t* col_scales, float* g_out, float* amax_out) {
    float* x;
    float amax, g, six_g;
    int64_t i, r, c;
    int st;
    if (!src || !row_codes || !row_scales || !col_codes || !col_scales || R <= 0 || C <= 0) return ORC_ERR_ARG;
    if (R % 16 || C % 16) return ORC_ERR_SHAPE;
    st = check_finite(src, src_f32, R * C);
    if (st) return st;
    if (global_given && !(isfinite(g_in) && g_in >= 0.0f)) return ORC_ERR_ARG;
    amax = orc_tensor_amax(src, src_f32, R * C);
    g = global_given ? g_in : amax / 2688.0f; /* one fp32 division, 2688 = 6 * 448 */
    six_g = 6.0f * g;                          /* one fp32 multiplication */
    x = (float*)malloc((size_t)(R * C) * sizeof(float));
    if (!x) return ORC_ERR_ARG;
    for (i = 0; i < R * C; ++i) x[i] = load_src(src, src_f32, i);
#pragma omp parallel for schedule(static)
    for (r = 0; r < R; ++r) {
        int64_t b;
        unsigned codes[16];
        int k;
        for (b = 0; b < C / 16; ++b) {
            row_scales[r * (C / 16) + b] =
                nv_block(x + r * C + b * 16, 1, g, six_g, sr, seed, 0, (uint64_t)(r * C + b * 16), codes);
            for (k = 0; k < 16; ++k) put_code(ORC_NVFP4, row_codes, r * C + b * 16 + k, codes[k]);
        }
    }
#pragma omp parallel for schedule(static)
    for (c = 0; c < C; ++c) {
        int64_t b;
        unsigned codes[16];
        int k;
        for (b = 0; b < R / 16; ++b) {
            col_scales[c * (R / 16) + b] =
                nv_block(x + (b * 16) * C + c, C, g, six_g, sr, seed, 1, (uint64_t)(c * R + b * 16), codes);
            for (k = 0; k < 16; ++k) put_code(ORC_NVFP4, col_codes, c * R + b * 16 + k, codes[k]);
        }
    }
    free(x);
    if (g_out) *g_out = g;
    if (amax_out) *amax_out = amax;
    return ORC_OK;
}

/* Delayed per-tensor NVFP4 scale (reading R12): two fp32 operations. */
float orc_delayed_global_scale(float amax_prev, float headroom) {
    float a = amax_prev * headroom; /* fp32 multiplication */
    return a / 2688.0f;             /* fp32 division */
}

/* Transposed convolution, kernel 2, stride 2 (reading R13), from decoded fp64 operands:
 * A (batch*H*W) x Cin (NHWC input rows), B (4*Cout) x Cin, bias Cout bf16 bits (may be NULL),
 * out batch x 2H x 2W x Cout fp64, written by the definition one output pixel at a time. */
int orc_convt2x2(const double* A, const double* B, const uint16_t* bias, int64_t batch, int64_t H, int64_t W,
                 int64_t Cin, int64_t Cout, double alpha, int gelu, double* out) {
    int64_t b;
    if (!A || !B || !out || batch <= 0 || H <= 0 || W <= 0 || Cin <= 0 || Cout <= 0) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (b = 0; b < batch; ++b) {
        int64_t ho, wo, co, ci;
        for (ho = 0; ho < 2 * H; ++ho) {
            for (wo = 0; wo < 2 * W; ++wo) {
                const int64_t h = ho / 2, dy = ho % 2, w = wo / 2, dx = wo % 2;
                const double* a = A + ((b * H + h) * W + w) * Cin;
                double* o = out + ((b * 2 * H + ho) * 2 * W + wo) * Cout;
                for (co = 0; co < Cout; ++co) {
                    const double* wt = B + ((2 * dy + dx) * Cout + co) * Cin;
                    double acc = 0.0, v;
                    for (ci = 0; ci < Cin; ++ci) acc += a[ci] * wt[ci];
                    v = alpha * acc + (bias ? (double)orc_bf16_to_f32(bias[co]) : 0.0);
                    o[co] = gelu ? 0.5 * v * erfc(-v / sqrt(2.0)) : v;
                }
            }
        }
    }
    return ORC_OK;
}
