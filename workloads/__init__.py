"""Seeded synthetic inputs for the block-scaled linear layer (ViT-B/16, ViT-L/16 shapes).

This module only draws random numbers and rounds them to the storage dtype of the
inputs (fp32 or bf16). It holds none of the quantization or GEMM arithmetic, so both
the CPU oracle and the CUDA path can be fed from it without sharing any of the method.

Shapes and distributions follow the five workloads of the block-scaled ViT linear
layer study (lightly-train DINOv3 + EoMT on RTX 5090 README, §4.3 and §5.3: the
quantized GEMMs are qkv / proj / fc1 / fc2 of every ViT block):

  tiny_mxfp8      A fp32 128x256, B fp32 256x256 (stored N x K), N(0,1), 1% of A x50,
                  zero bias, MXFP8.
  vitb_fc1_mxfp8  ViT-B/16 fc1 at training shape: M = 14*1024, K = 768, N = 3072.
  vitl_mxfp8      ViT-L/16 qkv/proj/fc1/fc2 at M = 7*1024, MXFP8.
  vitl_nvfp4      the same sweep in NVFP4 with Student-t(4) activations.
  vitl_mlp_large  M = 32*1600 tokens, fc1 1024->4096 and fc2 4096->1024, MXFP4 and NVFP4;
                  fc2's input is GELU of an N(0,1) pre-activation.
  vitl_mlp_*_fused / _unfused
                  one ViT-L/16 MLP, fc1 -> GELU -> fc2, with fc2's operand produced by fc1's
                  epilogue (fused) or by a bf16 output and a separate quantize pass (unfused).
  vitb_fc1_mxfp8_train[_sr]
                  one training step of the ViT-B/16 fc1 layer at training shape: forward,
                  dgrad (dX = dY W) and wgrad (dW = dY^T X), every operand from the dual-layout
                  quantizer; the output gradient dY rounded to nearest or stochastically.
  eomt_head_vitl_mxfp8
                  the head's two transposed convolutions (kernel 2, stride 2, ConvT -> GELU of
                  the ScaleBlocks): 32x32 -> 64x64 and 64x64 -> 128x128 grids of a 512x512 frame
                  (ViT-L/16: 1024 channels in and out), a batch of 8 frames.
  vitb_fc1_nvfp4_train_sr
                  the same step in NVFP4 (the README's FP4 training path): X and W with their
                  own per-tensor scales, dY stochastically rounded with the delayed scale of
                  the previous step (headroom 32).

Recipe (every array is drawn in fp64 by numpy's default_rng, cast to fp32 with
round-to-nearest, then to bf16 with round-to-nearest-even where the input is bf16):
  * sub-streams: A <- seed, B <- seed + 1, bias <- seed + 2, pre-activation <- seed + 3;
  * activations N(0,1) (t(4) for the NVFP4 sweep); 0.5 % of the K channels,
    round(0.005 * K) of them picked without replacement from A's stream, scaled x20;
  * weights N(0, 0.02), bias N(0, 0.01);
  * output gradient dY[M, N] N(0, 1e-3) from stream seed + 5 (training workloads);
  * tiny case: round(0.01 * M * K) entries of A picked without replacement, scaled x50.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np

MXFP8 = "mxfp8"
NVFP4 = "nvfp4"
MXFP4 = "mxfp4"


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 values (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Gemm:
    """One quantized linear layer: out[M,N] = A[M,K] . B[N,K]^T + bias[N]."""

    name: str
    fmt: str
    M: int
    K: int
    N: int
    a_dist: str = "normal"          # normal | student_t4 | gelu_normal | normal_outlier50
    a_outlier_channels: bool = True  # 0.5 % of channels x20
    src_f32: bool = False           # the tiny case feeds fp32 activations and weights
    w_std: float = 0.02
    bias_std: Optional[float] = 0.01  # None = zero bias
    seed: int = 0
    # head transposed convolution (kernel 2, stride 2): (batch, H, W) of the NHWC input; then
    # M = batch H W tokens, K = C_in, N = 4 C_out (weight rows (2 dy + dx) C_out + co), bias C_out
    convt: Optional[tuple] = None

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    description: str
    gemms: List[Gemm]
    # "fused" / "unfused": gemms = [fc1, fc2] of one MLP, fc2's A being GELU of fc1's output
    # (quantized in fc1's epilogue, or written as bf16 and quantized by a separate pass);
    # "ln_fused": as "fused", with fc1's A = LayerNorm of the activations, quantized by the
    # LN + quantize kernel; "train": gemms = [the layer], one training step (forward, dgrad,
    # wgrad) with dual-layout operands
    chain: Optional[str] = None
    grad_sr: bool = False  # "train": stochastic rounding of the output gradient
    grad_headroom: Optional[float] = None  # "train", NVFP4: dY's scale delayed by one step, this headroom


def _vitl_sweep(fmt: str, a_dist: str) -> List[Gemm]:
    M = 7 * 1024
    return [
        Gemm("qkv", fmt, M, 1024, 3072, a_dist),
        Gemm("proj", fmt, M, 1024, 1024, a_dist),
        Gemm("fc1", fmt, M, 1024, 4096, a_dist),
        Gemm("fc2", fmt, M, 4096, 1024, a_dist),
    ]


WORKLOADS: Dict[str, Workload] = {
    "tiny_mxfp8": Workload(
        "tiny_mxfp8",
        "A fp32 128x256, B fp32 256x256, N(0,1), 1% of A x50, zero bias, MXFP8",
        [Gemm("tiny", MXFP8, 128, 256, 256, "normal_outlier50", a_outlier_channels=False,
              src_f32=True, w_std=1.0, bias_std=None)],
    ),
    "vitb_fc1_mxfp8": Workload(
        "vitb_fc1_mxfp8",
        "ViT-B/16 MLP fc1 at training shape, MXFP8: M=14336, K=768, N=3072",
        [Gemm("fc1", MXFP8, 14 * 1024, 768, 3072)],
    ),
    "vitl_mxfp8": Workload(
        "vitl_mxfp8", "ViT-L/16 qkv/proj/fc1/fc2 at M=7168, MXFP8", _vitl_sweep(MXFP8, "normal")),
    "vitl_nvfp4": Workload(
        "vitl_nvfp4", "ViT-L/16 qkv/proj/fc1/fc2 at M=7168, NVFP4, Student-t(4) activations",
        _vitl_sweep(NVFP4, "student_t4")),
    "vitl_mlp_large": Workload(
        "vitl_mlp_large",
        "ViT-L/16 MLP at M=51200 tokens (32 frames of 640x640), MXFP4 and NVFP4",
        [
            Gemm("fc1_mxfp4", MXFP4, 32 * 1600, 1024, 4096),
            Gemm("fc2_mxfp4", MXFP4, 32 * 1600, 4096, 1024, "gelu_normal", a_outlier_channels=False),
            Gemm("fc1_nvfp4", NVFP4, 32 * 1600, 1024, 4096),
            Gemm("fc2_nvfp4", NVFP4, 32 * 1600, 4096, 1024, "gelu_normal", a_outlier_channels=False),
        ],
    ),
}


def _mlp_chain(name: str, fmt: str, M: int, chain: str) -> Workload:
    # fc1 weights N(0, 1/sqrt(1024)) so that fc1's outputs spread over the range where GELU
    # bends; fc2 as in the other workloads
    return Workload(name, "ViT-L/16 MLP %sfc1 -> GELU -> fc2 at M=%d, %s, fc2 operand %s" % (
        "LN -> " if chain == "ln_fused" else "", M, fmt.upper(),
        "from bf16 + a quantize pass" if chain == "unfused" else "quantized in fc1's epilogue"),
        [Gemm("fc1", fmt, M, 1024, 4096, w_std=1.0 / 32.0), Gemm("fc2", fmt, M, 4096, 1024)], chain)


for _fmt, _M, _tag in ((MXFP8, 7 * 1024, "vitl_mlp_mxfp8"), (MXFP4, 32 * 1600, "vitl_mlp_large_mxfp4")):
    for _chain in ("fused", "unfused", "ln_fused"):
        WORKLOADS["%s_%s" % (_tag, _chain)] = _mlp_chain("%s_%s" % (_tag, _chain), _fmt, _M, _chain)


for _sr in (False, True):
    _n = "vitb_fc1_mxfp8_train" + ("_sr" if _sr else "")
    WORKLOADS[_n] = Workload(
        _n, "ViT-B/16 MLP fc1 training step (forward, dgrad, wgrad) at M=14336, K=768, N=3072, MXFP8, "
            "dual-layout operands, output gradient rounded %s" % ("stochastically" if _sr else "to nearest even"),
        [Gemm("fc1", MXFP8, 14 * 1024, 768, 3072)], "train", _sr)
WORKLOADS["eomt_head_vitl_mxfp8"] = Workload(
    "eomt_head_vitl_mxfp8",
    "EoMT head transposed convolutions (k2 s2, GELU fused) of ViT-L/16 on 512x512 frames, batch 8, MXFP8: "
    "ConvT1 32x32 -> 64x64, ConvT2 64x64 -> 128x128, 1024 channels",
    [Gemm("convt1", MXFP8, 8 * 32 * 32, 1024, 4 * 1024, convt=(8, 32, 32)),
     Gemm("convt2", MXFP8, 8 * 64 * 64, 1024, 4 * 1024, convt=(8, 64, 64))])
WORKLOADS["vitb_fc1_nvfp4_train_sr"] = Workload(
    "vitb_fc1_nvfp4_train_sr",
    "ViT-B/16 MLP fc1 training step (forward, dgrad, wgrad) at M=14336, K=768, N=3072, NVFP4, dual-layout "
    "operands; dY rounded stochastically with the previous step's amax times headroom 32 as its scale",
    [Gemm("fc1", NVFP4, 14 * 1024, 768, 3072)], "train", True, 32.0)


def _gelu_erf(x: np.ndarray) -> np.ndarray:
    # exact erf form of GELU, fp64; part of the input recipe for fc2's activations
    from scipy.special import erf

    return 0.5 * x * (1.0 + erf(x / math.sqrt(2.0)))


def _store(x64: np.ndarray, src_f32: bool) -> np.ndarray:
    x32 = x64.astype(np.float32)
    return x32 if src_f32 else f32_to_bf16_bits(x32)


def make_activations(g: Gemm, rows: Optional[int] = None) -> np.ndarray:
    """A[M, K] (fp32 values, or uint16 bf16 bits). `rows` < M draws only the leading rows
    of the same stream (the values of those rows are identical to the full draw)."""
    M = g.M if rows is None else rows
    if g.a_dist == "gelu_normal":
        rng = np.random.default_rng(g.seed + 3)
        x = _gelu_erf(rng.standard_normal((M, g.K)))
        return _store(x, g.src_f32)
    rng = np.random.default_rng(g.seed)
    if g.a_dist == "student_t4":
        x = rng.standard_t(4, size=(M, g.K))
    else:
        x = rng.standard_normal((M, g.K))
    if g.a_outlier_channels:
        # channel choice comes from a separate stream so that `rows` slices agree with the full draw
        crng = np.random.default_rng([g.seed, 1])
        n_ch = int(round(0.005 * g.K))
        ch = crng.choice(g.K, size=n_ch, replace=False)
        x[:, ch] *= 20.0
    if g.a_dist == "normal_outlier50":
        assert rows is None, "the tiny case is always drawn whole"
        n_out = int(round(0.01 * M * g.K))
        idx = rng.choice(M * g.K, size=n_out, replace=False)
        x.reshape(-1)[idx] *= 50.0
    return _store(x, g.src_f32)


def make_weights(g: Gemm) -> np.ndarray:
    """B[N, K] (K contiguous, the layout of nn.Linear.weight)."""
    rng = np.random.default_rng(g.seed + 1)
    w = rng.standard_normal((g.N, g.K)) * g.w_std
    return _store(w, g.src_f32)


def make_output_grad(g: Gemm, rows: Optional[int] = None, std: float = 1e-3) -> np.ndarray:
    """dY[M, N], the gradient of the layer's output (bf16 bits, or fp32 for fp32 layers); `rows`
    < M draws only the leading rows of the same stream."""
    rng = np.random.default_rng(g.seed + 5)
    M = g.M if rows is None else rows
    return _store(rng.standard_normal((M, g.N)) * std, g.src_f32)


def make_bias(g: Gemm) -> Optional[np.ndarray]:
    """bias[N] (bias[C_out] for a transposed convolution) as uint16 bf16 bits, or None."""
    if g.bias_std is None:
        return None
    rng = np.random.default_rng(g.seed + 2)
    n = g.N // 4 if g.convt is not None else g.N
    return f32_to_bf16_bits((rng.standard_normal(n) * g.bias_std).astype(np.float32))


def random_matrix(rows: int, cols: int, seed: int, std: float = 1.0, dist: str = "normal",
                  src_f32: bool = False) -> np.ndarray:
    """Small seeded matrices for parity and edge-case tests."""
    rng = np.random.default_rng(seed)
    if dist == "student_t4":
        x = rng.standard_t(4, size=(rows, cols)) * std
    elif dist == "uniform_exp":
        # magnitudes spread over many binades, random signs
        x = np.exp2(rng.uniform(-30, 30, size=(rows, cols))) * rng.choice([-1.0, 1.0], size=(rows, cols))
    elif dist == "massive":
        # ViT-L block 0's input as the "lightly-train - DINOv3 + EoMT on RTX 5090" README describes it
        # (section 5.5): rms about 9, with massive activations on the class and register tokens
        # reaching 1992. Rows are tokens, 1024 per image; the first 5 of each image carry values of
        # magnitude 500..1992 in 2 channels, one of them exactly 1992.
        x = rng.standard_normal((rows, cols)) * 9.0
        tok = np.flatnonzero(np.arange(rows) % 1024 < 5)
        ch = rng.choice(cols, size=min(2, cols), replace=False)
        x[np.ix_(tok, ch)] = rng.uniform(500.0, 1992.0, size=(tok.size, ch.size)) * \
            rng.choice([-1.0, 1.0], size=(tok.size, ch.size))
        x[0, ch[0]] = 1992.0
    else:
        x = rng.standard_normal((rows, cols)) * std
    return _store(x, src_f32)


def make_layernorm_affine(cols: int, seed: int = 0):
    """LayerNorm gamma ~ 1 + N(0, 0.1) and beta ~ N(0, 0.1), bf16 bit patterns (stream seed + 4)."""
    rng = np.random.default_rng(seed + 4)
    g = f32_to_bf16_bits((1.0 + 0.1 * rng.standard_normal(cols)).astype(np.float32))
    b = f32_to_bf16_bits((0.1 * rng.standard_normal(cols)).astype(np.float32))
    return g, b
