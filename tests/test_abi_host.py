"""Host-side checks of the C ABI that need no GPU: the library loads and exports every
function include/bsq.h declares, the size helpers, and argument validation that returns
before any CUDA call."""
import ctypes
import importlib.util
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bsq.h")


@pytest.fixture(scope="module")
def bsq():
    spec = importlib.util.spec_from_file_location("_bsq_build", os.path.join(ROOT, "block_scaled_precision_bsq_gb300",
                                                                            "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    import block_scaled_precision_bsq_gb300 as b

    return b


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bsq_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(bsq):
    names = declared_functions()
    assert len(names) >= 8
    lib = ctypes.CDLL(bsq.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(bsq.EXPORTS)


@pytest.mark.parametrize("fmt", ["mxfp8", "nvfp4", "mxfp4"])
@pytest.mark.parametrize("rows,cols", [(1, 32), (128, 256), (200, 96), (7203, 1024), (51200, 4096)])
def test_size_helpers_match_the_oracle_layout(bsq, fmt, rows, cols):
    if fmt == "nvfp4" or cols % 32 == 0:
        assert bsq.bsq_codes_bytes(fmt, rows, cols) == oracle.codes_bytes(fmt, rows, cols)
        assert bsq.bsq_scales_bytes(fmt, rows, cols) == oracle.scales_tiled_bytes(fmt, rows, cols)


def test_size_helpers_reject_bad_args(bsq):
    assert bsq.bsq_codes_bytes(9, 4, 32) == 0
    assert bsq.bsq_scales_bytes("mxfp8", 0, 32) == 0
    assert bsq.bsq_codes_bytes("nvfp4", -1, 32) == 0


def test_argument_errors_before_any_cuda_call(bsq):
    p = 1 << 20  # a 16-byte aligned dummy address: never dereferenced on these paths
    assert bsq.bsq_quantize(7, p, 4, 32, p, p) == bsq.ERR_ARG                          # unknown format
    assert bsq.bsq_quantize(bsq.MXFP8 | 0x4000, p, 4, 32, p, p) == bsq.ERR_ARG         # unknown flag
    assert bsq.bsq_quantize(bsq.MXFP8, None, 4, 32, p, p) == bsq.ERR_ARG
    assert bsq.bsq_quantize(bsq.MXFP8, p, 0, 32, p, p) == bsq.ERR_ARG
    assert bsq.bsq_quantize(bsq.MXFP8, p, 4, 48, p, p) == bsq.ERR_SHAPE                # 48 % 32
    assert bsq.bsq_quantize(bsq.NVFP4, p, 4, 40, p, p) == bsq.ERR_SHAPE                # 40 % 16
    assert bsq.bsq_quantize(bsq.MXFP8, p, 1 << 31, 32, p, p) == bsq.ERR_SHAPE          # rows >= 2^31
    good = (p, 4, 64, p, p, None)
    assert bsq.bsq_quantize_batch(bsq.MXFP8, []) == bsq.ERR_ARG                        # count 0
    assert bsq.bsq_quantize_batch(bsq.MXFP8, [good] * 9) == bsq.ERR_ARG                # count > 8
    assert bsq.bsq_quantize_batch(bsq.MXFP8, [good, (p, 4, 48, p, p, None)]) == bsq.ERR_SHAPE  # item 2
    assert bsq.bsq_quantize_batch(bsq.MXFP8, [good, (p + 8, 4, 64, p, p, None)]) == bsq.ERR_ALIGN
    assert bsq.bsq_quantize_batch(bsq.NVFP4 | bsq.FLAG_GLOBAL_GIVEN, [good]) == bsq.ERR_ARG  # no g
    assert bsq.bsq_quantize(bsq.MXFP8, p, 4, 1 << 31, p, p) == bsq.ERR_SHAPE           # cols >= 2^31
    assert bsq.bsq_quantize(bsq.NVFP4 | bsq.FLAG_GLOBAL_GIVEN, p, 4, 32, p, p, None) == bsq.ERR_ARG
    assert bsq.bsq_quantize(bsq.MXFP8 | bsq.FLAG_GLOBAL_GIVEN, p, 4, 32, p, p, p) == bsq.ERR_ARG
    assert bsq.bsq_quantize(bsq.MXFP8, p + 8, 4, 32, p, p) == bsq.ERR_ALIGN
    assert bsq.bsq_last_error() == bsq.ERR_ALIGN
    assert bsq.bsq_gemm(bsq.MXFP8, p, p, p, p, None, p, 128, 256, 96) == bsq.ERR_SHAPE    # K % 128
    assert bsq.bsq_gemm(bsq.NVFP4, p, p, p, p, None, p, 128, 256, 128) == bsq.ERR_SHAPE   # K % 256
    assert bsq.bsq_gemm(bsq.MXFP4, p, p, p, p, None, p, 128, 260, 256) == bsq.ERR_SHAPE   # N % 8
    assert bsq.bsq_gemm_gelu(bsq.MXFP8, p, p, p, p, None, p, 128, 256, 96) == bsq.ERR_SHAPE  # K % 128
    ln = bsq.bsq_layernorm_quantize
    assert ln(bsq.NVFP4, p, p, p, 1e-6, 4, 64, p, p) == bsq.ERR_ARG          # MX formats only
    assert ln(bsq.MXFP8, p, None, p, 1e-6, 4, 64, p, p) == bsq.ERR_ARG       # gamma
    assert ln(bsq.MXFP8, p, p, p, -1.0, 4, 64, p, p) == bsq.ERR_ARG          # eps < 0
    assert ln(bsq.MXFP8, p, p, p, 1e-6, 4, 8224, p, p) == bsq.ERR_SHAPE      # row > 16 KB
    assert ln(bsq.MXFP8, p, p + 2, p, 1e-6, 4, 64, p, p) == bsq.ERR_ALIGN    # gamma alignment
    gq = bsq.bsq_gemm_gelu_quantize
    assert gq(bsq.MXFP8, p, p, p, p, None, bsq.NVFP4, p, p, 128, 256, 256) == bsq.ERR_ARG      # out fmt
    assert gq(bsq.MXFP8, p, p, p, p, None, bsq.MXFP8, p, None, 128, 256, 256) == bsq.ERR_ARG   # no scales
    assert gq(bsq.MXFP8, p, p, p, p, None, bsq.MXFP8, p, p, 128, 264, 256) == bsq.ERR_SHAPE   # N % 32
    assert gq(bsq.MXFP8, p, p, p, p, None, bsq.MXFP4, p, p + 4, 128, 256, 256) == bsq.ERR_ALIGN
    assert bsq.bsq_gemm(bsq.MXFP8, p, p, p, p, None, None, 128, 256, 256) == bsq.ERR_ARG
    assert bsq.bsq_gemm(bsq.MXFP8, p, p + 4, p, p, None, p, 128, 256, 256) == bsq.ERR_ALIGN
    assert bsq.bsq_gemm(bsq.MXFP8, p, p, p, p, p + 1, p, 128, 256, 256) == bsq.ERR_ALIGN
    assert bsq.bsq_selftest_timeout(10, None) == bsq.ERR_ARG
    cv = bsq.bsq_convt2x2
    assert cv(bsq.MXFP8, p, p, p, p, None, p, 0, 4, 4, 128, 64) == bsq.ERR_ARG           # batch
    assert cv(bsq.MXFP8, p, p, p, p, None, p, 1, 4, 4, 128, 48) == bsq.ERR_SHAPE         # C_out % 32
    assert cv(bsq.MXFP8, p, p, p, p, None, p, 1, 4, 48, 128, 64) == bsq.ERR_SHAPE        # W vs 32
    assert cv(bsq.MXFP8, p, p, p, p, None, p, 1, 4, 4, 96, 64) == bsq.ERR_SHAPE          # C_in % 128
    assert cv(bsq.NVFP4, p, p, p, p, None, p, 1, 4, 4, 128, 64) == bsq.ERR_SHAPE         # C_in % 256
    assert cv(bsq.MXFP8, p, p + 4, p, p, None, p, 1, 4, 4, 128, 64) == bsq.ERR_ALIGN
    ds = bsq.bsq_delayed_global_scale
    assert ds(None, 64, 64, 32.0, p) == bsq.ERR_ARG
    assert ds(p, 64, 64, 0.0, p) == bsq.ERR_ARG                                    # headroom
    assert ds(p, 64, 64, float("inf"), p) == bsq.ERR_ARG
    assert ds(p, 64, 40, 32.0, p) == bsq.ERR_SHAPE                                 # cols % 16
    assert ds(p, 64, 64, 32.0, p + 2) == bsq.ERR_ALIGN                             # g_out
    dq = bsq.bsq_quantize_dual
    assert dq(7, p, 64, 64, 0, p, p, p, p) == bsq.ERR_ARG                          # format
    assert dq(bsq.MXFP8 | bsq.FLAG_GLOBAL_GIVEN, p, 64, 64, 0, p, p, p, p, p) == bsq.ERR_ARG  # MX given g
    assert dq(bsq.NVFP4 | bsq.FLAG_GLOBAL_GIVEN, p, 64, 64, 0, p, p, p, p, None) == bsq.ERR_ARG  # no g
    assert dq(bsq.NVFP4, p, 64, 64, 0, p, p, p, p, p + 2) == bsq.ERR_ALIGN          # g alignment
    assert dq(bsq.MXFP8, p, 64, 64, 0, p, p, None, p) == bsq.ERR_ARG               # col codes
    assert dq(bsq.MXFP8, p, 0, 64, 0, p, p, p, p) == bsq.ERR_ARG                   # rows
    assert dq(bsq.MXFP8, p, 48, 64, 0, p, p, p, p) == bsq.ERR_SHAPE                # rows % 32
    assert dq(bsq.MXFP4 | bsq.FLAG_STOCHASTIC, p, 64, 80, 0, p, p, p, p) == bsq.ERR_SHAPE  # cols % 32
    assert dq(bsq.MXFP8, p, 1 << 31, 64, 0, p, p, p, p) == bsq.ERR_SHAPE           # rows >= 2^31
    assert dq(bsq.MXFP8, p, 64, 64, 0, p, p, p, p + 8) == bsq.ERR_ALIGN            # col scales
    assert dq(bsq.MXFP8 | bsq.FLAG_SRC_F32 | bsq.FLAG_STOCHASTIC, p + 4, 64, 64, 2 ** 64 - 1, p, p, p, p) == \
        bsq.ERR_ALIGN
    sk = bsq.bsq_gemm_splitk
    ws = 2 * 128 * 256 * 4
    assert sk(bsq.MXFP8, p, p, p, p, None, p, 128, 256, 96, 2, p, ws) == bsq.ERR_SHAPE       # K % 128
    assert sk(bsq.MXFP8, p, p, p, p, None, p, 128, 260, 1024, 2, p, ws) == bsq.ERR_SHAPE     # N % 8
    assert sk(bsq.MXFP8, p, p, p, p, None, p, 128, 256, 1024, 0, p, ws) == bsq.ERR_ARG       # splits
    assert sk(bsq.MXFP8, p, p, p, p, None, p, 128, 256, 1024, 9, p, ws) == bsq.ERR_ARG
    assert sk(bsq.NVFP4, p, p, p, p, None, p, 128, 256, 512, 3, p, 3 * ws) == bsq.ERR_ARG    # 2 K stages
    assert sk(bsq.MXFP8, p, p, p, p, None, p, 128, 256, 1024, 2, None, ws) == bsq.ERR_ARG    # no workspace
    assert sk(bsq.MXFP8, p, p, p, p, None, p, 128, 256, 1024, 2, p, ws - 1) == bsq.ERR_ARG   # too small
    assert sk(bsq.MXFP8, p, p, p, p, None, p, 128, 256, 1024, 2, p + 8, ws) == bsq.ERR_ALIGN
    assert bsq.bsq_gemm_splitk_splits(7, 128, 256, 1024) == bsq.ERR_ARG
    assert bsq.bsq_gemm_splitk_splits(bsq.MXFP8, 128, 0, 1024) == bsq.ERR_ARG
    sc = bsq.bsq_gemm_splitk_scratch
    assert sc(bsq.MXFP8, p, p, p, p, None, p, 128, 256, 96, 2) == bsq.ERR_SHAPE              # K % 128
    assert sc(bsq.MXFP8, p, p, p, p, None, p, 128, 256, 1024, 9) == bsq.ERR_ARG              # splits
    assert bsq.bsq_strerror(bsq.ERR_TIMEOUT).startswith("a kernel")
    assert bsq.bsq_strerror(12345) == "unknown status"


def test_no_multicast_bulk_or_tensor_copy_in_the_sources():
    """No bulk or tensor copy (load, store or reduce) in the library's sources uses cluster
    multicast: every CTA loads its own tiles. The tcgen05.commit multicast (an mbarrier signal
    to both CTAs of a pair, not a memory copy) is the only multicast form allowed."""
    csrc = os.path.join(ROOT, "block_scaled_precision_bsq_gb300", "csrc")
    offenders = []
    for name in sorted(os.listdir(csrc)):
        if not name.endswith((".cu", ".cuh", ".h")):
            continue
        text = open(os.path.join(csrc, name)).read()
        for m in re.finditer(r'"[^"\n]*multicast::cluster[^"\n]*"', text):
            if "cp.async.bulk" in m.group(0) or "tcgen05.commit" not in m.group(0):
                offenders.append("%s: %s" % (name, m.group(0)))
    assert not offenders, offenders


def test_stall_injection_argument_errors(bsq):
    inj = bsq.bsq_test_inject_stall
    assert inj(0, 1, 10**6) == bsq.ERR_ARG          # unknown kernel
    assert inj(4, 1, 10**6) == bsq.ERR_ARG
    assert inj(bsq.KERNEL_GEMM, -2, 10**6) == bsq.ERR_ARG
    assert inj(bsq.KERNEL_DUAL, 1, 999) == bsq.ERR_ARG
    assert inj(bsq.KERNEL_LAYERNORM, 1, 10**10 + 1) == bsq.ERR_ARG
    assert inj(bsq.KERNEL_GEMM, 0, 10**6) == bsq.OK   # armed for this thread's next GEMM launch
    assert inj(bsq.KERNEL_GEMM, -1, 10**6) == bsq.OK  # disarmed again


def test_checked_build_exports_the_same_symbols(bsq):
    spec = importlib.util.spec_from_file_location("_bsq_build2", os.path.join(ROOT, "block_scaled_precision_bsq_gb300",
                                                                             "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    lib = ctypes.CDLL(mod.build(checked=True))
    for n in declared_functions():
        assert hasattr(lib, n), n
