"""The checked build (libbsq_checked.so: every global access whose address a kernel computes is
tested against its buffer first; a failed test records BSQ_ERR_DEVICE_CHECK in the status word and
skips the access) -- the stand-in for a memory checker, which this pool does not offer.

The parity suite asserts a zero device status after every call, so running it on the checked
build shows that no kernel computes an out-of-range index on any of its shapes (ragged rows and
columns, guard regions, every epilogue mode, split-K, both dual layouts, LayerNorm, the injected
stalls) while producing the same oracle-exact results. It runs in a child process, which loads
the checked library in place of the normal one."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
# every GPU test file but this one and the last-collected no-allocation test; the full-size
# workload tests are left to the normal build (they take most of the suite's time)
FILES = ["test_gpu_backward.py", "test_gpu_convt.py", "test_gpu_dual.py", "test_gpu_failure.py", "test_gpu_fused.py",
         "test_gpu_gemm.py", "test_gpu_guards.py", "test_gpu_layernorm.py", "test_gpu_nv_quotient.py",
         "test_gpu_quantize.py", "test_gpu_splitk.py"]


def test_selftest_tells_the_builds_apart():
    code = ("import block_scaled_precision_bsq_gb300 as b; assert b.bsq_selftest_device_check() == b.OK; "
            "print(b.device_status())")
    got = {}
    for lib in ("normal", "checked"):
        env = dict(os.environ, BSQ_LIBRARY=lib)
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        got[lib] = int(r.stdout.strip().splitlines()[-1])
    assert got == {"normal": 0, "checked": -7}


def test_parity_suite_passes_on_the_checked_build():
    assert all(os.path.exists(os.path.join(ROOT, "tests", f)) for f in FILES)
    env = dict(os.environ, BSQ_LIBRARY="checked")
    cmd = [sys.executable, "-m", "pytest", "-m", "gpu", "-x", "-q", "-p", "no:cacheprovider", "-k", "not full_size"] + \
        [os.path.join("tests", f) for f in FILES]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, (r.stdout[-4000:], r.stderr[-2000:])
    assert " passed" in r.stdout and "failed" not in r.stdout
