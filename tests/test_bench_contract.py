"""bench.py's reference arm on CPU: one JSON line with the contract's keys, the oracle timed as the
reference (`impl`, `cpu_baseline`, an `e2e` with no host copies), on the small workload."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_mxfp8", "--steps", "2", "--warmup", "0"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout  # exactly one JSON line
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 0
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == "tiny_mxfp8"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def _launch_csv(path, launches):
    """An ncu --csv launch list (one row per metric) for `launches` = [(kernel name, read, write, ns)]."""
    import csv

    with open(path, "w", newline="") as f:
        f.write("==PROF== Connected to process 1\n")
        w = csv.writer(f, quoting=csv.QUOTE_ALL)
        w.writerow(["ID", "Process ID", "Process Name", "Host Name", "Kernel Name", "Context", "Stream", "Block Size",
                    "Grid Size", "Device", "CC", "Section Name", "Metric Name", "Metric Unit", "Metric Value"])
        for i, (name, rd, wr, ns) in enumerate(launches):
            for m, u, v in (("dram__bytes_read.sum", "byte", rd), ("dram__bytes_write.sum", "Mbyte", wr / 1e6),
                            ("gpu__time_duration.sum", "ns", ns)):
                w.writerow([i, 1, "python3", "h", name, 1, 7, "(256, 1, 1)", "(304, 1, 1)", 0, "10.3", "Command line "
                            "profiler metrics", m, u, "{:,}".format(v) if isinstance(v, int) else repr(v)])


def test_record_traffic_per_step_bytes(tmp_path):
    """--record-traffic: library launches only (the L2 flush is left out), GEMM and quantizer
    classes summed per step over the captured steps, units converted, keyed by the source hash;
    a launch count that does not match the steps captured is refused."""
    sys.path.insert(0, ROOT)
    import bench

    flush = "void at::native::vectorized_elementwise_kernel<4, at::native::FillFunctor<unsigned char>>(int)"
    step = [(flush, 0, 256_000_000, 60_000),
            ("void bsq::<unnamed>::amax_kernel<0>(const uint4 *, long, unsigned int *)", 1000, 0, 10_000),
            ("void bsq::<unnamed>::stream_kernel<2, 0, 1>(bsq::<unnamed>::QuantBatch)", 2000, 500_000, 20_000),
            ("void bsq::<unnamed>::gemm_kernel<2, 0>(bsq::<unnamed>::GemmArgs)", 3000, 4_000_000, 30_000)]
    csv_path, side, out = tmp_path / "l.csv", tmp_path / "side.json", tmp_path / "traffic.json"
    _launch_csv(csv_path, step * 3)
    side.write_text(json.dumps({"workload": "w", "steps": 3, "kernel_source_hash": "abc", "launches_per_step": 3}))
    bench.record_traffic(str(csv_path), str(side), "cmd", out_path=str(out))
    d = json.loads(out.read_text())["w"]
    assert d["kernel_source_hash"] == "abc" and d["steps_captured"] == 3 and d["command"] == "cmd"
    q, g = d["classes"]["quantize"], d["classes"]["gemm"]
    assert q["launches_per_step"] == 2 and q["dram_bytes_per_step"] == 1000 + 2000 + 500_000
    assert g["launches_per_step"] == 1 and g["dram_bytes_per_step"] == 3000 + 4_000_000
    assert abs(g["ncu_us_per_step"] - 30.0) < 1e-9
    assert d["kernels"]["stream_kernel<2, 0, 1>"]["dram_write_per_step"] == 500_000
    assert bench.recorded_traffic("abc", "w", "gemm", path=str(out)) == 4_003_000
    assert bench.recorded_traffic("abd", "w", "gemm", path=str(out)) is None  # sources changed since
    side.write_text(json.dumps({"workload": "w", "steps": 2, "kernel_source_hash": "abc", "launches_per_step": 3}))
    with pytest.raises(SystemExit):  # a launch list of 3 steps is not 2 steps
        bench.record_traffic(str(csv_path), str(side), "cmd", out_path=str(out))


def test_kernel_hash_ignores_comments_only():
    """The traffic record's key changes with the code, not with its comments or layout."""
    sys.path.insert(0, ROOT)
    import bench

    a = 'int f(int x) {  // doubles x\n  return 2 * x; /* two */ }\nconst char* s = "a // b";\n'
    b = '/* file header */\nint f(int x) {\n  return 2 * x;\n}\nconst char* s = "a // b";  // kept\n'
    c = 'int f(int x) { return 3 * x; }\nconst char* s = "a // b";\n'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert '"a // b"' in bench._code_only(a)
