"""The benchmark's reference arm on CPU: `bench.py --impl reference` times the
oracle on a sample of the workload and prints one JSON line with the contract's
keys; it runs the requested warm-up steps and sizes its sample to the time budget."""
import json
import os
import subprocess
import sys

from conftest import ROOT


def test_reference_arm_json_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
           "--warmup", "3", "--ref-budget-s", "3", "--workload", "tiny_T16_D256_I128_E9_K3"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["steps"] == 3 and line["warmup"] == 3
    assert line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "tiny_T16_D256_I128_E9_K3"


def test_algorithmic_bytes_of_the_decode_workload():
    """The roofline's byte count: touched experts x 3*I*D*17/32 (e2m1 weights plus one
    e8m0 byte per 32), plus the quantised hidden rows for the GEMM kernel; the whole
    call adds the bf16 hidden in, the bf16 output and 8 bytes per route."""
    import numpy as np

    import bench
    import workloads

    ids = np.array([[e, e + 1, 256] for e in range(0, 32, 2)], np.int32)  # 33 experts touched
    w = workloads.custom(16, 7168, 256, 257, 3)
    total, gemm, touched = bench.alg_bytes(w, ids)
    assert touched == 33
    per_expert = 3 * 256 * 7168 * 17 // 32  # 2.92 MB
    assert per_expert == 2_924_544
    assert gemm == 33 * per_expert + 16 * 7168 * 17 // 32
    assert total == 33 * per_expert + 2 * 16 * 7168 * 2 + 16 * 3 * 8
    _, gemm_bf16, _ = bench.alg_bytes(w, ids, bf16_act=True)
    assert gemm_bf16 == 33 * per_expert + 16 * 7168 * 2


def test_kernel_code_hash_ignores_comments_only():
    """The hash that ties a committed ncu summary to the GEMM sources changes with
    the code and not with comments or spacing."""
    import bench

    code = "int f(int a) {\n  return a + 1;  // one\n}\n/* block\n comment */\n"
    same = "int f(int a) { return a + 1; }\n// another comment\n"
    other = "int f(int a) { return a + 2; }\n"
    assert bench._code_only(code) == bench._code_only(same)
    assert bench._code_only(code) != bench._code_only(other)
