"""The oracle's pins catch plausible mistakes: each case plants one mistake in a
copy of oracle/moe_oracle.c (on the CPU), builds it, and runs the oracle's pin
suite (tests/test_oracle.py) against that build, which must fail.  The control
case builds the unchanged source the same way and must pass."""
import os
import shutil
import subprocess
import sys

import pytest

from conftest import ROOT

ORACLE = os.path.join(ROOT, "oracle")

# name -> (text in moe_oracle.c, replacement): each a one-line slip
MUTANTS = {
    "control": None,
    "gate_and_up_swapped": ("float s = g / (1.0f + expf(-g));\n                float v = s * u;",
                            "float s = u / (1.0f + expf(-u));\n                float v = s * g;"),
    "silu_dropped": ("float s = g / (1.0f + expf(-g));", "float s = g;"),
    "silu_sign_flipped": ("float s = g / (1.0f + expf(-g));", "float s = g / (1.0f + expf(g));"),
    "nibble_order_swapped": ("int nib = (j & 1) ? (byte >> 4) & 15 : byte & 15;",
                             "int nib = (j & 1) ? byte & 15 : (byte >> 4) & 15;"),
    "neighbouring_block_scale": ("g_e8m0[scales[j / 32]]", "g_e8m0[scales[(j / 32) ^ 1]]"),
    "e2m1_sign_dropped": ("return sign ? -mag : mag;", "return mag;"),
    "e2m1_subnormal_wrong": ("mag = 0.5f * (float)mant;", "mag = 1.0f * (float)mant;"),
    "shared_exponent_off_by_one": ("X = (e - 1) - 2;", "X = (e - 1) - 1;"),
    "intermediate_not_bf16": ("hv[n] = moe_oracle_bf16_value(moe_oracle_bf16_bits(v));", "hv[n] = v;"),
    "intermediate_not_requantised": ("if (quant_act) {\n                moe_oracle_quant_row(hv, I, qc, qs);",
                                     "if (0) {\n                moe_oracle_quant_row(hv, I, qc, qs);"),
    "topk_weight_dropped": ("float wk = topk_w[r];", "float wk = 1.0f;"),
    "hidden_not_quantised": ("if (quant_act) {\n            moe_oracle_quant_row(x, D, qc, qs);",
                             "if (0) {\n            moe_oracle_quant_row(x, D, qc, qs);"),
    "e8m0_bias_off_by_one": ("return ldexpf(1.0f, s - 127);", "return ldexpf(1.0f, s - 128);"),
    "routes_in_descending_order": ("for (int r = 0; r < R; ++r) {\n            if (topk_ids[r] == e) {",
                                   "for (int r = R - 1; r >= 0; --r) {\n            if (topk_ids[r] == e) {"),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    gcc = shutil.which("gcc") or pytest.skip("no C compiler")
    src = open(os.path.join(ORACLE, "moe_oracle.c")).read()
    if MUTANTS[name] is not None:
        old, new = MUTANTS[name]
        assert src.count(old) == 1, f"mutation site not unique: {old!r}"
        src = src.replace(old, new)
    shutil.copy(os.path.join(ORACLE, "moe_oracle.h"), tmp_path / "moe_oracle.h")
    (tmp_path / "moe_oracle.c").write_text(src)
    lib = tmp_path / "libmoe_oracle_mutant.so"
    subprocess.run([gcc, "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                    "-fPIC", "-shared", str(tmp_path / "moe_oracle.c"), "-o", str(lib), "-lm"],
                   check=True)
    env = dict(os.environ, MOE_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle.py"),
                        "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    if MUTANTS[name] is None:
        assert r.returncode == 0, r.stdout[-3000:]
    else:
        assert r.returncode == 1, f"the pins did not catch '{name}':\n{r.stdout[-2000:]}"
