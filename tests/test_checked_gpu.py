"""The bounds-checked build (compiled with MOE_CHECKED=1: every sorted-slot index,
route-tile field and tensor-memory column on the GEMM path checked before use)
runs the main launch paths -- separate kernels and the single launch, narrow and
128-route tiles, routing on many CTAs, multi-stage contractions, padded storage
and the dense shard -- with a clean device status word, and gives the product
build's outputs bit for bit (the checks change no arithmetic).  Each build runs
in a process of its own (the binding loads one library per process)."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _run(lib, out):
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_runner.py"), lib, out],
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return torch.load(out)


def test_checked_build_matches_product_build(tmp_path):
    from mixture_experts_mxfp4_gb300 import build

    product = build.build()
    checked = build.build(checked=True)
    a = _run(product, str(tmp_path / "product.pt"))
    b = _run(checked, str(tmp_path / "checked.pt"))
    assert "bounds-checked" in b["version"] and "bounds-checked" not in a["version"]
    names = [k for k in a if k != "version"]
    assert len(names) >= 9
    for name in names:
        out_a, st_a, dev_a = a[name]
        out_b, st_b, dev_b = b[name]
        assert st_b == 0 and dev_b == 0, f"{name}: checked build status word {st_b:#x}"
        assert st_a == 0 and dev_a == 0, name
        assert torch.equal(out_a, out_b), name
