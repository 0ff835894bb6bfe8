"""moe_mxfp4_forward_noalloc: the forward call for callers that cannot allocate
device memory (for example a serving runtime that has given all free device
memory to its own pool, or a plugin host that forbids allocation).  Instead of
a caller-owned workspace it uses a static scratch array inside the library.

Checked here through the C ABI: two calls in a row give the regular
moe_mxfp4_forward's output bit for bit (same kernels, same inputs) and leave a
clean status word in the array; the multi-kernel path (decode batch T = 128) is
covered as well as the single launch; a sequence of different shapes and launch
paths on the shared array, ending with the first shape again, gives each
shape's regular output; a T = 0 call only does the per-device set-up; a shape
whose workspace does not fit the array is rejected before any work.
This file is collected last so that a failure here never hides another test.
"""
import pytest
import torch

import workloads


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_mxfp4_gb300 import build

    build.build()
    import mixture_experts_mxfp4_gb300 as m

    m.load_library()
    return m


def test_oversized_shape_is_rejected(moe):
    w = workloads.WORKLOADS["prefill_zipf_T4096_D7168_I256_E257_K9"]
    assert moe.workspace_size(w.T, w.D, w.I, w.E, w.K) > moe.STATIC_WORKSPACE_BYTES
    fake = 1 << 20  # never dereferenced: the size check comes first
    code = moe.forward_noalloc_ptr(fake, fake, fake, fake, fake, fake, fake, fake,
                                   w.T, w.D, w.I, w.E, w.K, 0)
    assert code == 4  # MOE_ERR_WORKSPACE


class _Case:
    """Device inputs of one workload and its output from the regular forward."""

    def __init__(self, moe, name, seed=0):
        self.w = w = workloads.WORKLOADS[name]
        assert moe.workspace_size(w.T, w.D, w.I, w.E, w.K) <= moe.STATIC_WORKSPACE_BYTES
        inp = workloads.make_inputs(w, seed=seed)
        t = {k: v.cuda() for k, v in inp.items()}
        self.args = (t["hidden"], t["w13"], t["w13_scale"], t["w2"], t["w2_scale"],
                     t["topk_ids"], t["topk_weights"])
        m = moe.MoeMXFP4(w.T, w.D, w.I, w.E, w.K)
        self.ref = m.forward(*self.args).clone()
        torch.cuda.synchronize()
        assert m.device_status() == 0

    def noalloc(self, moe):
        w = self.w
        stream = torch.cuda.current_stream().cuda_stream
        out = torch.full((w.T, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        code = moe.forward_noalloc_ptr(*(x.data_ptr() for x in self.args), out.data_ptr(),
                                       w.T, w.D, w.I, w.E, w.K, stream)
        assert code == 0, moe.STATUS.get(code, code)
        # synchronises, then reads the status word of the array this call used
        assert moe.last_device_status(stream) == 0
        return out

    def check(self, out):
        assert torch.equal(out.view(torch.int16), self.ref.view(torch.int16))


@pytest.mark.gpu
@pytest.mark.parametrize("name", [workloads.TINY, workloads.DECODE_T16,
                                  "decode_T128_D7168_I256_E257_K9"])
def test_noalloc_matches_forward_twice(moe, name):
    w = workloads.WORKLOADS[name]
    # T = 0: the per-device set-up only (nothing is enqueued, pointers unused)
    assert moe.forward_noalloc_ptr(0, 0, 0, 0, 0, 0, 0, 0, 0, w.D, w.I, w.E, w.K, 0) == 0
    c = _Case(moe, name)
    for _ in range(2):
        c.check(c.noalloc(moe))


@pytest.mark.gpu
def test_noalloc_alternating_shapes(moe):
    """Shapes and launch paths alternate on the one shared array (separate kernels
    at T = 128, single launch at T = 16 and the tiny case), then the first shape
    runs again: every call matches its shape's regular forward bit for bit."""
    cases = [_Case(moe, n, seed=3) for n in ("decode_T128_D7168_I256_E257_K9",
                                               workloads.DECODE_T16, workloads.TINY)]
    for c in cases + [cases[1], cases[0], cases[2], cases[0]]:
        c.check(c.noalloc(moe))
