"""Run forward calls with one build of the library and save outputs and device
statuses (helper of test_checked_gpu.py; one library per process).

    python tests/checked_runner.py LIB OUT.pt
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import mixture_experts_mxfp4_gb300 as moe  # noqa: E402
import workloads  # noqa: E402

# (name, T, D, I, E, K, launch mode, padded storage (Dp, Ip) or None)
CASES = [
    ("tiny_separate", 16, 256, 128, 9, 3, 0, None),
    ("tiny_single", 16, 256, 128, 9, 3, 1, None),
    ("decode_T16", 16, 7168, 256, 257, 9, 2, None),
    ("decode_T128", 128, 7168, 256, 257, 9, 2, None),
    ("tiles128", 256, 512, 256, 5, 3, 2, None),
    ("multi_cta_routing", 820, 256, 128, 9, 5, 2, None),
    ("multi_stage", 64, 1024, 512, 3, 2, 2, None),
    ("padded", 40, 992, 416, 9, 3, 2, (1024, 512)),
    ("dense_T512", 512, 7168, 2048, 33, 9, 2, None),
]


def run(lib_path, out_path):
    moe.load_library(lib_path)
    dev = torch.device("cuda")
    res = {"version": moe.version()}
    for name, T, D, I, E, K, mode, pad in CASES:
        w = workloads.custom(T, D, I, E, K)
        inp = workloads.make_inputs(w, seed=13)
        if pad is not None:
            from test_parity_gpu import _padded_weights

            inp = _padded_weights(inp, *pad)
        moe.set_single_launch(mode)
        m = moe.MoeMXFP4(T, D, I, E, K, d_model_pad=pad[0] if pad else None,
                         d_inter_pad=pad[1] if pad else None)
        t = {k: v.to(dev) for k, v in inp.items()}
        out = m.forward(t["hidden"], t["w13"], t["w13_scale"], t["w2"], t["w2_scale"],
                        t["topk_ids"], t["topk_weights"])
        torch.cuda.synchronize()
        status = int(m.region("status", torch.int32, (16,)).cpu()[0])
        res[name] = (out.view(torch.int16).cpu(), status, m.device_status())
    moe.set_single_launch(2)
    torch.save(res, out_path)


if __name__ == "__main__":
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    run(sys.argv[1], sys.argv[2])
