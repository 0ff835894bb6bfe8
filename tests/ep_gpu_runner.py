"""Expert-parallel forward on one GPU through a one-rank NCCL process group, with
the library as each rank's local forward, against the library's own forward
(helper of test_ep_gpu.py; runs in a process of its own).

    python tests/ep_gpu_runner.py PORT
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

import mixture_experts_mxfp4_gb300 as moe  # noqa: E402
import workloads  # noqa: E402
from mixture_experts_mxfp4_gb300 import ep  # noqa: E402

CASES = [(16, 256, 128, 9, 3), (16, 7168, 256, 257, 9), (96, 512, 256, 5, 3)]


def main(port):
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        moe.load_library()
        dev = torch.device("cuda", 0)
        for case in CASES:
            T, D, I, E, K = case
            w = workloads.custom(T, D, I, E, K)
            inp = workloads.make_inputs(w, seed=21)
            inp["topk_ids"][0, 0] = -1
            t = {k: v.to(dev) for k, v in inp.items()}
            ref = moe.MoeMXFP4(T, D, I, E, K).forward(t["hidden"], t["w13"], t["w13_scale"], t["w2"],
                                                      t["w2_scale"], t["topk_ids"], t["topk_weights"])
            first, count = ep.expert_ranges(E, 1)[0]
            local = ep.library_local_forward(t["w13"], t["w13_scale"], t["w2"], t["w2_scale"], first, count)
            out = ep.ep_forward(t["hidden"], t["topk_ids"], t["topk_weights"], E, local)
            torch.cuda.synchronize()
            if not torch.equal(out.view(torch.int16), ref.view(torch.int16)):
                raise SystemExit(f"case {case}: expert-parallel forward differs from the forward")
        print("ok")
    finally:
        dist.destroy_process_group()


if __name__ == "__main__":
    main(int(sys.argv[1]))
