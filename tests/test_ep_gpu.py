"""Expert-parallel dispatch and combine on the GPU: a one-rank NCCL process group
(the GPU machines here have one GPU), the library as the local forward with one
route per row; the result must equal the library's forward bit for bit (the
library's P rows do not depend on which routes share a tile, and the combine
adds them in the top-k sum kernel's order)."""
import os
import socket
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_ep_forward_one_rank_nccl_matches_forward():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    r = subprocess.run([sys.executable, os.path.join(HERE, "ep_gpu_runner.py"), str(port)],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
