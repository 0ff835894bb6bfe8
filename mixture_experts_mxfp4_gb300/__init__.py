"""Fused MXFP4 Mixture-of-Experts forward for NVIDIA GB300 (sm_103a).

Thin Python binding over the C ABI in ``include/moe_mxfp4.h`` (ctypes, argument
marshalling only).  Every step of the forward runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback: if the library is missing or a
call fails, an exception is raised.

    import torch, mixture_experts_mxfp4_gb300 as moe
    m = moe.MoeMXFP4(T, d_model, d_inter, E, topk)        # owns its workspace
    out = m.forward(hidden, w13, w13_scale, w2, w2_scale, topk_ids, topk_weights)
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmoe_mxfp4.so")
# bounds-checked variant (build.build(checked=True)): same ABI, test aid
CHECKED_LIB_PATH = os.path.join(_PKG, "_lib", "libmoe_mxfp4_checked.so")

STATUS = {
    0: "MOE_OK",
    1: "MOE_ERR_INVALID_ARG",
    2: "MOE_ERR_UNSUPPORTED_SHAPE",
    3: "MOE_ERR_MISALIGNED",
    4: "MOE_ERR_WORKSPACE",
    5: "MOE_ERR_CUDA",
    6: "MOE_ERR_DEVICE_TIMEOUT",
}
MOE_OK = 0

REGIONS = ["status", "counters", "sorted_ids", "sorted_w", "block_expert", "seg_start",
           "route_pos", "num_valid", "tiles", "a1q", "a1s", "a2q", "a2s", "P", "partial",
           "a1b", "a2b", "wscale"]

# Exported C symbols (kept in step with include/moe_mxfp4.h).
EXPORTS = [
    "moe_mxfp4_workspace_size",
    "moe_mxfp4_set_workspace",
    "moe_mxfp4_forward",
    "moe_mxfp4_status_string",
    "moe_mxfp4_last_device_status",
    "moe_mxfp4_get_plan",
    "moe_mxfp4_get_gemm_config",
    "moe_mxfp4_topk_sum",
    "moe_mxfp4_version",
    "moe_mxfp4_num_kernels",
    "moe_mxfp4_set_kernel_timing",
    "moe_mxfp4_set_nvtx",
    "moe_mxfp4_kernel_times",
    "moe_mxfp4_last_call_ms",
    "moe_mxfp4_forward_noalloc",
    "moe_mxfp4_check_wait_timeout",
    "moe_mxfp4_set_single_launch",
    "moe_mxfp4_call_launches",
    "moe_mxfp4_forward_padded",
    "moe_mxfp4_forward_w4a16",
    "moe_mxfp4_workspace_size_w4a16",
    "moe_mxfp4_get_plan_w4a16",
    "moe_mxfp4_pointer_kind",
    "moe_mxfp4_set_tuning",
    "moe_mxfp4_tensor_probe",
]

# Size of the library's static scratch array used by moe_mxfp4_forward_noalloc.
STATIC_WORKSPACE_BYTES = 64 << 20

KERNEL_NAMES = ["route", "quant", "gemm", "topk_sum"]


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, code)}")
        self.code = code


class Plan(ctypes.Structure):
    _fields_ = [
        ("block_m", ctypes.c_int),
        ("tile_rows", ctypes.c_int),
        ("cap", ctypes.c_int),
        ("a1s_stride", ctypes.c_int),
        ("a2s_stride", ctypes.c_int),
        ("stage1_splits", ctypes.c_int),
        ("max_tiles", ctypes.c_int),
        ("bf16_act", ctypes.c_int),
        ("d_model_run", ctypes.c_int),
        ("d_inter_run", ctypes.c_int),
        ("offset", ctypes.c_size_t * len(REGIONS)),
        ("bytes", ctypes.c_size_t * len(REGIONS)),
        ("workspace_bytes", ctypes.c_size_t),
    ]

    def region(self, name: str):
        i = REGIONS.index(name)
        return int(self.offset[i]), int(self.bytes[i])


class GemmConfig(ctypes.Structure):
    """moe_mxfp4_gemm_config_t: launch geometry of the fused GEMM kernel."""
    _fields_ = [(n, ctypes.c_int) for n in (
        "tile_rows", "stage1_k", "stage2_k", "stage2_blocks", "num_stages", "mma_warps", "acc_bufs",
        "epi_groups", "sf_by_layout_warp", "wide_sf", "lookahead")] + \
        [(n, ctypes.c_uint) for n in (
            "slot_bytes", "smem_bytes", "smem_limit", "acc_cols", "sf_col0", "sf_cols", "tmem_cols")]

    def as_dict(self):
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libmoe_mxfp4.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} not found: build it with mixture_experts_mxfp4_gb300/build.py")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i = ctypes.c_int
    lib.moe_mxfp4_workspace_size.restype = ctypes.c_size_t
    lib.moe_mxfp4_workspace_size.argtypes = [i, i, i, i, i]
    lib.moe_mxfp4_set_workspace.restype = i
    lib.moe_mxfp4_set_workspace.argtypes = [P, ctypes.c_size_t]
    lib.moe_mxfp4_forward.restype = i
    lib.moe_mxfp4_forward.argtypes = [P, P, P, P, P, P, P, P, i, i, i, i, i, P]
    lib.moe_mxfp4_forward_padded.restype = i
    lib.moe_mxfp4_forward_padded.argtypes = [P, P, P, P, P, P, P, P, i, i, i, i, i, i, i, P]
    lib.moe_mxfp4_status_string.restype = ctypes.c_char_p
    lib.moe_mxfp4_status_string.argtypes = [i]
    lib.moe_mxfp4_last_device_status.restype = i
    lib.moe_mxfp4_last_device_status.argtypes = [P]
    lib.moe_mxfp4_get_plan.restype = i
    lib.moe_mxfp4_get_plan.argtypes = [i, i, i, i, i, ctypes.POINTER(Plan)]
    lib.moe_mxfp4_topk_sum.restype = i
    lib.moe_mxfp4_topk_sum.argtypes = [P, P, P, i, i, i, P]
    lib.moe_mxfp4_get_gemm_config.restype = i
    lib.moe_mxfp4_get_gemm_config.argtypes = [i, i, i, i, i, ctypes.POINTER(GemmConfig)]
    lib.moe_mxfp4_get_plan_w4a16.restype = i
    lib.moe_mxfp4_get_plan_w4a16.argtypes = [i, i, i, i, i, ctypes.POINTER(Plan)]
    lib.moe_mxfp4_workspace_size_w4a16.restype = ctypes.c_size_t
    lib.moe_mxfp4_workspace_size_w4a16.argtypes = [i, i, i, i, i]
    lib.moe_mxfp4_forward_w4a16.restype = i
    lib.moe_mxfp4_forward_w4a16.argtypes = [P, P, P, P, P, P, P, P, i, i, i, i, i, P]
    lib.moe_mxfp4_version.restype = ctypes.c_char_p
    lib.moe_mxfp4_version.argtypes = []
    lib.moe_mxfp4_pointer_kind.restype = i
    lib.moe_mxfp4_pointer_kind.argtypes = [P]
    lib.moe_mxfp4_num_kernels.restype = i
    lib.moe_mxfp4_num_kernels.argtypes = []
    lib.moe_mxfp4_set_kernel_timing.restype = i
    lib.moe_mxfp4_set_kernel_timing.argtypes = [i]
    lib.moe_mxfp4_set_nvtx.restype = i
    lib.moe_mxfp4_set_nvtx.argtypes = [i]
    lib.moe_mxfp4_set_single_launch.restype = i
    lib.moe_mxfp4_set_single_launch.argtypes = [i]
    lib.moe_mxfp4_set_tuning.restype = i
    lib.moe_mxfp4_set_tuning.argtypes = [i, i]
    lib.moe_mxfp4_tensor_probe.restype = i
    lib.moe_mxfp4_tensor_probe.argtypes = [i, i, i, i, ctypes.POINTER(ctypes.c_double), P]
    lib.moe_mxfp4_call_launches.restype = i
    lib.moe_mxfp4_call_launches.argtypes = [i, i, i, i, i]
    lib.moe_mxfp4_kernel_times.restype = i
    lib.moe_mxfp4_kernel_times.argtypes = [ctypes.POINTER(ctypes.c_float), i]
    lib.moe_mxfp4_last_call_ms.restype = ctypes.c_float
    lib.moe_mxfp4_last_call_ms.argtypes = []
    lib.moe_mxfp4_check_wait_timeout.restype = i
    lib.moe_mxfp4_check_wait_timeout.argtypes = [ctypes.c_uint32, P]
    lib.moe_mxfp4_forward_noalloc.restype = i
    lib.moe_mxfp4_forward_noalloc.argtypes = [P, P, P, P, P, P, P, P, i, i, i, i, i, P]
    _lib = lib
    return lib


def _check(code: int, where: str):
    if code != MOE_OK:
        raise MoeError(code, where)


def workspace_size(T, d_model, d_inter, E, topk) -> int:
    return int(load_library().moe_mxfp4_workspace_size(T, d_model, d_inter, E, topk))


def get_plan(T, d_model, d_inter, E, topk) -> Plan:
    pl = Plan()
    _check(load_library().moe_mxfp4_get_plan(T, d_model, d_inter, E, topk, ctypes.byref(pl)),
           "moe_mxfp4_get_plan")
    return pl


def topk_sum_ptr(P_ptr, route_pos_ptr, out_ptr, T, d_model, topk, stream=0) -> int:
    """moe_mxfp4_topk_sum on raw pointers; returns the status code."""
    return int(load_library().moe_mxfp4_topk_sum(ctypes.c_void_p(P_ptr), ctypes.c_void_p(route_pos_ptr),
                                                 ctypes.c_void_p(out_ptr), T, d_model, topk,
                                                 ctypes.c_void_p(stream)))


def topk_sum(P, route_pos, out):
    """Deterministic top-k sum (moe_mxfp4_topk_sum) of P (f32 [T*topk, d_model],
    rows by route id) over the routes with route_pos >= 0 (int32 [T*topk]) into
    out (bf16 [T, d_model]), on the current stream.  The tensors must be
    contiguous and on the device."""
    import torch

    R, D = P.shape
    T = out.shape[0]
    if T == 0:
        return out
    if R % T != 0 or route_pos.numel() != R or out.shape[1] != D:
        raise ValueError("P [T*topk, d_model], route_pos [T*topk], out [T, d_model]")
    for x, dt in ((P, torch.float32), (route_pos, torch.int32), (out, torch.bfloat16)):
        if x.dtype != dt or not x.is_contiguous():
            raise ValueError("P f32, route_pos int32, out bf16, all contiguous")
    stream = torch.cuda.current_stream(out.device).cuda_stream
    _check(topk_sum_ptr(P.data_ptr(), route_pos.data_ptr(), out.data_ptr(), T, D, R // T, stream),
           "moe_mxfp4_topk_sum")
    return out


def gemm_config(T, d_model, d_inter, E, topk) -> GemmConfig:
    """Launch geometry of the fused GEMM kernel for this shape (host only)."""
    cfg = GemmConfig()
    _check(load_library().moe_mxfp4_get_gemm_config(T, d_model, d_inter, E, topk, ctypes.byref(cfg)),
           "moe_mxfp4_get_gemm_config")
    return cfg


def get_plan_w4a16(T, d_model, d_inter, E, topk) -> Plan:
    """Workspace layout of the bf16-activation (W4A16) forward."""
    pl = Plan()
    _check(load_library().moe_mxfp4_get_plan_w4a16(T, d_model, d_inter, E, topk, ctypes.byref(pl)),
           "moe_mxfp4_get_plan_w4a16")
    return pl


def forward_w4a16_ptr(hidden, w13, w13_scale, w2, w2_scale, topk_ids, topk_weights, out,
                      T, d_model, d_inter, E, topk, stream: int = 0) -> int:
    """Raw-pointer call of moe_mxfp4_forward_w4a16; returns the status code."""
    return int(load_library().moe_mxfp4_forward_w4a16(
        ctypes.c_void_p(hidden), ctypes.c_void_p(w13), ctypes.c_void_p(w13_scale),
        ctypes.c_void_p(w2), ctypes.c_void_p(w2_scale), ctypes.c_void_p(topk_ids),
        ctypes.c_void_p(topk_weights), ctypes.c_void_p(out), T, d_model, d_inter, E, topk,
        ctypes.c_void_p(stream)))


def set_workspace(ptr: int, nbytes: int):
    _check(load_library().moe_mxfp4_set_workspace(ctypes.c_void_p(ptr), nbytes),
           "moe_mxfp4_set_workspace")


def forward_padded_ptr(hidden, w13, w13_scale, w2, w2_scale, topk_ids, topk_weights, out,
                       T, d_model, d_inter, d_model_pad, d_inter_pad, E, topk,
                       stream: int = 0) -> int:
    """Raw-pointer call of moe_mxfp4_forward_padded; returns the status code."""
    return int(load_library().moe_mxfp4_forward_padded(
        ctypes.c_void_p(hidden), ctypes.c_void_p(w13), ctypes.c_void_p(w13_scale),
        ctypes.c_void_p(w2), ctypes.c_void_p(w2_scale), ctypes.c_void_p(topk_ids),
        ctypes.c_void_p(topk_weights), ctypes.c_void_p(out), T, d_model, d_inter,
        d_model_pad, d_inter_pad, E, topk, ctypes.c_void_p(stream)))


def forward_ptr(hidden, w13, w13_scale, w2, w2_scale, topk_ids, topk_weights, out,
                T, d_model, d_inter, E, topk, stream: int = 0) -> int:
    """Raw-pointer call of moe_mxfp4_forward; returns the status code."""
    return int(load_library().moe_mxfp4_forward(
        ctypes.c_void_p(hidden), ctypes.c_void_p(w13), ctypes.c_void_p(w13_scale),
        ctypes.c_void_p(w2), ctypes.c_void_p(w2_scale), ctypes.c_void_p(topk_ids),
        ctypes.c_void_p(topk_weights), ctypes.c_void_p(out), T, d_model, d_inter, E, topk,
        ctypes.c_void_p(stream)))


def forward_noalloc_ptr(hidden, w13, w13_scale, w2, w2_scale, topk_ids, topk_weights, out,
                        T, d_model, d_inter, E, topk, stream: int = 0) -> int:
    """Raw-pointer call of moe_mxfp4_forward_noalloc (no workspace, nothing
    allocated: the scratch is a static array inside the library); returns the
    status code."""
    return int(load_library().moe_mxfp4_forward_noalloc(
        ctypes.c_void_p(hidden), ctypes.c_void_p(w13), ctypes.c_void_p(w13_scale),
        ctypes.c_void_p(w2), ctypes.c_void_p(w2_scale), ctypes.c_void_p(topk_ids),
        ctypes.c_void_p(topk_weights), ctypes.c_void_p(out), T, d_model, d_inter, E, topk,
        ctypes.c_void_p(stream)))


def check_wait_timeout(limit_us: int, stream: int = 0) -> int:
    """Enqueue the bounded-wait self-check (see include/moe_mxfp4.h); status code."""
    return int(load_library().moe_mxfp4_check_wait_timeout(int(limit_us), ctypes.c_void_p(stream)))


def last_device_status(stream: int = 0) -> int:
    return int(load_library().moe_mxfp4_last_device_status(ctypes.c_void_p(stream)))


def set_single_launch(mode):
    """Launch mode: 0 separate kernels; 1 route and quantise inside the GEMM kernel
    wherever the shape allows; 2 (default) single launch for decode-sized calls."""
    _check(load_library().moe_mxfp4_set_single_launch(int(mode)), "moe_mxfp4_set_single_launch")


def set_tuning(tile_rows=0, sf_copies=0):
    """Tuning override: route-tile width (16/32/64/128) and scale-factor copy
    scheme (1 MMA warps, 2 separate warp, 3 separate warp with two-chunk copies);
    0 the library's choice."""
    _check(load_library().moe_mxfp4_set_tuning(int(tile_rows), int(sf_copies)), "moe_mxfp4_set_tuning")


def tensor_probe(n, iters, copies_per_mma=0, variant=0, stream: int = 0) -> float:
    """Enqueue the MXFP4 tensor-core throughput probe (needs a registered
    workspace); returns the operation count of the enqueued kernel."""
    fl = ctypes.c_double(0.0)
    _check(load_library().moe_mxfp4_tensor_probe(int(n), int(iters), int(copies_per_mma),
                                                  int(variant), ctypes.byref(fl),
                                                  ctypes.c_void_p(stream)),
           "moe_mxfp4_tensor_probe")
    return float(fl.value)


def call_launches(T, d_model, d_inter, E, topk) -> int:
    """Kernels one forward call of this shape launches under the current launch mode."""
    return int(load_library().moe_mxfp4_call_launches(T, d_model, d_inter, E, topk))


def set_nvtx(on: bool):
    """NVTX ranges around every forward call and kernel launch (off by default)."""
    _check(load_library().moe_mxfp4_set_nvtx(1 if on else 0), "moe_mxfp4_set_nvtx")


def set_kernel_timing(mode):
    """0 off, 1 events around every kernel, 2 events around the whole call only."""
    _check(load_library().moe_mxfp4_set_kernel_timing(int(mode)), "moe_mxfp4_set_kernel_timing")


def last_call_ms() -> float:
    """Device time (ms) of the last forward call on this device (timing mode 1 or 2)."""
    t = float(load_library().moe_mxfp4_last_call_ms())
    if t < 0:
        raise MoeError(5, "moe_mxfp4_last_call_ms")
    return t


def kernel_times():
    """Per-kernel durations (ms) of the last forward call on this device, by name
    (None for a slot in which the call launched nothing)."""
    lib = load_library()
    n = lib.moe_mxfp4_num_kernels()
    buf = (ctypes.c_float * n)()
    got = lib.moe_mxfp4_kernel_times(buf, n)
    if got < 0:
        raise MoeError(5, "moe_mxfp4_kernel_times")
    return {KERNEL_NAMES[i]: (float(buf[i]) if buf[i] >= 0 else None) for i in range(got)}


def version() -> str:
    return load_library().moe_mxfp4_version().decode()


_MAPPED = {}


def _host_mapped(ptr: int, device) -> bool:
    """The device reads and writes this pinned host address at the same pointer
    (moe_mxfp4_pointer_kind == 1); remembered per (device, address)."""
    import torch

    key = (device.index, ptr)
    if key not in _MAPPED:
        with torch.cuda.device(device):
            _MAPPED[key] = load_library().moe_mxfp4_pointer_kind(ctypes.c_void_p(ptr)) == 1
        if len(_MAPPED) > 4096:
            _MAPPED.clear()
    return _MAPPED[key]


class MoeMXFP4:
    """One MoE layer shape with its own device workspace (a torch uint8 tensor).

    The workspace is registered for the current device on every call, so several
    instances can coexist as long as their calls are ordered on the GPU.  With
    d_model_pad / d_inter_pad the weights are stored with those padded sizes
    (moe_mxfp4_forward_padded); hidden and out keep d_model columns.  With
    activations="bf16" the forward keeps the activations in bf16 (W4A16,
    moe_mxfp4_forward_w4a16).  hidden, topk_ids, topk_weights and out may be
    pinned host tensors: the kernels read and write them in place.
    """

    def __init__(self, T, d_model, d_inter, E, topk, device="cuda", d_model_pad=None,
                 d_inter_pad=None, activations="mxfp4"):
        import torch

        if activations not in ("mxfp4", "bf16"):
            raise ValueError("activations must be 'mxfp4' or 'bf16'")
        self.shape = (T, d_model, d_inter, E, topk)
        self.pad = (d_model_pad or d_model, d_inter_pad or d_inter)
        self.bf16_act = activations == "bf16"
        if self.bf16_act and self.pad != (d_model, d_inter):
            raise ValueError("padded storage is not available with bf16 activations")
        self.plan = (get_plan_w4a16 if self.bf16_act else get_plan)(T, self.pad[0], self.pad[1], E,
                                                                       topk)
        n = max(int(self.plan.workspace_bytes), 256)
        # zero-filled: the status region must start at zero (the calls keep it so)
        self.workspace = torch.zeros(n + 256, dtype=torch.uint8, device=device)
        base = self.workspace.data_ptr()
        self.ws_ptr = (base + 255) // 256 * 256
        self.ws_bytes = n

    def region(self, name: str, dtype, shape):
        """A torch view of one workspace region (for inspection in tests)."""
        import torch

        off, nbytes = self.plan.region(name)
        start = self.ws_ptr - self.workspace.data_ptr() + off
        elem = torch.empty((), dtype=dtype).element_size()
        count = 1
        for s in shape:
            count *= s
        assert count * elem <= nbytes or nbytes == 0
        return self.workspace[start:start + count * elem].view(dtype).view(*shape)

    def forward(self, hidden, w13, w13_scale, w2, w2_scale, topk_ids, topk_weights, out=None,
                stream=None):
        import torch

        T, D, I, E, K = self.shape
        if out is None:
            out = torch.empty((T, D), dtype=torch.bfloat16, device=hidden.device,
                              pin_memory=not hidden.is_cuda)
        for t in (w13, w13_scale, w2, w2_scale):
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError("weights and scales must be contiguous CUDA tensors")
        # the per-call tensors may also live in pinned host memory, which the
        # kernels read and write in place (mapped into the device's address space)
        for t in (hidden, topk_ids, topk_weights, out):
            if not t.is_contiguous() or not (t.is_cuda or t.is_pinned()):
                raise ValueError("hidden, topk_ids, topk_weights and out must be contiguous "
                                 "CUDA tensors or pinned host tensors")
            if t.is_cuda and t.device != w13.device:
                raise ValueError("all CUDA tensors must be on the weights' device")
            if not t.is_cuda and t.numel() and not _host_mapped(t.data_ptr(), w13.device):
                raise ValueError("a pinned host tensor that the device cannot address at "
                                 "the same pointer")
        if hidden.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
            raise ValueError("hidden and out must be bfloat16")
        if topk_ids.dtype != torch.int32 or topk_weights.dtype != torch.float32:
            raise ValueError("topk_ids must be int32 and topk_weights float32")
        if stream is None:
            stream = torch.cuda.current_stream(w13.device).cuda_stream
        set_workspace(self.ws_ptr, self.ws_bytes)
        if self.bf16_act:
            code = forward_w4a16_ptr(hidden.data_ptr(), w13.data_ptr(), w13_scale.data_ptr(),
                                     w2.data_ptr(), w2_scale.data_ptr(), topk_ids.data_ptr(),
                                     topk_weights.data_ptr(), out.data_ptr(), T, D, I, E, K, stream)
            _check(code, "moe_mxfp4_forward_w4a16")
        elif self.pad == (D, I):
            code = forward_ptr(hidden.data_ptr(), w13.data_ptr(), w13_scale.data_ptr(),
                               w2.data_ptr(), w2_scale.data_ptr(), topk_ids.data_ptr(),
                               topk_weights.data_ptr(), out.data_ptr(), T, D, I, E, K, stream)
            _check(code, "moe_mxfp4_forward")
        else:
            code = forward_padded_ptr(hidden.data_ptr(), w13.data_ptr(), w13_scale.data_ptr(),
                                      w2.data_ptr(), w2_scale.data_ptr(), topk_ids.data_ptr(),
                                      topk_weights.data_ptr(), out.data_ptr(), T, D, I,
                                      self.pad[0], self.pad[1], E, K, stream)
            _check(code, "moe_mxfp4_forward_padded")
        return out

    def device_status(self, stream=None) -> int:
        import torch

        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        set_workspace(self.ws_ptr, self.ws_bytes)
        return last_device_status(stream)
