"""Python binding of the GB300 MoE expert-layer library (libmoe_gb300.so).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (PyTorch provides device memory
and streams); the functions carry the C ABI's names and argument order
(include/moe.h) and raise MoEError on a non-zero status.  There is no CPU
fallback: importing works without a GPU, but every call needs the built
library and a compute capability 10.3 device.
"""
from __future__ import annotations

import ctypes
import os

__all__ = ["MoEError", "MoEShape", "MoEViews", "lib_path", "load", "shape", "capacity",
           "workspace_size", "alloc_workspace", "workspace_init", "workspace_views",
           "last_device_status", "check_wait_timeout", "alloc_route_outputs", "moe_route",
           "moe_grouped_gemm_up", "moe_grouped_gemm_up_rows", "moe_grouped_gemm_down", "moe_combine",
           "moe_forward", "STATUS_NAMES", "EXPORTS", "FORWARD_KERNELS"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE",
                3: "MOE_ERR_MISALIGNED", 4: "MOE_ERR_ARCH", 5: "MOE_ERR_CUDA",
                6: "MOE_ERR_TIMEOUT", 7: "MOE_ERR_DEVICE_BOUNDS", 8: "MOE_ERR_SCRATCH_LIMIT"}

# kernels one moe_forward launches: the routing kernel, the permutation with the
# row gather, the gate/up and down GEMMs, the combine
FORWARD_KERNELS = 5

# every function include/moe.h declares
EXPORTS = ["moe_status_string", "moe_capacity", "moe_workspace_size", "moe_workspace_init",
           "moe_last_device_status", "moe_route", "moe_grouped_gemm_up", "moe_grouped_gemm_down",
           "moe_combine", "moe_forward", "moe_workspace_views", "moe_route_noalloc",
           "moe_grouped_gemm_up_rows", "moe_check_wait_timeout"]


class MoEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s" % (where, STATUS_NAMES.get(code, "status %d" % code)))


class MoEShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32)]


class MoEViews(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("topk_ids", "topk_w", "counts", "off_pad",
                                                "block_expert", "num_blocks", "gather_idx",
                                                "scatter_idx", "h", "Y", "Xp")]


_lib = None


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Loads libmoe_gb300.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError("libmoe_gb300.so is not built: run __graft_entry__.build() "
                           "(the layer has no CPU fallback)")
    lib = ctypes.CDLL(_LIB_PATH)
    P, S = ctypes.c_void_p, ctypes.POINTER(MoEShape)
    st = ctypes.c_int
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_status_string.argtypes = [st]
    lib.moe_capacity.restype = st
    lib.moe_capacity.argtypes = [S, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]
    lib.moe_workspace_size.restype = st
    lib.moe_workspace_size.argtypes = [S, ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_workspace_init.restype = st
    lib.moe_workspace_init.argtypes = [S, P, P]
    lib.moe_workspace_views.restype = st
    lib.moe_workspace_views.argtypes = [S, P, ctypes.POINTER(MoEViews)]
    lib.moe_last_device_status.restype = st
    lib.moe_last_device_status.argtypes = [P, P]
    lib.moe_check_wait_timeout.restype = st
    lib.moe_check_wait_timeout.argtypes = [P, P]
    lib.moe_route.restype = st
    lib.moe_route.argtypes = [S] + [P] * 11
    lib.moe_route_noalloc.restype = st
    lib.moe_route_noalloc.argtypes = [S] + [P] * 10
    lib.moe_grouped_gemm_up.restype = st
    lib.moe_grouped_gemm_up.argtypes = [S] + [P] * 9
    lib.moe_grouped_gemm_up_rows.restype = st
    lib.moe_grouped_gemm_up_rows.argtypes = [S] + [P] * 8
    lib.moe_grouped_gemm_down.restype = st
    lib.moe_grouped_gemm_down.argtypes = [S] + [P] * 7
    lib.moe_combine.restype = st
    lib.moe_combine.argtypes = [S] + [P] * 6
    lib.moe_forward.restype = st
    lib.moe_forward.argtypes = [S] + [P] * 8
    _lib = lib
    return lib


def _check(rc: int, where: str):
    if rc != 0:
        raise MoEError(rc, where)


def shape(T: int, H: int, I: int, E: int, k: int) -> MoEShape:
    return MoEShape(T, H, I, E, k)


def _sp(s):
    if isinstance(s, MoEShape):
        return ctypes.byref(s)
    return ctypes.byref(MoEShape(*s))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev_tensor(t, dtype, min_numel, name):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if t.numel() < min_numel:
        raise ValueError("%s holds %d elements, needs %d" % (name, t.numel(), min_numel))
    return t.data_ptr()


def capacity(s) -> tuple:
    mb, mr = ctypes.c_int64(), ctypes.c_int64()
    _check(load().moe_capacity(_sp(s), ctypes.byref(mb), ctypes.byref(mr)), "moe_capacity")
    return mb.value, mr.value


def workspace_size(s) -> int:
    n = ctypes.c_size_t()
    _check(load().moe_workspace_size(_sp(s), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def workspace_init(s, ws, stream=None):
    _check(load().moe_workspace_init(_sp(s), _ptr(ws), _stream(stream)), "moe_workspace_init")


def alloc_workspace(s, device="cuda", stream=None):
    """A uint8 CUDA tensor of moe_workspace_size bytes with its status word cleared."""
    import torch
    ws = torch.empty(workspace_size(s), dtype=torch.uint8, device=device)
    workspace_init(s, ws, stream)
    return ws


def workspace_views(s, ws) -> MoEViews:
    v = MoEViews()
    _check(load().moe_workspace_views(_sp(s), _ptr(ws), ctypes.byref(v)), "moe_workspace_views")
    return v


def last_device_status(ws, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the kernels' status."""
    return load().moe_last_device_status(_ptr(ws), _stream(stream))


def check_wait_timeout(ws, stream=None) -> None:
    """Launches the diagnostic kernel whose bounded wait runs out (about 2 s);
    the next last_device_status(ws) reports MOE_ERR_TIMEOUT."""
    _check(load().moe_check_wait_timeout(_ptr(ws), _stream(stream)), "moe_check_wait_timeout")


def alloc_route_outputs(s, device="cuda") -> dict:
    """Device buffers for moe_route's outputs, sized to the shape's capacity."""
    import torch
    if not isinstance(s, MoEShape):
        s = MoEShape(*s)
    mb, mr = capacity(s)
    i32 = dict(dtype=torch.int32, device=device)
    return {
        "topk_ids": torch.empty((s.T, s.k), **i32),
        "topk_w": torch.empty((s.T, s.k), dtype=torch.float32, device=device),
        "counts": torch.empty(s.E, **i32),
        "off_pad": torch.empty(s.E + 1, **i32),
        "block_expert": torch.empty(mb, **i32),
        "num_blocks": torch.empty(1, **i32),
        "gather_idx": torch.empty(mr, **i32),
        "scatter_idx": torch.empty((s.T, s.k), **i32),
    }


def _shape_obj(s) -> MoEShape:
    return s if isinstance(s, MoEShape) else MoEShape(*s)


def moe_route(s, logits, topk_ids, topk_w, counts, off_pad, block_expert, num_blocks,
              gather_idx, scatter_idx, ws, stream=None):
    import torch
    s = _shape_obj(s)
    mb, mr = capacity(s)
    args = [_dev_tensor(logits, torch.float32, s.T * s.E, "logits"),
            _dev_tensor(topk_ids, torch.int32, s.T * s.k, "topk_ids"),
            _dev_tensor(topk_w, torch.float32, s.T * s.k, "topk_w"),
            _dev_tensor(counts, torch.int32, s.E, "counts"),
            _dev_tensor(off_pad, torch.int32, s.E + 1, "off_pad"),
            _dev_tensor(block_expert, torch.int32, mb, "block_expert"),
            _dev_tensor(num_blocks, torch.int32, 1, "num_blocks"),
            _dev_tensor(gather_idx, torch.int32, mr, "gather_idx"),
            _dev_tensor(scatter_idx, torch.int32, s.T * s.k, "scatter_idx"),
            _dev_tensor(ws, torch.uint8, workspace_size(s), "ws")]
    _check(load().moe_route(ctypes.byref(s), *args, _stream(stream)), "moe_route")


def moe_route_noalloc(s, logits, topk_ids, topk_w, counts, off_pad, block_expert, num_blocks,
                      gather_idx, scatter_idx, stream=None):
    """moe_route without a workspace (fixed library-owned scratch; see
    include/moe.h for its size limit and the rule that overlapping calls race)."""
    import torch
    s = _shape_obj(s)
    mb, mr = capacity(s)
    args = [_dev_tensor(logits, torch.float32, s.T * s.E, "logits"),
            _dev_tensor(topk_ids, torch.int32, s.T * s.k, "topk_ids"),
            _dev_tensor(topk_w, torch.float32, s.T * s.k, "topk_w"),
            _dev_tensor(counts, torch.int32, s.E, "counts"),
            _dev_tensor(off_pad, torch.int32, s.E + 1, "off_pad"),
            _dev_tensor(block_expert, torch.int32, mb, "block_expert"),
            _dev_tensor(num_blocks, torch.int32, 1, "num_blocks"),
            _dev_tensor(gather_idx, torch.int32, mr, "gather_idx"),
            _dev_tensor(scatter_idx, torch.int32, s.T * s.k, "scatter_idx")]
    _check(load().moe_route_noalloc(ctypes.byref(s), *args, _stream(stream)), "moe_route_noalloc")


def moe_grouped_gemm_up(s, X, scatter_idx, counts, off_pad, W_gate, W_up, h, ws, stream=None):
    import torch
    s = _shape_obj(s)
    mb, mr = capacity(s)
    bf = torch.bfloat16
    args = [_dev_tensor(X, bf, s.T * s.H, "X"),
            _dev_tensor(scatter_idx, torch.int32, s.T * s.k, "scatter_idx"),
            _dev_tensor(counts, torch.int32, s.E, "counts"),
            _dev_tensor(off_pad, torch.int32, s.E + 1, "off_pad"),
            _dev_tensor(W_gate, bf, s.E * s.H * s.I, "W_gate"),
            _dev_tensor(W_up, bf, s.E * s.H * s.I, "W_up"),
            _dev_tensor(h, bf, mr * s.I, "h"),
            _dev_tensor(ws, torch.uint8, workspace_size(s), "ws")]
    _check(load().moe_grouped_gemm_up(ctypes.byref(s), *args, _stream(stream)), "moe_grouped_gemm_up")


def moe_grouped_gemm_up_rows(s, Xp, counts, off_pad, W_gate, W_up, h, ws, stream=None):
    """The gate/up GEMM on rows already in expert order (no row gather)."""
    import torch
    s = _shape_obj(s)
    mb, mr = capacity(s)
    bf = torch.bfloat16
    args = [_dev_tensor(Xp, bf, mr * s.H, "Xp"),
            _dev_tensor(counts, torch.int32, s.E, "counts"),
            _dev_tensor(off_pad, torch.int32, s.E + 1, "off_pad"),
            _dev_tensor(W_gate, bf, s.E * s.H * s.I, "W_gate"),
            _dev_tensor(W_up, bf, s.E * s.H * s.I, "W_up"),
            _dev_tensor(h, bf, mr * s.I, "h"),
            _dev_tensor(ws, torch.uint8, workspace_size(s), "ws")]
    _check(load().moe_grouped_gemm_up_rows(ctypes.byref(s), *args, _stream(stream)), "moe_grouped_gemm_up_rows")


def moe_grouped_gemm_down(s, h, counts, off_pad, W_down, Y, ws, stream=None):
    import torch
    s = _shape_obj(s)
    mb, mr = capacity(s)
    bf = torch.bfloat16
    args = [_dev_tensor(h, bf, mr * s.I, "h"),
            _dev_tensor(counts, torch.int32, s.E, "counts"),
            _dev_tensor(off_pad, torch.int32, s.E + 1, "off_pad"),
            _dev_tensor(W_down, bf, s.E * s.I * s.H, "W_down"),
            _dev_tensor(Y, bf, mr * s.H, "Y"),
            _dev_tensor(ws, torch.uint8, workspace_size(s), "ws")]
    _check(load().moe_grouped_gemm_down(ctypes.byref(s), *args, _stream(stream)),
           "moe_grouped_gemm_down")


def moe_combine(s, Y, scatter_idx, topk_w, out, ws=None, stream=None):
    import torch
    s = _shape_obj(s)
    mb, mr = capacity(s)
    bf = torch.bfloat16
    args = [_dev_tensor(Y, bf, mr * s.H, "Y"),
            _dev_tensor(scatter_idx, torch.int32, s.T * s.k, "scatter_idx"),
            _dev_tensor(topk_w, torch.float32, s.T * s.k, "topk_w"),
            _dev_tensor(out, bf, s.T * s.H, "out"),
            None if ws is None else _dev_tensor(ws, torch.uint8, workspace_size(s), "ws")]
    _check(load().moe_combine(ctypes.byref(s), *args, _stream(stream)), "moe_combine")


def moe_forward(s, logits, X, W_gate, W_up, W_down, out, ws, stream=None):
    import torch
    s = _shape_obj(s)
    bf = torch.bfloat16
    args = [_dev_tensor(logits, torch.float32, s.T * s.E, "logits"),
            _dev_tensor(X, bf, s.T * s.H, "X"),
            _dev_tensor(W_gate, bf, s.E * s.H * s.I, "W_gate"),
            _dev_tensor(W_up, bf, s.E * s.H * s.I, "W_up"),
            _dev_tensor(W_down, bf, s.E * s.I * s.H, "W_down"),
            _dev_tensor(out, bf, s.T * s.H, "out"),
            _dev_tensor(ws, torch.uint8, workspace_size(s), "ws")]
    _check(load().moe_forward(ctypes.byref(s), *args, _stream(stream)), "moe_forward")


def moe_forward_raw(s, logits_ptr, x_ptr, wg_ptr, wu_ptr, wd_ptr, out_ptr, ws_ptr, stream_handle):
    """moe_forward on raw device pointers (no per-call tensor checks)."""
    s = _shape_obj(s)
    _check(load().moe_forward(ctypes.byref(s), logits_ptr, x_ptr, wg_ptr, wu_ptr, wd_ptr, out_ptr,
                              ws_ptr, stream_handle), "moe_forward")
