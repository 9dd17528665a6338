"""Python binding of the GB300 FP4 MoE (QMoE W4A16) C-ABI library.

Argument marshalling only: every step of the layer runs in the CUDA kernels
of ``_build/libqmoe.so`` (declared in ``include/qmoe.h``).  PyTorch supplies
device memory and the current stream.  There is no CPU fallback: importing
works without a GPU, but every call needs the built library and CUDA tensors
and raises otherwise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from .build import LIB, build

NVFP4 = 0
MXFP4 = 1
SCALES_KMAJOR = 0x100  # OR'd into fmt of the forward calls: block scales are [E, K/bs, N]
# OR'd into fmt of moe_forward: the workspace's first WORKSPACE_HEADER_BYTES
# bytes are zero (zeroed once by the caller; the library keeps them zero), so
# decode calls skip their header reset and chain by programmatic dependent launch
WORKSPACE_PRIMED = 0x200
# OR'd with SCALES_KMAJOR into fmt of moe_forward: decode calls run on the
# multi-row kernel whatever their size (without it, short weight streams run on
# the one-row-per-pass kernel)
DECODE_MULTIROW = 0x400
WORKSPACE_HEADER_BYTES = 64
BLOCK = {NVFP4: 16, MXFP4: 32}
GEMV_MAX_ROWS = 64

STATUS = {0: "QMOE_OK", 1: "QMOE_ERR_INVALID_ARG", 2: "QMOE_ERR_MISALIGNED",
          3: "QMOE_ERR_UNSUPPORTED", 4: "QMOE_ERR_WORKSPACE", 5: "QMOE_ERR_CUDA",
          6: "QMOE_ERR_DEVICE"}

# Every symbol include/qmoe.h declares.
EXPORTS = ("qmoe_route_topk", "qmoe_fp4_moe_forward", "qmoe_fp4_dequant", "qmoe_last_error",
           "qmoe_set_stage_events", "qmoe_fp4_moe_forward_no_alloc", "qmoe_fp4_scales_kmajor",
           "qmoe_check_device_error", "qmoe_binary_version")


class QMoEError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS.get(status, status)}: {message}")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return LIB


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the CUDA library (it must have been built with ``build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB
            if not os.path.exists(p):
                raise RuntimeError(f"QMoE CUDA library not built ({p} missing): call "
                                   "block_scaled_fp4_gb300.build() first")
            L = ctypes.CDLL(p)
            P, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.POINTER(ctypes.c_size_t)
            L.qmoe_route_topk.restype = i
            L.qmoe_route_topk.argtypes = [P, P, i, i, i, i, P, P, P, P, P, P, sz, P]
            L.qmoe_fp4_moe_forward.restype = i
            L.qmoe_fp4_moe_forward.argtypes = [P, P, P, P, P, P, P, P, P, P, P, i, i, i, i, i, i, i, i,
                                               f, f, f, P, P, P, sz, P]
            L.qmoe_fp4_dequant.restype = i
            L.qmoe_fp4_dequant.argtypes = [P, P, P, i, i, i, i, P, P]
            L.qmoe_fp4_scales_kmajor.restype = i
            L.qmoe_fp4_scales_kmajor.argtypes = [P, i, i, i, i, P, P]
            L.qmoe_last_error.restype = ctypes.c_char_p
            L.qmoe_last_error.argtypes = []
            L.qmoe_set_stage_events.restype = i
            L.qmoe_set_stage_events.argtypes = [P, i]
            L.qmoe_check_device_error.restype = i
            L.qmoe_check_device_error.argtypes = [P, P]
            L.qmoe_binary_version.restype = i
            L.qmoe_binary_version.argtypes = []
            L.qmoe_fp4_moe_forward_no_alloc.restype = i
            L.qmoe_fp4_moe_forward_no_alloc.argtypes = [P, P, P, P, P, P, P, P, i, i, i, i, i, i, i, i,
                                                        f, f, f, P, P, P]
            _lib = L
    return _lib


def _check(rc: int) -> None:
    if rc != 0:
        msg = load().qmoe_last_error().decode(errors="replace")
        raise QMoEError(rc, msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(t, name):
    if t is not None and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t is not None and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def route_topk(logits, k: int, normalize: int = 1, stream=None, router_weights=None):
    """Top-k softmax routing + permute-by-expert maps.  Returns a dict of
    CUDA tensors: ids [T,k] int32, weights [T,k] f32, offsets [E+1],
    perm_to_expanded [T*k], expanded_to_perm [T*k].  ``router_weights``
    f32 [T,E] (optional): the mixing weights, gathered at the experts the
    logits select."""
    import torch
    _cuda(logits, "logits")
    _cuda(router_weights, "router_weights")
    T, E = logits.shape
    dev = logits.device
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    p2e = torch.empty(T * k, dtype=torch.int32, device=dev)
    e2p = torch.empty(T * k, dtype=torch.int32, device=dev)
    nbytes = ctypes.c_size_t(0)
    _check(load().qmoe_route_topk(_ptr(logits), _ptr(router_weights), T, E, k, int(normalize), _ptr(ids), _ptr(w),
                                  _ptr(off), _ptr(p2e), _ptr(e2p), None, ctypes.byref(nbytes),
                                  _stream(stream)))
    return dict(ids=ids, weights=w, offsets=off, perm_to_expanded=p2e, expanded_to_perm=e2p)


def forward_workspace_bytes(T, H, I, E, k, fmt=NVFP4, with_dequantized=False) -> int:
    """Workspace bytes ``moe_forward`` needs for these sizes.
    ``with_dequantized``: True when both FCs' bf16 dequantised weights are
    given, or a pair (fc1 given, fc2 given)."""
    w1d, w2d = with_dequantized if isinstance(with_dequantized, tuple) else (with_dequantized,) * 2
    nbytes = ctypes.c_size_t(0)
    dummy = ctypes.c_void_p(16)
    _check(load().qmoe_fp4_moe_forward(None, dummy, None, None, None, None, None, None, None,
                                       dummy if w1d else None,
                                       dummy if w2d else None, fmt, T, H, I, E, k, 1, 1,
                                       1.0, 0.0, math.inf, None, None, None, ctypes.byref(nbytes),
                                       None))
    return nbytes.value


def moe_forward(x, logits, w1, s1, g1, w2, s2, g2, fmt: int, k: int, normalize: int = 1,
                alpha: float = 1.0, beta: float = 0.0, limit: float = math.inf,
                w1_dequant=None, w2_dequant=None, out=None, topk_ids=None, workspace=None,
                stream=None, swiglu_fusion: int = 1, router_weights=None):
    """The MoE layer.  x bf16 [T,H]; logits f32 [T,E]; w1 uint8 [E,H,I];
    s1 uint8 [E,2I,H/bs]; g1 f32 [E] or None; w2 uint8 [E,I,H/2];
    s2 uint8 [E,H,I/bs]; g2 f32 [E] or None.  With ``fmt | SCALES_KMAJOR``
    s1 is [E,H/bs,2I] and s2 [E,I/bs,H] (see ``scales_kmajor``).
    ``router_weights`` f32 [T,E] (optional): the mixing weights, gathered at
    the experts the logits select.  Returns out bf16 [T,H]."""
    import torch
    for t, n in ((x, "x"), (logits, "logits"), (w1, "w1"), (s1, "s1"), (g1, "g1"), (w2, "w2"),
                 (s2, "s2"), (g2, "g2"), (w1_dequant, "w1_dequant"), (w2_dequant, "w2_dequant"),
                 (router_weights, "router_weights")):
        _cuda(t, n)
    T, H = x.shape
    E, _, I = w1.shape
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    need = forward_workspace_bytes(T, H, I, E, k, fmt, (w1_dequant is not None, w2_dequant is not None))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    nbytes = ctypes.c_size_t(workspace.numel() * workspace.element_size())
    _check(load().qmoe_fp4_moe_forward(_ptr(x), _ptr(logits), _ptr(router_weights), _ptr(w1), _ptr(s1),
                                       _ptr(g1), _ptr(w2),
                                       _ptr(s2), _ptr(g2), _ptr(w1_dequant), _ptr(w2_dequant), fmt, T,
                                       H, I, E, k, int(normalize), int(swiglu_fusion), float(alpha),
                                       float(beta), float(limit), _ptr(out), _ptr(topk_ids),
                                       _ptr(workspace), ctypes.byref(nbytes), _stream(stream)))
    return out


def moe_forward_no_alloc(x, logits, w1, s1, g1, w2, s2, g2, fmt: int, k: int, normalize: int = 1,
                         alpha: float = 1.0, beta: float = 0.0, limit: float = math.inf, out=None,
                         topk_ids=None, stream=None, swiglu_fusion: int = 1):
    """The MoE layer through the entry point that allocates no device memory
    (its scratch is a fixed array inside the library; see include/qmoe.h).
    ``out`` must be given by callers that cannot allocate; when it is None a
    bf16 [T,H] tensor is created here for convenience."""
    import torch
    for t, n in ((x, "x"), (logits, "logits"), (w1, "w1"), (s1, "s1"), (g1, "g1"), (w2, "w2"),
                 (s2, "s2"), (g2, "g2"), (out, "out")):
        _cuda(t, n)
    T, H = x.shape
    E, _, I = w1.shape
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    _check(load().qmoe_fp4_moe_forward_no_alloc(_ptr(x), _ptr(logits), _ptr(w1), _ptr(s1), _ptr(g1),
                                                _ptr(w2), _ptr(s2), _ptr(g2), fmt, T, H, I, E, k,
                                                int(normalize), int(swiglu_fusion), float(alpha),
                                                float(beta), float(limit), _ptr(out), _ptr(topk_ids),
                                                _stream(stream)))
    return out


def dequant(packed, scales, gscale, fmt: int, out=None, stream=None):
    """packed uint8 [E,K,N/2], scales uint8 [E,N,K/bs], gscale f32 [E] or
    None -> bf16 [E,N,K]."""
    import torch
    for t, n in ((packed, "packed"), (scales, "scales"), (gscale, "gscale")):
        _cuda(t, n)
    E, K, N2 = packed.shape
    N = 2 * N2
    if out is None:
        out = torch.empty((E, N, K), dtype=torch.bfloat16, device=packed.device)
    _check(load().qmoe_fp4_dequant(_ptr(packed), _ptr(scales), _ptr(gscale), E, N, K, fmt, _ptr(out),
                                   _stream(stream)))
    return out


def scales_kmajor(scales, fmt: int, out=None, stream=None):
    """Block scales uint8 [E,N,K/bs] -> k-major uint8 [E,K/bs,N] (bytes
    unchanged), the layout the forward calls take with ``fmt | SCALES_KMAJOR``.
    A once-per-weight-set preparation step."""
    import torch
    _cuda(scales, "scales")
    E, N, nb = scales.shape
    K = nb * BLOCK[fmt]
    if out is None:
        out = torch.empty((E, nb, N), dtype=torch.uint8, device=scales.device)
    _cuda(out, "out")
    _check(load().qmoe_fp4_scales_kmajor(_ptr(scales), E, N, K, fmt, _ptr(out), _stream(stream)))
    return out


def check_device_error(workspace=None, stream=None) -> None:
    """Read and clear the device error flag of a forward workspace (``None``:
    the no-alloc entry point's static scratch on the current device).  Raises
    QMoEError (QMOE_ERR_DEVICE) when a bounded wait inside a kernel gave up
    since the last check.  Synchronises the stream."""
    _cuda(workspace, "workspace")
    _check(load().qmoe_check_device_error(_ptr(workspace), _stream(stream)))


def binary_version() -> int:
    """Compute capability the library's decode kernel was built for, as the
    runtime reports it on the current device (103 for sm_103a)."""
    return int(load().qmoe_binary_version())


def set_stage_events(events) -> int:
    """Record ``events[i]`` (torch.cuda.Event) around the forward's kernels;
    ``None`` switches it off.  Returns the number of kernels per decode call."""
    global _stage_keepalive
    L = load()
    if events is None:
        _stage_keepalive = None
        return L.qmoe_set_stage_events(None, 0)
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _stage_keepalive = arr
    return L.qmoe_set_stage_events(ctypes.cast(arr, ctypes.c_void_p), len(events))


_stage_keepalive = None

__all__ = ["NVFP4", "MXFP4", "BLOCK", "GEMV_MAX_ROWS", "QMoEError", "build", "load", "library_path",
           "route_topk", "moe_forward", "moe_forward_no_alloc", "forward_workspace_bytes", "dequant",
           "scales_kmajor", "SCALES_KMAJOR", "DECODE_MULTIROW", "set_stage_events", "check_device_error", "binary_version",
           "EXPORTS"]
