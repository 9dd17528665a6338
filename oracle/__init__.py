"""Plain CPU oracle for the QMoE W4A16 layer -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``qmoe_oracle.c`` (plain C, double precision, compiled
here with gcc, no CUDA).  This module only compiles it, loads it with ctypes
and marshals numpy arrays.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import it; the product path never does.

bf16 tensors cross this boundary as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

NVFP4 = 0
MXFP4 = 1
BLOCK = {NVFP4: 16, MXFP4: 32}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmoe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libqmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i, d = ctypes.c_int, ctypes.c_double
            L.oracle_e2m1.restype = d
            L.oracle_e2m1.argtypes = [ctypes.c_uint]
            L.oracle_e4m3fn.restype = d
            L.oracle_e4m3fn.argtypes = [ctypes.c_uint]
            L.oracle_e8m0.restype = d
            L.oracle_e8m0.argtypes = [ctypes.c_uint]
            L.oracle_bf16_rne.restype = ctypes.c_uint16
            L.oracle_bf16_rne.argtypes = [d]
            L.oracle_bf16_to_double.restype = d
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_swiglu.restype = d
            L.oracle_swiglu.argtypes = [d, d, d, d, d]
            L.oracle_dequant_element.restype = d
            L.oracle_dequant_element.argtypes = [P, P, P, i, i, i, i, i, i]
            L.oracle_dequant.restype = i
            L.oracle_dequant.argtypes = [P, P, P, i, i, i, i, P]
            L.oracle_scales_kmajor.restype = i
            L.oracle_scales_kmajor.argtypes = [P, i, i, i, P]
            L.oracle_route.restype = i
            L.oracle_route.argtypes = [P, i, i, i, i, P, P, P, P, P]
            L.oracle_route_mixed.restype = i
            L.oracle_route_mixed.argtypes = [P, P, i, i, i, i, P, P, P, P, P]
            L.oracle_expert_fc1.restype = i
            L.oracle_expert_fc1.argtypes = [P, i, P, P, P, i, i, i, P]
            L.oracle_expert_fc2.restype = i
            L.oracle_expert_fc2.argtypes = [P, i, P, P, P, i, i, i, P]
            L.oracle_expert_ffn.restype = i
            L.oracle_expert_ffn.argtypes = [P, i, P, P, P, P, P, P, i, i, i, d, d, d, i, P]
            L.oracle_moe_forward.restype = i
            L.oracle_moe_forward.argtypes = [P, P, P, P, P, P, P, P, P, i, i, i, i, i, i, i,
                                             d, d, d, i, P, i, P, i]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (status {rc})")


# ---- codecs ----------------------------------------------------------------

def e2m1(code: int) -> float:
    return lib().oracle_e2m1(code)


def e4m3fn(byte: int) -> float:
    return lib().oracle_e4m3fn(byte)


def e8m0(byte: int) -> float:
    return lib().oracle_e8m0(byte)


def bf16_rne(v: float) -> int:
    return int(lib().oracle_bf16_rne(float(v)))


def bf16_to_float(bits) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def swiglu(gate: float, value: float, alpha=1.0, beta=0.0, limit=float("inf")) -> float:
    return lib().oracle_swiglu(gate, value, alpha, beta, limit)


# ---- dequantisation ------------------------------------------------------------

def dequant_element(packed, scales, gscale, fmt, e, n, k) -> float:
    packed, scales, gscale = _c(packed, np.uint8), _c(scales, np.uint8), _c(gscale, np.float32)
    K, N = packed.shape[1], packed.shape[2] * 2
    return lib().oracle_dequant_element(_ptr(packed), _ptr(scales), _ptr(gscale),
                                        N, K, fmt, e, n, k)


def dequant(packed, scales, gscale, fmt) -> np.ndarray:
    """packed uint8 [E,K,N/2], scales uint8 [E,N,K/bs], gscale f32 [E] or None
    -> bf16 bits uint16 [E,N,K]."""
    packed, scales, gscale = _c(packed, np.uint8), _c(scales, np.uint8), _c(gscale, np.float32)
    E, K, N = packed.shape[0], packed.shape[1], packed.shape[2] * 2
    assert scales.shape == (E, N, K // BLOCK[fmt])
    out = np.empty((E, N, K), dtype=np.uint16)
    _check(lib().oracle_dequant(_ptr(packed), _ptr(scales), _ptr(gscale), E, N, K, fmt,
                                _ptr(out)), "dequant")
    return out


def scales_kmajor(scales) -> np.ndarray:
    """Block scales uint8 [E,N,nb] -> uint8 [E,nb,N], out[e,b,n] = in[e,n,b]."""
    scales = _c(scales, np.uint8)
    E, N, nb = scales.shape
    out = np.empty((E, nb, N), dtype=np.uint8)
    _check(lib().oracle_scales_kmajor(_ptr(scales), E, N, nb, _ptr(out)), "scales_kmajor")
    return out


# ---- routing -----------------------------------------------------------------

def route(logits, k: int, normalize: int = 1, router_weights=None) -> dict:
    """Top-k routing and the permute maps.  With ``router_weights`` [T, E]
    (operator input 14) the logits only select and the mixing weights are
    ``router_weights[t][id]`` gathered at the selected experts (renormalised
    over the k when ``normalize``)."""
    logits = _c(logits, np.float32)
    rw = None if router_weights is None else _c(router_weights, np.float32)
    T, E = logits.shape
    R = T * k
    ids = np.empty(R, np.int32)
    w = np.empty(R, np.float64)
    off = np.empty(E + 1, np.int32)
    p2e = np.empty(max(R, 1), np.int32)
    e2p = np.empty(max(R, 1), np.int32)
    _check(lib().oracle_route_mixed(_ptr(logits), _ptr(rw), T, E, k, normalize, _ptr(ids), _ptr(w),
                                    _ptr(off), _ptr(p2e), _ptr(e2p)), "route")
    return dict(ids=ids.reshape(T, k), weights=w.reshape(T, k), offsets=off,
                perm_to_expanded=p2e[:R], expanded_to_perm=e2p[:R])


# ---- experts and the layer -------------------------------------------------------

def expert_fc1(x_row, e, w1, s1, g1, fmt) -> np.ndarray:
    x_row, w1, s1, g1 = _c(x_row, np.uint16), _c(w1, np.uint8), _c(s1, np.uint8), _c(g1, np.float32)
    H, I = w1.shape[1], w1.shape[2]
    h = np.empty(2 * I, np.float64)
    _check(lib().oracle_expert_fc1(_ptr(x_row), e, _ptr(w1), _ptr(s1), _ptr(g1), fmt, H, I,
                                   _ptr(h)), "expert_fc1")
    return h


def expert_fc2(a, e, w2, s2, g2, fmt) -> np.ndarray:
    a, w2, s2, g2 = _c(a, np.float64), _c(w2, np.uint8), _c(s2, np.uint8), _c(g2, np.float32)
    I, H = w2.shape[1], w2.shape[2] * 2
    y = np.empty(H, np.float64)
    _check(lib().oracle_expert_fc2(_ptr(a), e, _ptr(w2), _ptr(s2), _ptr(g2), fmt, H, I,
                                   _ptr(y)), "expert_fc2")
    return y


def expert_ffn(x_row, e, w1, s1, g1, w2, s2, g2, fmt, alpha=1.0, beta=0.0,
               limit=float("inf"), fusion=1) -> np.ndarray:
    x_row = _c(x_row, np.uint16)
    w1, s1, g1 = _c(w1, np.uint8), _c(s1, np.uint8), _c(g1, np.float32)
    w2, s2, g2 = _c(w2, np.uint8), _c(s2, np.uint8), _c(g2, np.float32)
    H, I = w1.shape[1], w1.shape[2]
    y = np.empty(H, np.float64)
    _check(lib().oracle_expert_ffn(_ptr(x_row), e, _ptr(w1), _ptr(s1), _ptr(g1), _ptr(w2),
                                   _ptr(s2), _ptr(g2), fmt, H, I, alpha, beta, limit, fusion,
                                   _ptr(y)), "expert_ffn")
    return y


def moe_forward(x, logits, w1, s1, g1, w2, s2, g2, fmt, k, normalize=1, alpha=1.0,
                beta=0.0, limit=float("inf"), tokens=None, nthreads=None, fusion=1,
                router_weights=None) -> np.ndarray:
    """The whole layer.  x bf16 bits [T,H], logits f32 [T,E], fc1 packed
    [E,H,I] + scales [E,2I,H/bs] + global [E]/None, fc2 packed [E,I,H/2] +
    scales [E,H,I/bs] + global [E]/None.  ``fusion`` is swiglu_fusion: FC1's
    gate/linear columns interleaved (1, and 0 read as 1) or concatenated (2).
    ``router_weights`` [T, E] or None: the mixing weights (see ``route``).
    Returns bf16 bits [len(tokens),H] (all T tokens when ``tokens`` is None)."""
    x, logits = _c(x, np.uint16), _c(logits, np.float32)
    rw = None if router_weights is None else _c(router_weights, np.float32)
    w1, s1, g1 = _c(w1, np.uint8), _c(s1, np.uint8), _c(g1, np.float32)
    w2, s2, g2 = _c(w2, np.uint8), _c(s2, np.uint8), _c(g2, np.float32)
    T, H = x.shape
    E, I = w1.shape[0], w1.shape[2]
    tok = None if tokens is None else np.ascontiguousarray(tokens, np.int32)
    ntok = T if tok is None else len(tok)
    out = np.empty((ntok, H), np.uint16)
    nth = nthreads if nthreads else (os.cpu_count() or 1)
    _check(lib().oracle_moe_forward(_ptr(x), _ptr(logits), _ptr(rw), _ptr(w1), _ptr(s1), _ptr(g1),
                                    _ptr(w2), _ptr(s2), _ptr(g2), fmt, T, H, I, E, k,
                                    normalize, alpha, beta, limit, fusion, _ptr(tok), ntok,
                                    _ptr(out), nth), "moe_forward")
    return out
