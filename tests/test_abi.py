"""The C-ABI library: it builds for sm_103a, exports every symbol the header
declares, and rejects invalid calls on the host before launching anything
(these calls need no GPU)."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qm():
    import block_scaled_fp4_gb300 as q
    q.build()
    return q


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(qmoe_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol(qm):
    declared = _declared()
    assert {"qmoe_route_topk", "qmoe_fp4_moe_forward", "qmoe_fp4_dequant"} <= declared
    lib = ctypes.CDLL(qm.library_path())
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert declared == set(qm.EXPORTS)


def test_built_for_sm103a_only(qm):
    """The build compiles one image, for sm_103a (the runtime check of the
    image a GB300 loads is test_gpu_errors.test_kernels_run_the_sm103a_image)."""
    import importlib
    b = importlib.import_module("block_scaled_fp4_gb300.build")
    assert b.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


# The validation tests below pass placeholder pointers, which the host checks
# must reject before any launch.  They run in a child process that sees no GPU,
# so a validation regression can never launch a kernel on those pointers.
def _in_child_without_gpu(body: str) -> None:
    import subprocess
    import sys
    import textwrap
    code = textwrap.dedent("""
        import ctypes, math, os, sys
        sys.path.insert(0, %r)
        sys.path.insert(0, %r)
        import block_scaled_fp4_gb300 as qm
        L = qm.load()
        import test_abi as T
    """) % (ROOT, os.path.join(ROOT, "tests")) + textwrap.dedent(body)
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="-1")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr


def _fwd(L, **kw):
    P = ctypes.c_void_p
    a = dict(x=P(256), logits=P(256), rw=None, w1=P(256), s1=P(256), g1=None, w2=P(256), s2=P(256), g2=None,
             wd1=None, wd2=None, fmt=0, T=4, H=2048, I=512, E=256, k=8, normalize=1, fusion=1,
             alpha=1.0, beta=0.0, limit=math.inf, out=P(256), ids=None, ws=None)
    a.update(kw)
    nb = ctypes.c_size_t(a.pop("nbytes", 0))
    rc = L.qmoe_fp4_moe_forward(a["x"], a["logits"], a["rw"], a["w1"], a["s1"], a["g1"], a["w2"], a["s2"],
                                a["g2"], a["wd1"], a["wd2"], a["fmt"], a["T"], a["H"], a["I"], a["E"],
                                a["k"], a["normalize"], a["fusion"], a["alpha"], a["beta"],
                                a["limit"], a["out"], a["ids"], a["ws"], ctypes.byref(nb), None)
    return rc, nb.value


def check_forward_validation(L):
    rc, need = _fwd(L)
    assert rc == 0 and need > 0                                   # size query
    assert _fwd(L, k=9)[0] == 1                                   # k > 8
    assert _fwd(L, E=4, k=5)[0] == 1                              # k > E
    assert _fwd(L, E=257)[0] == 3                                 # E > 256
    assert _fwd(L, T=0)[0] == 1
    assert _fwd(L, logits=None)[0] == 1
    assert _fwd(L, H=2000)[0] == 3                                # H % 64
    assert _fwd(L, fusion=3)[0] == 3                              # no such SwiGLU layout
    assert _fwd(L, fusion=-1)[0] == 3
    assert _fwd(L, fusion=2) == (0, need)                         # concatenated: same workspace
    assert _fwd(L, fusion=0) == (0, need)                         # read as interleaved
    assert _fwd(L, fmt=2)[0] == 3
    assert _fwd(L, alpha=float("nan"))[0] == 1
    assert _fwd(L, rw=ctypes.c_void_p(258))[0] == 2               # router_weights not 4-byte aligned
    assert _fwd(L, rw=ctypes.c_void_p(256)) == (0, need)          # router_weights: same workspace
    ws = ctypes.c_void_p(1 << 20)
    assert _fwd(L, ws=ws, nbytes=need - 1)[0] == 4                # workspace too small
    assert _fwd(L, ws=ws, nbytes=need, x=ctypes.c_void_p(258))[0] == 2   # misaligned
    assert _fwd(L, ws=ws, nbytes=need, out=None)[0] == 1
    assert b"workspace" in L.qmoe_last_error() or True


def test_forward_validation(qm):
    _in_child_without_gpu("T.check_forward_validation(L)")


def check_route_and_dequant_validation(L):
    P = ctypes.c_void_p
    nb = ctypes.c_size_t(99)
    assert L.qmoe_route_topk(P(256), None, 4, 256, 8, 1, None, None, None, None, None, None,
                             ctypes.byref(nb), None) == 0 and nb.value == 0
    assert L.qmoe_route_topk(P(256), None, 4, 256, 9, 1, None, None, None, None, None, None,
                             ctypes.byref(nb), None) == 1
    assert L.qmoe_route_topk(P(258), None, 4, 256, 8, 1, P(256), P(256), P(256), P(256), P(256), None,
                             ctypes.byref(nb), None) == 2
    assert L.qmoe_route_topk(P(256), P(258), 4, 256, 8, 1, P(256), P(256), P(256), P(256), P(256), None,
                             ctypes.byref(nb), None) == 2
    assert L.qmoe_fp4_dequant(None, P(256), None, 1, 64, 64, 0, P(256), None) == 1
    assert L.qmoe_fp4_dequant(P(256), P(256), None, 1, 96, 64, 0, P(256), None) == 3
    assert L.qmoe_fp4_dequant(P(264), P(256), None, 1, 64, 64, 0, P(256), None) == 2
    assert L.qmoe_fp4_dequant(P(256), P(256), None, 1, 64, 64, 7, P(256), None) == 3
    assert b"format" in L.qmoe_last_error()


def test_route_and_dequant_validation(qm):
    _in_child_without_gpu("T.check_route_and_dequant_validation(L)")


def test_binding_constants_match_the_header(qm):
    """The flag and size constants the binding passes through are the header's."""
    src = open(os.path.join(ROOT, "include", "qmoe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)

    def value(name):
        m = re.search(r"\b" + name + r"\s*=\s*(0x[0-9A-Fa-f]+|\d+)", src) or \
            re.search(r"#define\s+" + name + r"\s+(0x[0-9A-Fa-f]+|\d+)", src)
        assert m, name
        return int(m.group(1), 0)

    assert value("QMOE_NVFP4") == qm.NVFP4 and value("QMOE_MXFP4") == qm.MXFP4
    assert value("QMOE_SCALES_KMAJOR") == qm.SCALES_KMAJOR
    assert value("QMOE_WORKSPACE_PRIMED") == qm.WORKSPACE_PRIMED
    assert value("QMOE_WORKSPACE_HEADER_BYTES") == qm.WORKSPACE_HEADER_BYTES
    assert value("QMOE_GEMV_MAX_ROWS") == qm.GEMV_MAX_ROWS
    # the flags are distinct bits above the format codes
    assert qm.SCALES_KMAJOR & qm.WORKSPACE_PRIMED == 0 and min(qm.SCALES_KMAJOR, qm.WORKSPACE_PRIMED) > qm.MXFP4


def check_primed_flag(qm, L):
    """dequant and scales_kmajor take a plain format: the flag is rejected there."""
    dummy = ctypes.c_void_p(256)
    for fmt in (qm.NVFP4 | qm.WORKSPACE_PRIMED, qm.MXFP4 | qm.WORKSPACE_PRIMED):
        assert L.qmoe_fp4_dequant(dummy, dummy, None, 1, 64, 64, fmt, dummy, None) == 3
        assert L.qmoe_fp4_scales_kmajor(dummy, 1, 64, 64, fmt, ctypes.c_void_p(1 << 20), None) == 3
    # the forward size query accepts it and the size does not depend on it
    base = qm.forward_workspace_bytes(4, 2048, 512, 256, 8, qm.NVFP4 | qm.SCALES_KMAJOR)
    assert base == qm.forward_workspace_bytes(4, 2048, 512, 256, 8,
                                              qm.NVFP4 | qm.SCALES_KMAJOR | qm.WORKSPACE_PRIMED)
    assert base >= qm.WORKSPACE_HEADER_BYTES


def test_primed_flag_is_a_format_flag_only_for_the_forward_calls(qm):
    _in_child_without_gpu("T.check_primed_flag(qm, L)")


def test_plan_accepts_every_supported_decode_shape(qm):
    """The decode plan (column tiling, ring, work-split bounds) exists for every
    shape inside the documented gate: H and I multiples of 64 up to 16384,
    1 <= k <= min(8, E), E <= 256, T * k <= 64, both formats and scale layouts
    (a size query: host logic only, nothing is launched)."""
    shapes = [(1, 8, 2), (4, 256, 8), (8, 256, 8), (64, 8, 1), (64, 64, 1), (16, 32, 4), (32, 2, 2),
              (1, 1, 1), (21, 3, 3)]
    dims = (64, 128, 192, 320, 1024, 2048, 2880, 4096, 7168, 16384)
    for fmt in (qm.NVFP4, qm.MXFP4, qm.NVFP4 | qm.SCALES_KMAJOR, qm.MXFP4 | qm.SCALES_KMAJOR):
        for H in dims:
            for I in dims:
                for T, E, k in shapes:
                    assert T * k <= qm.GEMV_MAX_ROWS
                    assert qm.forward_workspace_bytes(T, H, I, E, k, fmt) > 0, (fmt, H, I, T, E, k)


def test_binding_has_no_cpu_fallback(qm):
    """The Python binding refuses host tensors instead of computing anything
    on the CPU, for every compute entry point."""
    import torch
    import synthetic as syn
    wl = syn.small("cpu", T=2, E=4, k=2, H=64, I=64)
    L = syn.layer(wl, seed=1)
    t = {k: (None if v is None else torch.from_numpy(np.ascontiguousarray(v))) for k, v in L.items()}
    x = t["x"].view(torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        qm.moe_forward(x, t["logits"], t["w1"], t["s1"], t["g1"], t["w2"], t["s2"], t["g2"], wl.fmt, wl.k)
    with pytest.raises(ValueError, match="CUDA tensor"):
        qm.moe_forward_no_alloc(x, t["logits"], t["w1"], t["s1"], t["g1"], t["w2"], t["s2"], t["g2"],
                                wl.fmt, wl.k)
    with pytest.raises(ValueError, match="CUDA tensor"):
        qm.route_topk(t["logits"], wl.k)
    with pytest.raises(ValueError, match="CUDA tensor"):
        qm.dequant(t["w1"], t["s1"], t["g1"], wl.fmt)
    with pytest.raises(ValueError, match="CUDA tensor"):
        qm.scales_kmajor(t["s1"], wl.fmt)


def test_no_alloc_rejects_sizes_beyond_its_scratch(qm):
    """A shape whose scratch need exceeds the no-alloc entry point's fixed array
    is refused with a clear error before anything is launched (in a child that
    sees no GPU; the size check needs none)."""
    import re
    hdr = open(os.path.join(ROOT, "include", "qmoe.h")).read()
    m = re.search(r"#define QMOE_NO_ALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", hdr)
    scratch = int(m.group(1)) << int(m.group(2))
    need = qm.forward_workspace_bytes(64, 8192, 4096, 64, 1, qm.NVFP4)
    assert need > scratch
    _in_child_without_gpu("""
        P = ctypes.c_void_p
        bad = P(0x1001)
        rc = L.qmoe_fp4_moe_forward_no_alloc(bad, P(256), bad, bad, None, bad, bad, None, 0, 64, 8192, 4096,
                                             64, 1, 1, 1, ctypes.c_float(1.0), ctypes.c_float(0.0),
                                             ctypes.c_float(math.inf), bad, None, None)
        assert rc == 4, rc
        assert b"static scratch" in L.qmoe_last_error()
    """)


def test_prefill_workspace_sizes(qm):
    """Prefill shapes (T * k > 64): the fused GEMMs need no bf16 weight copy;
    block scales as stored add their k-major rewrite (E * N * K / bs bytes per
    FC) to the workspace, an FC given as bf16 weights does not."""
    T, H, I, E, k = 2048, 2048, 1536, 128, 8
    page = qm.forward_workspace_bytes(T, H, I, E, k, qm.NVFP4)
    km = qm.forward_workspace_bytes(T, H, I, E, k, qm.NVFP4 | qm.SCALES_KMAJOR)
    s1_bytes, s2_bytes = E * 2 * I * (H // 16), E * H * (I // 16)
    assert page - km == s1_bytes + s2_bytes
    # the fused FC1 reads x gathered in expert order (bf16 [R, H])
    R = T * k
    xp_bytes = R * H * 2
    assert qm.forward_workspace_bytes(T, H, I, E, k, qm.NVFP4, True) == km - xp_bytes
    assert qm.forward_workspace_bytes(T, H, I, E, k, qm.NVFP4, (True, False)) == km - xp_bytes + s2_bytes
    assert qm.forward_workspace_bytes(T, H, I, E, k, qm.NVFP4, (False, True)) == km + s1_bytes
    # routing maps, gathered x, activations (bf16 [R, I]) and FC2 rows (fp32 [R, H]) at least
    assert km >= qm.WORKSPACE_HEADER_BYTES + xp_bytes + R * I * 2 + R * H * 4
    assert km < qm.WORKSPACE_HEADER_BYTES + xp_bytes + R * I * 2 + R * H * 4 + 64 * R + 8192
