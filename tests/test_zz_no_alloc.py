"""The forward entry point that allocates no device memory.

It exists for callers that cannot allocate: for example a plug-in that lives
inside another engine's memory pool and only receives its input and output
buffers, or a decode loop in which cudaMalloc (which can stall the device) is
forbidden.  Its scratch is a fixed array inside the library.  These tests call
it through the C ABI, twice in a row on different layers (the second call
finds the first call's leftovers in the shared array), and compare each
result with the ordinary workspace-taking entry point on the same inputs.
This file is collected last on purpose, and it also passes on its own in a
fresh process.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import synthetic as syn
from helpers import OUTPUT_RTOL, bf16_tensor_bits, row_rel_l2, to_dev

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _no_alloc_call(lib, d, wl, out, ids):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.qmoe_fp4_moe_forward_no_alloc(
        _ptr(d["x"]), _ptr(d["logits"]), _ptr(d["w1"]), _ptr(d["s1"]), _ptr(d["g1"]), _ptr(d["w2"]),
        _ptr(d["s2"]), _ptr(d["g2"]), wl.fmt, wl.T, wl.H, wl.I, wl.E, wl.k, wl.normalize, 1,
        ctypes.c_float(wl.alpha), ctypes.c_float(wl.beta), ctypes.c_float(wl.limit), _ptr(out),
        _ptr(ids), stream)


@pytest.mark.parametrize("name", ["nvfp4_mtp_decode", "mxfp4_decode"])
def test_no_alloc_matches_workspace_entry_point_twice(qgpu, name):
    lib = qgpu.load()
    wl = syn.WORKLOADS[name]
    for seed in (0, 1):                      # two calls in a row on different layers
        d = to_dev(syn.layer(wl, seed=seed))
        ref_ids = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
        ref = qgpu.moe_forward(d["x"], d["logits"], d["w1"], d["s1"], d["g1"], d["w2"], d["s2"],
                               d["g2"], wl.fmt, wl.k, wl.normalize, wl.alpha, wl.beta, wl.limit,
                               topk_ids=ref_ids)
        out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
        ids = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
        rc = _no_alloc_call(lib, d, wl, out, ids)
        assert rc == 0, lib.qmoe_last_error()
        torch.cuda.synchronize()
        err, _ = row_rel_l2(bf16_tensor_bits(out), bf16_tensor_bits(ref))
        assert err <= OUTPUT_RTOL, (name, seed, err)
        assert torch.equal(ids, ref_ids)


def test_no_alloc_rejects_sizes_beyond_its_scratch(qgpu):
    """A shape whose scratch need exceeds the fixed array is refused with a
    clear error before anything is launched.  Only the router logits are a
    real buffer; every other pointer is deliberately misaligned, so that a
    call that got past the size check would stop at argument validation
    instead of launching anything."""
    lib = qgpu.load()
    wl = syn.small("big", T=64, E=64, k=1, H=8192, I=4096)
    need = qgpu.forward_workspace_bytes(wl.T, wl.H, wl.I, wl.E, wl.k, wl.fmt)
    assert need > lib_scratch_bytes()
    logits = torch.zeros((wl.T, wl.E), dtype=torch.float32, device="cuda")
    bad = ctypes.c_void_p(0x1001)
    rc = lib.qmoe_fp4_moe_forward_no_alloc(bad, _ptr(logits), bad, bad, None, bad, bad, None, wl.fmt, wl.T,
                                           wl.H, wl.I, wl.E, wl.k, 1, 1, ctypes.c_float(1.0),
                                           ctypes.c_float(0.0), ctypes.c_float(math.inf), bad, None, None)
    assert rc == 4
    assert b"static scratch" in lib.qmoe_last_error()


def lib_scratch_bytes():
    """QMOE_NO_ALLOC_SCRATCH_BYTES as declared in the public header."""
    import os
    import re
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "qmoe.h")
    m = re.search(r"#define QMOE_NO_ALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", open(hdr).read())
    return int(m.group(1)) << int(m.group(2))
