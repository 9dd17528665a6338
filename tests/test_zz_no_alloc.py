"""The forward entry point that allocates no device memory.

It exists for callers that cannot allocate: for example a plug-in that lives
inside another engine's memory pool and only receives its input and output
buffers, or a decode loop in which cudaMalloc (which can stall the device) is
forbidden.  Its scratch is a fixed array inside the library.  These tests call
it through the C ABI, twice in a row on different layers (the second call
finds the first call's leftovers in the shared array), and compare each
result bit for bit with the ordinary workspace-taking entry point on the same
inputs (the same kernels on the same data).  The rejection of sizes beyond the
array is tested on the CPU (test_abi.py).  This file is collected last on
purpose, and it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import synthetic as syn
from helpers import bf16_tensor_bits, to_dev

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


def _workspace_call(qgpu, d, wl):
    ids = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    out = qgpu.moe_forward(d["x"], d["logits"], d["w1"], d["s1"], d["g1"], d["w2"], d["s2"], d["g2"], wl.fmt,
                           wl.k, wl.normalize, wl.alpha, wl.beta, wl.limit, topk_ids=ids)
    return out, ids


def _compare(qgpu, lib, wl, seed):
    """One no-alloc call against the workspace entry point on the same inputs:
    the same kernels run on the same data, so the results agree bit for bit."""
    d = to_dev(syn.layer(wl, seed=seed))
    ref, ref_ids = _workspace_call(qgpu, d, wl)
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    rc = _no_alloc_call(lib, d, wl, out, ids)
    assert rc == 0, lib.qmoe_last_error()
    torch.cuda.synchronize()
    assert np.array_equal(bf16_tensor_bits(out), bf16_tensor_bits(ref)), (wl.name, seed)
    assert torch.equal(ids, ref_ids)


@pytest.mark.parametrize("name", ["nvfp4_mtp_decode", "mxfp4_decode"])
def test_no_alloc_matches_workspace_entry_point_twice(qgpu, name):
    lib = qgpu.load()
    wl = syn.WORKLOADS[name]
    for seed in (0, 1):                      # two calls in a row on different layers
        _compare(qgpu, lib, wl, seed)
    qgpu.check_device_error(None)            # the static scratch's error flag stayed clear


def test_no_alloc_prefill_between_decodes(qgpu):
    """A prefill-sized call (more than 64 expanded rows) on the shared array
    between two decode calls: the prefill path leaves the decode header alone,
    so the decode call after it still matches."""
    lib = qgpu.load()
    dec = syn.WORKLOADS["nvfp4_mtp_decode"]
    pre = syn.small("no_alloc_prefill", T=40, E=16, k=4, H=256, I=128)
    _compare(qgpu, lib, dec, 2)
    _compare(qgpu, lib, pre, 3)
    _compare(qgpu, lib, dec, 4)
    qgpu.check_device_error(None)
