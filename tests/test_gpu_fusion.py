"""swiglu_fusion on the GPU: the concatenated FC1 layout (2: column m = gate,
I + m = linear) against the oracle on both paths (decode GEMV and prefill
GEMM, page-layout and k-major scales, caller-dequantised weights), and 0 read
as the interleaved layout 1, bit for bit."""
import numpy as np
import pytest
import torch

import synthetic as syn
from helpers import OUTPUT_RTOL, bf16_tensor_bits, concatenated_fc1, row_rel_l2, to_dev

pytestmark = pytest.mark.gpu


def _concat_layer(wl, seed):
    L = syn.layer(wl, seed)
    w1c, s1c = concatenated_fc1(L["w1"], L["s1"])
    return dict(L, w1=w1c, s1=s1c)


def _gpu(qgpu, wl, L, fusion, kmajor=False, dequantised=False):
    d = to_dev(L)
    s1, s2, fmt = d["s1"], d["s2"], wl.fmt
    kw = {}
    if dequantised:
        kw["w1_dequant"] = qgpu.dequant(d["w1"], d["s1"], d["g1"], wl.fmt)
        kw["w2_dequant"] = qgpu.dequant(d["w2"], d["s2"], d["g2"], wl.fmt)
    if kmajor:
        s1, s2, fmt = qgpu.scales_kmajor(s1, wl.fmt), qgpu.scales_kmajor(s2, wl.fmt), wl.fmt | qgpu.SCALES_KMAJOR
    out = qgpu.moe_forward(d["x"], d["logits"], d["w1"], s1, d["g1"], d["w2"], s2, d["g2"], fmt, wl.k,
                           wl.normalize, wl.alpha, wl.beta, wl.limit, swiglu_fusion=fusion, **kw)
    torch.cuda.synchronize()
    return bf16_tensor_bits(out)


def _ref(oracle, wl, L, fusion, tokens=None):
    return oracle.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"],
                              wl.fmt, wl.k, wl.normalize, wl.alpha, wl.beta, wl.limit, tokens=tokens,
                              fusion=fusion)


DECODE = [
    syn.small("dec_nv", T=4, E=32, k=4, H=256, I=192),
    syn.small("dec_tiles", T=2, E=8, k=2, H=256, I=2304),          # FC1 N = 4608 in 9 tiles: gate and linear apart
    syn.small("dec_mx", T=3, E=8, k=2, H=320, I=192, fmt=1),
    syn.small("dec_gptoss", T=4, E=32, k=4, H=192, I=128, fmt=1, alpha=1.702, beta=1.0, limit=7.0),
]
PREFILL = [
    syn.small("pf_nv", T=20, E=16, k=4, H=256, I=128),
    syn.small("pf_mx", T=40, E=8, k=2, H=320, I=192, fmt=1),
]


@pytest.mark.parametrize("wl", DECODE + PREFILL, ids=lambda w: w.name)
def test_concatenated_swiglu(qgpu, oracle, wl):
    L = _concat_layer(wl, 31)
    ref = _ref(oracle, wl, L, 2)
    for kw in (dict(), dict(kmajor=True)):
        err, elem = row_rel_l2(_gpu(qgpu, wl, L, 2, **kw), ref)
        assert err <= OUTPUT_RTOL, (wl.name, kw, err, elem)


@pytest.mark.parametrize("wl", PREFILL, ids=lambda w: w.name)
def test_concatenated_swiglu_dequantised_weights(qgpu, oracle, wl):
    L = _concat_layer(wl, 32)
    err, elem = row_rel_l2(_gpu(qgpu, wl, L, 2, dequantised=True), _ref(oracle, wl, L, 2))
    assert err <= OUTPUT_RTOL, (wl.name, err, elem)


def test_concatenated_swiglu_mtp_decode_workload(qgpu, oracle):
    wl = syn.WORKLOADS["nvfp4_mtp_decode"]
    L = _concat_layer(wl, 33)
    err, elem = row_rel_l2(_gpu(qgpu, wl, L, 2, kmajor=True), _ref(oracle, wl, L, 2))
    assert err <= OUTPUT_RTOL, (err, elem)


@pytest.mark.parametrize("wl", [DECODE[0], PREFILL[0]], ids=lambda w: w.name)
def test_fusion_zero_is_interleaved(qgpu, wl):
    L = syn.layer(wl, 34)
    assert np.array_equal(_gpu(qgpu, wl, L, 0), _gpu(qgpu, wl, L, 1))
