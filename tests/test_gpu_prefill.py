"""The prefill path (more than 64 expanded rows: two grouped GEMMs on the
tensor cores -- the fused W4A16 GEMM over the packed weights, or the bf16 one
over caller-dequantised weights -- and the weighted un-permute) against the
oracle, row-L2 relative error <= 1e-2: small shapes in full, the NVFP4
prefill workload on 128 sampled tokens, the caller-dequantised-weights
variant (both FCs or one), k-major scales, experts whose rows split into
several chunks and experts with no rows."""
import numpy as np
import pytest
import torch

import synthetic as syn
from helpers import OUTPUT_RTOL, bf16_tensor_bits, row_rel_l2, to_dev

pytestmark = pytest.mark.gpu


def _run(qgpu, wl, L, kmajor=False, dequantised=False):
    """dequantised: True (both FCs), "fc1" or "fc2" (that FC alone) given as bf16."""
    d = to_dev(L)
    s1, s2, fmt = d["s1"], d["s2"], wl.fmt
    kw = {}
    if dequantised in (True, "fc1"):
        kw["w1_dequant"] = qgpu.dequant(d["w1"], d["s1"], d["g1"], wl.fmt)
    if dequantised in (True, "fc2"):
        kw["w2_dequant"] = qgpu.dequant(d["w2"], d["s2"], d["g2"], wl.fmt)
    if kmajor:
        s1, s2, fmt = qgpu.scales_kmajor(s1, wl.fmt), qgpu.scales_kmajor(s2, wl.fmt), wl.fmt | qgpu.SCALES_KMAJOR
    ids = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    out = qgpu.moe_forward(d["x"], d["logits"], d["w1"], s1, d["g1"], d["w2"], s2, d["g2"], fmt, wl.k,
                           wl.normalize, wl.alpha, wl.beta, wl.limit, topk_ids=ids, **kw)
    torch.cuda.synchronize()
    return bf16_tensor_bits(out), ids.cpu().numpy()


def _ref(oracle, wl, L, tokens=None):
    return oracle.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"],
                              wl.fmt, wl.k, wl.normalize, wl.alpha, wl.beta, wl.limit, tokens=tokens)


SMALL = [
    syn.small("pf_nv", T=20, E=16, k=4, H=256, I=128),                     # R = 80: just past the window
    syn.small("pf_mx", T=40, E=8, k=2, H=320, I=192, fmt=1),                # MXFP4, N not a multiple of 128
    syn.small("pf_gptoss", T=70, E=12, k=3, H=192, I=256, fmt=1, alpha=1.702, beta=1.0, limit=7.0),
    syn.small("pf_nonorm", T=33, E=32, k=4, H=128, I=320, normalize=0),
    syn.small("pf_rows", T=300, E=4, k=2, H=256, I=192),                    # > 128 rows per expert: several row tiles
    syn.small("pf_chunks", T=700, E=4, k=2, H=128, I=128),                  # > 256 rows per expert: split into chunks
    syn.small("pf_sparse", T=9, E=64, k=8, H=128, I=64),                    # 72 rows over 64 experts: most empty
    syn.small("pf_mx_chunks", T=520, E=2, k=1, H=192, I=192, fmt=1),        # MXFP4, 260 rows each, H % 128 = 64
    syn.small("pf_min_dims", T=40, E=4, k=2, H=64, I=64),                    # one 64-deep stage, half a column tile
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_prefill_small(qgpu, oracle, wl):
    L = syn.layer(wl, 21)
    got, ids = _run(qgpu, wl, L)
    assert np.array_equal(ids, oracle.route(L["logits"], wl.k, wl.normalize)["ids"])
    err, elem = row_rel_l2(got, _ref(oracle, wl, L))
    assert err <= OUTPUT_RTOL, (wl.name, err, elem)


@pytest.mark.parametrize("wl", SMALL[:2] + SMALL[5:6], ids=lambda w: w.name)
def test_prefill_kmajor_and_dequantised(qgpu, oracle, wl):
    L = syn.layer(wl, 22)
    ref = _ref(oracle, wl, L)
    for kw in (dict(kmajor=True), dict(dequantised=True), dict(dequantised="fc1"),
               dict(dequantised="fc2", kmajor=True)):
        got, _ = _run(qgpu, wl, L, **kw)
        err, elem = row_rel_l2(got, ref)
        assert err <= OUTPUT_RTOL, (wl.name, kw, err, elem)


def test_prefill_workload_sampled_tokens(qgpu, oracle):
    """The 2048-token prefill workload (128 experts, top-8, H = 2048,
    I = 1536) in full on the GPU; the oracle checks 128 tokens drawn by seed
    (plus the first and last token), every expert they route to included."""
    wl = syn.WORKLOADS["nvfp4_prefill"]
    L = syn.layer(wl, 0)
    got, ids = _run(qgpu, wl, L)
    assert np.array_equal(ids, oracle.route(L["logits"], wl.k, wl.normalize)["ids"])
    draw = np.random.default_rng(5).choice(np.arange(1, wl.T - 1), size=126, replace=False)
    tokens = np.sort(np.concatenate([[0, wl.T - 1], draw]))
    assert len(tokens) == 128
    err, elem = row_rel_l2(got[tokens], _ref(oracle, wl, L, tokens=tokens))
    assert err <= OUTPUT_RTOL, (err, elem)
