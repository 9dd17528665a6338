"""router_weights (operator input 14) on the GPU against the oracle: the
logits select (ids and maps bit-exact), the mixing weights are router_weights
gathered at the selected experts (renormalised over the k when asked), on the
routing entry point, both decode kernels, both scale layouts and the prefill
path."""
import numpy as np
import pytest
import torch

import synthetic as syn
from helpers import OUTPUT_RTOL, bf16_tensor_bits, row_rel_l2, to_dev

pytestmark = pytest.mark.gpu

# gathered weights are exact; renormalising adds an fp32 sum of k <= 8 terms
# and a division
W_RTOL = 2e-6


def _mix(T, E, seed):
    return np.random.default_rng(seed).uniform(0.05, 2.0, (T, E)).astype(np.float32)


@pytest.mark.parametrize("T,E,k", [(4, 256, 8), (8, 32, 4), (1, 8, 2), (200, 256, 8), (65, 64, 3)])
@pytest.mark.parametrize("normalize", [0, 1])
def test_route_router_weights(qgpu, oracle, T, E, k, normalize):
    rng = np.random.default_rng(T + E + k)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    rw = _mix(T, E, 7)
    r = qgpu.route_topk(torch.from_numpy(lg).cuda(), k, normalize, router_weights=torch.from_numpy(rw).cuda())
    torch.cuda.synchronize()
    ref = oracle.route(lg, k, normalize, router_weights=rw)
    assert np.array_equal(r["ids"].cpu().numpy(), ref["ids"])
    assert np.array_equal(r["expanded_to_perm"].cpu().numpy(), ref["expanded_to_perm"])
    np.testing.assert_allclose(r["weights"].cpu().numpy(), ref["weights"], rtol=W_RTOL, atol=1e-30)


def _forward(qgpu, oracle, wl, seed, kmajor=False, multirow=False):
    L = syn.layer(wl, seed)
    rw = _mix(wl.T, wl.E, seed + 100)
    d = to_dev(L)
    s1, s2, fmt = d["s1"], d["s2"], wl.fmt
    if kmajor:
        s1, s2 = qgpu.scales_kmajor(s1, wl.fmt), qgpu.scales_kmajor(s2, wl.fmt)
        fmt |= qgpu.SCALES_KMAJOR | (qgpu.DECODE_MULTIROW if multirow else 0)
    ids = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    out = qgpu.moe_forward(d["x"], d["logits"], d["w1"], s1, d["g1"], d["w2"], s2, d["g2"], fmt, wl.k,
                           wl.normalize, wl.alpha, wl.beta, wl.limit, topk_ids=ids,
                           router_weights=torch.from_numpy(rw).cuda())
    torch.cuda.synchronize()
    ref = oracle.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"],
                             wl.fmt, wl.k, wl.normalize, wl.alpha, wl.beta, wl.limit, router_weights=rw)
    assert np.array_equal(ids.cpu().numpy(), oracle.route(L["logits"], wl.k, wl.normalize)["ids"])
    err, elem = row_rel_l2(bf16_tensor_bits(out), ref)
    assert err <= OUTPUT_RTOL, (wl.name, err, elem)
    # the mixing weights change the layer (compared with the softmax-mixed oracle)
    base = oracle.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"],
                              wl.fmt, wl.k, wl.normalize, wl.alpha, wl.beta, wl.limit)
    assert row_rel_l2(bf16_tensor_bits(out), base)[0] > 2 * OUTPUT_RTOL


@pytest.mark.parametrize("name", ["nvfp4_mtp_decode", "mxfp4_decode"])
@pytest.mark.parametrize("layout", ["page", "kmajor", "kmajor_multirow"])
def test_forward_router_weights_decode(qgpu, oracle, name, layout):
    _forward(qgpu, oracle, syn.WORKLOADS[name], seed=1, kmajor=layout != "page",
             multirow=layout == "kmajor_multirow")


@pytest.mark.parametrize("wl", [syn.small("rw_nonorm", T=4, E=32, k=4, H=256, I=192, normalize=0),
                                syn.small("rw_prefill", T=20, E=16, k=4, H=256, I=128),
                                syn.small("rw_prefill_mx", T=40, E=8, k=2, H=320, I=192, fmt=1)],
                         ids=lambda w: w.name)
def test_forward_router_weights_small(qgpu, oracle, wl):
    _forward(qgpu, oracle, wl, seed=3)
    _forward(qgpu, oracle, wl, seed=3, kmajor=True, multirow=wl.T * wl.k <= 64)
