"""k-major block scales on the GPU: the conversion is bit-exact against the
oracle, and the layer on k-major scales matches the oracle (row-L2 relative
error <= 1e-2) on every decode workload and on edge cases, with the decode
kernel chosen by the shape and with the multi-row kernel forced."""
import numpy as np
import pytest
import torch

import synthetic as syn
from helpers import OUTPUT_RTOL, bf16_tensor_bits, row_rel_l2, to_dev

pytestmark = pytest.mark.gpu


# (E, N, blocks, format): one tile, ragged 64-block tiles, many tiles
@pytest.mark.parametrize("E,N,nb,fmt", [(1, 64, 4, 0), (3, 192, 90, 1), (2, 128, 6, 1), (2, 64, 12, 0),
                                        (5, 1024, 128, 0), (7, 2880, 90, 1)])
def test_scales_kmajor_bit_exact(qgpu, oracle, E, N, nb, fmt):
    rng = np.random.default_rng(E * 1000 + nb)
    s = rng.integers(0, 256, (E, N, nb), dtype=np.uint8)
    got = qgpu.scales_kmajor(torch.from_numpy(s).cuda(), fmt)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), oracle.scales_kmajor(s))


def test_scales_kmajor_full_size(qgpu, oracle):
    # the FC1 scales of the 256-expert NVFP4 decode shape (H = 2048, 2I = 1024)
    L = syn.layer(syn.WORKLOADS["nvfp4_mtp_decode"], 0)
    got = qgpu.scales_kmajor(torch.from_numpy(L["s1"]).cuda(), qgpu.NVFP4)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), oracle.scales_kmajor(L["s1"]))


def _check_kmajor(qgpu, oracle, wl, seed, multirow=False):
    L = syn.layer(wl, seed)
    d = to_dev(L)
    s1 = qgpu.scales_kmajor(d["s1"], wl.fmt)
    s2 = qgpu.scales_kmajor(d["s2"], wl.fmt)
    ids = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    out = qgpu.moe_forward(d["x"], d["logits"], d["w1"], s1, d["g1"], d["w2"], s2, d["g2"],
                           wl.fmt | qgpu.SCALES_KMAJOR | (qgpu.DECODE_MULTIROW if multirow else 0), wl.k,
                           wl.normalize, wl.alpha, wl.beta, wl.limit,
                           topk_ids=ids)
    torch.cuda.synchronize()
    ref = oracle.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"],
                             wl.fmt, wl.k, wl.normalize, wl.alpha, wl.beta, wl.limit)
    assert np.array_equal(ids.cpu().numpy(), oracle.route(L["logits"], wl.k, wl.normalize)["ids"])
    err, elem = row_rel_l2(bf16_tensor_bits(out), ref)
    assert err <= OUTPUT_RTOL, (wl.name, err, elem)


DECODE = ["tiny_nvfp4_decode", "nvfp4_mtp_decode", "mxfp4_decode", "nvfp4_verify_edge"]


@pytest.mark.parametrize("name", DECODE)
def test_forward_kmajor_decode_workloads(qgpu, oracle, name):
    _check_kmajor(qgpu, oracle, syn.WORKLOADS[name], seed=0)


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("name", DECODE)
def test_forward_kmajor_multirow_workloads(qgpu, oracle, name, seed):
    _check_kmajor(qgpu, oracle, syn.WORKLOADS[name], seed=seed, multirow=True)


EDGE = [
    syn.small("t1k1", T=1, E=4, k=1, H=64, I=64),
    syn.small("rows64_k1", T=64, E=8, k=1, H=128, I=128),
    syn.small("nonorm", T=4, E=32, k=4, H=256, I=192, normalize=0),
    syn.small("gptoss", T=4, E=32, k=4, H=192, I=128, fmt=1, alpha=1.702, beta=1.0, limit=7.0),
    syn.small("mx_odd_tiles", T=2, E=8, k=2, H=2880, I=320, fmt=1),
    syn.small("nv_ragged", T=5, E=9, k=3, H=320, I=448),
    syn.small("wide_n", T=2, E=4, k=2, H=4096, I=2048),               # N = 4096: 4 blocks per window
]


@pytest.mark.parametrize("multirow", [False, True])
@pytest.mark.parametrize("wl", EDGE, ids=lambda w: w.name)
def test_forward_kmajor_edge_cases(qgpu, oracle, wl, multirow):
    _check_kmajor(qgpu, oracle, wl, seed=13, multirow=multirow)


def test_kmajor_api_errors(qgpu):
    s = torch.zeros((2, 64, 4), dtype=torch.uint8, device="cuda")
    with pytest.raises(qgpu.QMoEError) as ei:   # the multi-row kernel takes k-major scales only
        qgpu.forward_workspace_bytes(4, 256, 128, 8, 2, qgpu.NVFP4 | qgpu.DECODE_MULTIROW)
    assert ei.value.status == 3
    with pytest.raises(qgpu.QMoEError) as ei:   # dequant takes the page layout only
        qgpu.dequant(torch.zeros((2, 64, 32), dtype=torch.uint8, device="cuda"), s, None,
                     qgpu.NVFP4 | qgpu.SCALES_KMAJOR)
    assert ei.value.status == 3
    with pytest.raises(qgpu.QMoEError) as ei:   # in place is refused
        qgpu.scales_kmajor(s, qgpu.NVFP4, out=s.view(2, 4, 64))
    assert ei.value.status == 1
    with pytest.raises(qgpu.QMoEError) as ei:   # misaligned output
        buf = torch.zeros(2 * 64 * 4 + 16, dtype=torch.uint8, device="cuda")
        qgpu.scales_kmajor(s, qgpu.NVFP4, out=buf[1:1 + 2 * 64 * 4].view(2, 4, 64))
    assert ei.value.status == 2
