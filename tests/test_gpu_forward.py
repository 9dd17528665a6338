"""The MoE layer on the GPU against the oracle (row-L2 relative error <= 1e-2),
on every decode workload at full size and on edge cases."""
import math

import numpy as np
import pytest
import torch

import synthetic as syn
from helpers import OUTPUT_RTOL, bf16_tensor_bits, row_rel_l2, to_dev

pytestmark = pytest.mark.gpu


def _gpu_forward(qgpu, L, wl, **kw):
    d = to_dev(L)
    ids = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    out = qgpu.moe_forward(d["x"], d["logits"], d["w1"], d["s1"], d["g1"], d["w2"], d["s2"], d["g2"],
                           wl.fmt, wl.k, wl.normalize, wl.alpha, wl.beta, wl.limit, topk_ids=ids, **kw)
    torch.cuda.synchronize()
    return bf16_tensor_bits(out), ids.cpu().numpy()


def _oracle_forward(oracle, L, wl, tokens=None):
    return oracle.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"],
                              L["g2"], wl.fmt, wl.k, wl.normalize, wl.alpha, wl.beta, wl.limit,
                              tokens=tokens)


def _check(qgpu, oracle, wl, seed=0, L=None):
    L = L if L is not None else syn.layer(wl, seed)
    got, ids = _gpu_forward(qgpu, L, wl)
    ref = _oracle_forward(oracle, L, wl)
    assert np.array_equal(ids, oracle.route(L["logits"], wl.k, wl.normalize)["ids"])
    err, elem = row_rel_l2(got, ref)
    assert err <= OUTPUT_RTOL, (wl.name, err, elem)
    return err


DECODE = ["tiny_nvfp4_decode", "nvfp4_mtp_decode", "mxfp4_decode", "nvfp4_verify_edge"]


@pytest.mark.parametrize("name", DECODE)
def test_forward_decode_workloads(qgpu, oracle, name):
    _check(qgpu, oracle, syn.WORKLOADS[name], seed=0)


@pytest.mark.parametrize("seed", [1, 2])
@pytest.mark.parametrize("name", DECODE[1:])
def test_forward_decode_workloads_more_seeds(qgpu, oracle, name, seed):
    _check(qgpu, oracle, syn.WORKLOADS[name], seed=seed)


EDGE = [
    syn.small("t1k1", T=1, E=4, k=1, H=64, I=64),
    syn.small("e_eq_k", T=3, E=4, k=4, H=128, I=64),
    syn.small("rows64_k1", T=64, E=8, k=1, H=128, I=128),            # many rows per expert
    syn.small("window_edge", T=8, E=16, k=8, H=256, I=128),           # R = 64 exactly
    syn.small("nonorm", T=4, E=32, k=4, H=256, I=192, normalize=0),
    syn.small("gptoss", T=4, E=32, k=4, H=192, I=128, fmt=1, alpha=1.702, beta=1.0, limit=7.0),
    syn.small("mx_odd_tiles", T=2, E=8, k=2, H=2880, I=320, fmt=1),   # N/64 odd, K/32 ragged
    syn.small("nv_ragged", T=5, E=9, k=3, H=320, I=448),
]


@pytest.mark.parametrize("wl", EDGE, ids=lambda w: w.name)
def test_forward_edge_cases(qgpu, oracle, wl):
    _check(qgpu, oracle, wl, seed=11)


def test_forward_all_tokens_same_expert(qgpu, oracle):
    wl = syn.small("same", T=16, E=8, k=2, H=256, I=128)
    L = syn.layer(wl, seed=3)
    L["logits"][:, 5] += 10.0
    L["logits"][:, 2] += 9.0
    _check(qgpu, oracle, wl, L=L)


def test_forward_large_activations_stay_exact_range(qgpu, oracle):
    """Activations far outside fp16 range (and tiny ones) are handled by the
    per-row power-of-two rescale."""
    wl = syn.small("range", T=3, E=4, k=2, H=256, I=128)
    L = syn.layer(wl, seed=4)
    x = L["x"].view(np.uint16)
    f = (x.astype(np.uint32) << 16).view(np.float32)
    f[0] *= 3.0e6
    f[1] *= 1.0e-9
    L["x"] = syn.to_bf16_bits(f)
    _check(qgpu, oracle, wl, L=L)


def test_forward_non_power_of_two_global_scales(qgpu, oracle):
    wl = syn.small("g", T=4, E=8, k=2, H=256, I=128)
    L = syn.layer(wl, seed=5)
    L["g1"] = np.linspace(0.013, 1.7, 8).astype(np.float32)
    L["g2"] = np.linspace(3.1, 0.07, 8).astype(np.float32)
    _check(qgpu, oracle, wl, L=L)


def test_forward_repeat_is_deterministic(qgpu):
    wl = syn.WORKLOADS["nvfp4_mtp_decode"]
    L = syn.layer(wl, seed=0)
    a, _ = _gpu_forward(qgpu, L, wl)
    b, _ = _gpu_forward(qgpu, L, wl)
    assert np.array_equal(a, b)


def test_forward_poisoned_workspace(qgpu):
    """Workspace contents left by anything else never change the output."""
    wl = syn.WORKLOADS["nvfp4_mtp_decode"]
    L = syn.layer(wl, seed=1)
    d = to_dev(L)
    need = qgpu.forward_workspace_bytes(wl.T, wl.H, wl.I, wl.E, wl.k, wl.fmt)
    outs = []
    for fill in (0x00, 0xFF, 0x7F, 0x80):
        ws = torch.full((need,), fill, dtype=torch.uint8, device="cuda")
        out = qgpu.moe_forward(d["x"], d["logits"], d["w1"], d["s1"], d["g1"], d["w2"], d["s2"],
                               d["g2"], wl.fmt, wl.k, workspace=ws)
        torch.cuda.synchronize()
        outs.append(bf16_tensor_bits(out))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_forward_errors_launch_nothing(qgpu):
    wl = syn.small("err", T=2, E=4, k=2, H=64, I=64)
    d = to_dev(syn.layer(wl, seed=1))
    with pytest.raises(qgpu.QMoEError) as ei:
        qgpu.moe_forward(d["x"], d["logits"], d["w1"], d["s1"], d["g1"], d["w2"], d["s2"], d["g2"],
                         0, 5)
    assert ei.value.status == 1
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(qgpu.QMoEError) as ei:
        qgpu.moe_forward(d["x"], d["logits"], d["w1"], d["s1"], d["g1"], d["w2"], d["s2"], d["g2"],
                         0, 2, workspace=small)
    assert ei.value.status == 4
    xs = torch.empty(2 * 64 + 1, dtype=torch.bfloat16, device="cuda")[1:].view(2, 64)
    with pytest.raises(qgpu.QMoEError) as ei:
        qgpu.moe_forward(xs, d["logits"], d["w1"], d["s1"], d["g1"], d["w2"], d["s2"], d["g2"], 0, 2)
    assert ei.value.status == 2
