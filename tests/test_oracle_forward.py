"""Pins of the oracle's layer: a dense brute force (torch fp64 matmul on the
dequantised matrices, routing by Python sort, no permutation), a one-hot
activation, exact scaling by the global scales, and the token subset."""
import math

import numpy as np
import pytest
import torch

import synthetic as syn
from helpers import concatenated_fc1

NV, MX = 0, 1


def _f(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_round(a):
    """Round float64 -> bf16 via an exactness-preserving path: torch rounds
    float64 -> bfloat16 directly."""
    return torch.from_numpy(np.asarray(a, np.float64)).to(torch.bfloat16).to(torch.float64).numpy()


def _dense_layer(oracle, L, wl, fusion=1, router_weights=None):
    x = torch.from_numpy(_f(L["x"]))
    W1 = torch.from_numpy(_f(oracle.dequant(L["w1"], L["s1"], L["g1"], wl.fmt)))  # [E,2I,H]
    W2 = torch.from_numpy(_f(oracle.dequant(L["w2"], L["s2"], L["g2"], wl.fmt)))  # [E,H,I]
    T = x.shape[0]
    out = torch.zeros(T, wl.H, dtype=torch.float64)
    for t in range(T):
        row = [float(v) for v in L["logits"][t]]
        order = sorted(range(wl.E), key=lambda e: (-row[e], e))[: wl.k]
        mx = max(row)
        den = math.fsum(math.exp(v - mx) for v in row)
        p = [math.exp(row[e] - mx) / den for e in order]
        if router_weights is not None:  # selection by the logits, mixing by router_weights
            p = [float(router_weights[t][e]) for e in order]
        if wl.normalize:
            s = math.fsum(p)
            p = [v / s for v in p]
        for j, e in enumerate(order):
            h = W1[e] @ x[t]
            if fusion == 2:
                gate, lin = h[: wl.I].numpy(), h[wl.I:].numpy()
            else:
                gate, lin = h[0::2].numpy(), h[1::2].numpy()
            act = np.array([oracle.swiglu(a, b, wl.alpha, wl.beta, wl.limit)
                            for a, b in zip(gate, lin)])
            a = torch.from_numpy(_bf16_round(act))
            out[t] += p[j] * (W2[e] @ a)
    return out.numpy()


CASES = [
    syn.small("nv", T=3, E=6, k=2, H=64, I=32, fmt=NV),
    syn.small("nv_nonorm", T=2, E=5, k=3, H=32, I=16, fmt=NV, normalize=0),
    syn.small("mx", T=3, E=4, k=2, H=64, I=64, fmt=MX),
    syn.small("gptoss", T=2, E=4, k=2, H=64, I=32, fmt=MX, alpha=1.702, beta=1.0, limit=7.0),
    syn.small("ek", T=2, E=3, k=3, H=32, I=32, fmt=NV),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_layer_matches_dense_brute_force(oracle, wl):
    L = syn.layer(wl, seed=3)
    got = _f(oracle.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"],
                                L["s2"], L["g2"], wl.fmt, wl.k, wl.normalize, wl.alpha,
                                wl.beta, wl.limit))
    ref = _dense_layer(oracle, L, wl)
    ref_bf = _bf16_round(ref)
    # identical up to summation order: at most one bf16 ulp apart, mostly equal
    ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8)
    assert np.all(np.abs(got - ref_bf) <= ulp + 1e-300)
    assert np.mean(got == ref_bf) > 0.97


def test_one_hot_activation_reads_a_dequantised_column(oracle):
    wl = syn.small("oh", T=1, E=3, k=1, H=64, I=16, fmt=NV)
    L = syn.layer(wl, seed=4)
    W1 = _f(oracle.dequant(L["w1"], L["s1"], L["g1"], NV))
    for e in range(3):
        for k0 in (0, 5, 63):
            x = np.zeros(64, np.uint16)
            x[k0] = 0x3F80  # bf16 1.0
            h = oracle.expert_fc1(x, e, L["w1"], L["s1"], L["g1"], NV)
            assert np.array_equal(h, W1[e, :, k0])


def test_global_scales_scale_exactly(oracle):
    wl = syn.small("sc", T=1, E=2, k=1, H=64, I=32, fmt=NV)
    L = syn.layer(wl, seed=5)
    x = L["x"][0]
    h1 = oracle.expert_fc1(x, 1, L["w1"], L["s1"], L["g1"], NV)
    h2 = oracle.expert_fc1(x, 1, L["w1"], L["s1"], L["g1"] * 2, NV)
    assert np.array_equal(h2, 2 * h1)
    a = _f(syn.to_bf16_bits(np.random.default_rng(0).standard_normal(32)))
    y1 = oracle.expert_fc2(a, 0, L["w2"], L["s2"], L["g2"], NV)
    y2 = oracle.expert_fc2(a, 0, L["w2"], L["s2"], L["g2"] * 0.25, NV)
    assert np.array_equal(y2, 0.25 * y1)


def test_token_subset(oracle):
    wl = syn.small("sub", T=5, E=6, k=2, H=32, I=16, fmt=NV)
    L = syn.layer(wl, seed=6)
    args = (L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"], NV, 2)
    full = oracle.moe_forward(*args)
    sub = oracle.moe_forward(*args, tokens=[4, 0, 2])
    assert np.array_equal(sub, full[[4, 0, 2]])
    with pytest.raises(ValueError):
        oracle.moe_forward(*args, tokens=[5])


def test_output_is_weighted_sum_of_expert_outputs(oracle):
    """k experts, one token: out = bf16(sum_j w_j y_j) with y_j from expert_ffn."""
    wl = syn.small("ws", T=1, E=5, k=3, H=32, I=32, fmt=MX)
    L = syn.layer(wl, seed=7)
    r = oracle.route(L["logits"], 3, 1)
    ys = [oracle.expert_ffn(L["x"][0], int(e), L["w1"], L["s1"], L["g1"], L["w2"], L["s2"],
                            L["g2"], MX) for e in r["ids"][0]]
    acc = sum(w * y for w, y in zip(r["weights"][0], ys))
    out = oracle.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"],
                             L["s2"], L["g2"], MX, 3)
    assert np.array_equal(out[0], np.array([oracle.bf16_rne(v) for v in acc], np.uint16))


# ---- swiglu_fusion: concatenated (2) and the remapped 0 ---------------------------

@pytest.mark.parametrize("wl", CASES[:4], ids=lambda w: w.name)
def test_concatenated_swiglu_matches_dense_brute_force(oracle, wl):
    """swiglu_fusion = 2 pairs column m (gate) with column I + m (linear)."""
    L = syn.layer(wl, seed=21)
    w1c, s1c = concatenated_fc1(L["w1"], L["s1"])
    Lc = dict(L, w1=w1c, s1=s1c)
    ref = _dense_layer(oracle, Lc, wl, fusion=2)
    got = _f(oracle.moe_forward(Lc["x"], Lc["logits"], Lc["w1"], Lc["s1"], Lc["g1"], Lc["w2"], Lc["s2"],
                                Lc["g2"], wl.fmt, wl.k, wl.normalize, wl.alpha, wl.beta, wl.limit,
                                fusion=2))
    np.testing.assert_allclose(got, ref, rtol=2 ** -7, atol=1e-6 * np.abs(ref).max())


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_concatenated_layout_is_a_column_permutation(oracle, wl):
    """The same weights, columns rewritten from interleaved to concatenated
    order, give the identical layer (every FC1 dot product is the same)."""
    L = syn.layer(wl, seed=22)
    args = (L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"], wl.fmt, wl.k,
            wl.normalize, wl.alpha, wl.beta, wl.limit)
    w1c, s1c = concatenated_fc1(L["w1"], L["s1"])
    interleaved = oracle.moe_forward(*args)
    concatenated = oracle.moe_forward(L["x"], L["logits"], w1c, s1c, *args[4:], fusion=2)
    assert np.array_equal(interleaved, concatenated)
    # read the other way round, the layouts differ (the pin is not vacuous)
    assert not np.array_equal(interleaved, oracle.moe_forward(*args, fusion=2))


def test_fusion_zero_reads_as_interleaved(oracle):
    wl = CASES[0]
    L = syn.layer(wl, seed=23)
    args = (L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"], L["g2"], wl.fmt, wl.k)
    assert np.array_equal(oracle.moe_forward(*args, fusion=0), oracle.moe_forward(*args, fusion=1))
    with pytest.raises(Exception):
        oracle.moe_forward(*args, fusion=3)


def test_concatenated_fc1_helper_moves_columns():
    """The test helper itself: one nonzero code per column lands where the
    concatenated order puts it, and the scales move with it."""
    E, H, I = 1, 2, 4
    w1 = np.zeros((E, H, I), np.uint8)
    s1 = np.zeros((E, 2 * I, 1), np.uint8)
    for n in range(2 * I):
        k = n % H
        w1[0, k, n // 2] |= np.uint8((n + 1) << (4 * (n % 2)))
        s1[0, n, 0] = n + 100
    w1c, s1c = concatenated_fc1(w1, s1)
    for c in range(2 * I):
        src = 2 * c if c < I else 2 * (c - I) + 1
        assert s1c[0, c, 0] == src + 100
        for k in range(H):
            code = (int(w1c[0, k, c // 2]) >> (4 * (c % 2))) & 0xF
            assert code == ((src + 1) if src % H == k else 0)


# ---- router_weights (operator input 14): the logits select, router_weights mix ----

@pytest.mark.parametrize("wl", CASES[:3], ids=lambda w: w.name)
def test_router_weights_layer_matches_dense_brute_force(oracle, wl):
    L = syn.layer(wl, seed=5)
    rw = np.random.default_rng(11).uniform(0.05, 2.0, (wl.T, wl.E)).astype(np.float32)
    got = _f(oracle.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"],
                                L["s2"], L["g2"], wl.fmt, wl.k, wl.normalize, wl.alpha,
                                wl.beta, wl.limit, router_weights=rw))
    ref = _dense_layer(oracle, L, wl, router_weights=rw)
    ref_bf = _bf16_round(ref)
    ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 8)
    assert np.all(np.abs(got - ref_bf) <= ulp + 1e-300)
    # and the mixing weights matter: the default path gives another layer
    base = _f(oracle.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"],
                                 L["s2"], L["g2"], wl.fmt, wl.k, wl.normalize, wl.alpha,
                                 wl.beta, wl.limit))
    assert not np.array_equal(base, got)


def test_router_weights_one_hot_is_one_expert(oracle):
    """router_weights 1 at each token's first selected expert and 0 elsewhere
    (no renormalisation): the layer is that one expert's FFN, exactly."""
    wl = syn.small("rw1", T=2, E=5, k=3, H=32, I=32, fmt=MX, normalize=0)
    L = syn.layer(wl, seed=9)
    ids = oracle.route(L["logits"], wl.k, 0)["ids"]
    rw = np.zeros((wl.T, wl.E), np.float32)
    for t in range(wl.T):
        rw[t, ids[t, 0]] = 1.0
    out = oracle.moe_forward(L["x"], L["logits"], L["w1"], L["s1"], L["g1"], L["w2"], L["s2"],
                             L["g2"], MX, wl.k, 0, router_weights=rw)
    for t in range(wl.T):
        y = oracle.expert_ffn(L["x"][t], int(ids[t, 0]), L["w1"], L["s1"], L["g1"], L["w2"],
                              L["s2"], L["g2"], MX)
        assert np.array_equal(out[t], np.array([oracle.bf16_rne(v) for v in y], np.uint16))
