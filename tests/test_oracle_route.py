"""Pins of the oracle's routing and permute-by-expert maps: brute force with
Python's own sort and math.exp on small inputs, numpy's stable argsort for the
maps, and the special cases (all-equal logits, E == k, k == 1, +-0.0 ties)."""
import math

import numpy as np
import pytest

import synthetic as syn


def _brute(logits, k, normalize):
    T, E = logits.shape
    ids = np.zeros((T, k), np.int64)
    w = np.zeros((T, k))
    for t in range(T):
        row = [float(v) for v in logits[t]]
        order = sorted(range(E), key=lambda e: (-row[e], e))[:k]
        mx = max(row)
        den = math.fsum(math.exp(v - mx) for v in row)
        p = [math.exp(row[e] - mx) / den for e in order]
        if normalize:
            s = math.fsum(p)
            p = [v / s for v in p]
        ids[t] = order
        w[t] = p
    return ids, w


@pytest.mark.parametrize("E,k", [(6, 1), (6, 2), (6, 6), (33, 8), (256, 8), (8, 2)])
@pytest.mark.parametrize("normalize", [0, 1])
def test_route_matches_brute_force(oracle, E, k, normalize):
    rng = np.random.default_rng(E * 100 + k)
    lg = rng.standard_normal((37, E)).astype(np.float32)
    lg[::5, : E // 2] = lg[::5, E // 2: 2 * (E // 2)]      # exact duplicates
    r = oracle.route(lg, k, normalize)
    ids, w = _brute(lg, k, normalize)
    assert np.array_equal(r["ids"], ids)
    np.testing.assert_allclose(r["weights"], w, rtol=1e-13, atol=0)


def test_route_ties_workload(oracle):
    wl = syn.WORKLOADS["nvfp4_verify_edge"]
    lg = syn.logits(syn.rng_for(0, 1), wl.T, wl.E, wl.logit_std, True, wl.k)
    r = oracle.route(lg, wl.k, 1)
    ids, _ = _brute(lg, wl.k, 1)
    assert np.array_equal(r["ids"], ids)
    # every row has a tie decided by the index rule at the k-th place
    for t in range(wl.T):
        kth = lg[t, ids[t, -1]]
        assert np.sum(lg[t] == kth) >= 2


def test_all_equal_logits(oracle):
    lg = np.full((3, 16), 0.25, np.float32)
    r = oracle.route(lg, 4, 1)
    assert np.array_equal(r["ids"], np.tile(np.arange(4), (3, 1)))
    np.testing.assert_allclose(r["weights"], 0.25, rtol=1e-15)
    r0 = oracle.route(lg, 4, 0)
    np.testing.assert_allclose(r0["weights"], 1.0 / 16, rtol=1e-15)


def test_e_equals_k_selects_all(oracle):
    rng = np.random.default_rng(1)
    lg = rng.standard_normal((5, 8)).astype(np.float32)
    r = oracle.route(lg, 8, 0)
    for t in range(5):
        assert sorted(r["ids"][t].tolist()) == list(range(8))
        np.testing.assert_allclose(r["weights"][t].sum(), 1.0, rtol=1e-14)
        assert np.all(np.diff(lg[t, r["ids"][t]]) <= 0)


def test_signed_zero_tie(oracle):
    lg = np.array([[-0.0, 0.0, -1.0]], np.float32)
    assert oracle.route(lg, 1, 1)["ids"].tolist() == [[0]]
    lg = np.array([[0.0, -0.0, -1.0]], np.float32)
    assert oracle.route(lg, 2, 1)["ids"].tolist() == [[0, 1]]


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (4, 256, 8), (8, 32, 4), (64, 16, 3), (300, 128, 8)])
def test_maps_are_stable_rank_by_expert(oracle, T, E, k):
    rng = np.random.default_rng(T + E + k)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    r = oracle.route(lg, k, 1)
    flat = r["ids"].reshape(-1)
    # offsets: exclusive scan of the per-expert counts
    counts = np.bincount(flat, minlength=E)
    assert np.array_equal(r["offsets"], np.concatenate([[0], np.cumsum(counts)]))
    # permuted order = stable sort of expanded indices by expert
    assert np.array_equal(r["perm_to_expanded"], np.argsort(flat, kind="stable"))
    inv = np.empty_like(r["perm_to_expanded"])
    inv[r["perm_to_expanded"]] = np.arange(T * k)
    assert np.array_equal(r["expanded_to_perm"], inv)


# ---- router_weights (operator input 14) -------------------------------------------

@pytest.mark.parametrize("normalize", [0, 1])
def test_router_weights_gathered_at_the_selection(oracle, normalize):
    """The logits alone select (same ids as without router_weights); the weights
    are router_weights at the selected experts, renormalised over the k when
    asked (brute force with Python's sort and math.fsum)."""
    rng = np.random.default_rng(21)
    logits = rng.standard_normal((5, 33)).astype(np.float32)
    rw = rng.uniform(0.01, 3.0, (5, 33)).astype(np.float32)
    r = oracle.route(logits, 8, normalize, router_weights=rw)
    ids, _ = _brute(logits, 8, normalize)
    assert np.array_equal(r["ids"], ids)
    assert np.array_equal(r["ids"], oracle.route(logits, 8, normalize)["ids"])
    for t in range(5):
        p = [float(rw[t][e]) for e in ids[t]]
        if normalize:
            s = math.fsum(p)
            p = [v / s for v in p]
        assert np.allclose(r["weights"][t], p, rtol=1e-15, atol=0)


def test_router_weights_special_cases(oracle):
    rng = np.random.default_rng(22)
    logits = rng.standard_normal((3, 16)).astype(np.float32)
    const = np.full((3, 16), 0.375, np.float32)
    assert np.all(oracle.route(logits, 4, 1, router_weights=const)["weights"] == 0.25)  # 1/k exactly
    assert np.all(oracle.route(logits, 4, 0, router_weights=const)["weights"] == 0.375)
    # the softmax of the logits as router_weights gives the default weights
    # (up to the fp32 rounding of the supplied probabilities)
    l64 = logits.astype(np.float64)
    prob = np.exp(l64 - l64.max(1, keepdims=True))
    prob = (prob / prob.sum(1, keepdims=True)).astype(np.float32)
    for normalize in (0, 1):
        a = oracle.route(logits, 4, normalize, router_weights=prob)["weights"]
        b = oracle.route(logits, 4, normalize)["weights"]
        assert np.allclose(a, b, rtol=2e-7, atol=0)
