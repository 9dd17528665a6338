"""Routing and permute-by-expert maps on the GPU against the oracle:
bit-exact ids and maps, weights within the fp32 softmax error bound."""
import numpy as np
import pytest
import torch

import synthetic as syn

pytestmark = pytest.mark.gpu

# fp32 softmax with a tree sum over E terms: relative error <= (log2(E) + 8) * 2^-24
# for the sum plus a few ulp for exp and the division.
W_RTOL = 2e-6


def _check(qgpu, oracle, lg, k, normalize=1):
    r = qgpu.route_topk(torch.from_numpy(lg).cuda(), k, normalize)
    torch.cuda.synchronize()
    ref = oracle.route(lg, k, normalize)
    assert np.array_equal(r["ids"].cpu().numpy(), ref["ids"])
    assert np.array_equal(r["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(r["perm_to_expanded"].cpu().numpy(), ref["perm_to_expanded"])
    assert np.array_equal(r["expanded_to_perm"].cpu().numpy(), ref["expanded_to_perm"])
    np.testing.assert_allclose(r["weights"].cpu().numpy(), ref["weights"], rtol=W_RTOL, atol=1e-30)


@pytest.mark.parametrize("name", list(syn.WORKLOADS))
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_route_workloads(qgpu, oracle, name, seed):
    wl = syn.WORKLOADS[name]
    lg = syn.logits(syn.rng_for(seed, 1), wl.T, wl.E, wl.logit_std, wl.ties, wl.k)
    _check(qgpu, oracle, lg, wl.k, wl.normalize)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (1, 8, 8), (3, 33, 5), (64, 256, 1), (65, 64, 8),
                                   (200, 256, 8), (7, 100, 3), (1, 256, 8), (33, 32, 2)])
@pytest.mark.parametrize("normalize", [0, 1])
def test_route_shapes(qgpu, oracle, T, E, k, normalize):
    rng = np.random.default_rng(T * 1000 + E + k)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    _check(qgpu, oracle, lg, k, normalize)


def test_route_ties_and_signed_zero(qgpu, oracle):
    rng = np.random.default_rng(5)
    lg = rng.integers(-3, 3, size=(40, 64)).astype(np.float32)   # many exact ties
    lg[0] = 0.0
    lg[1, ::2] = -0.0
    lg[2] = 1.25
    _check(qgpu, oracle, lg, 8, 1)
    _check(qgpu, oracle, lg, 8, 0)


def test_route_all_tokens_one_expert(qgpu, oracle):
    lg = np.zeros((64, 16), np.float32)
    lg[:, 11] = 5.0
    _check(qgpu, oracle, lg, 1, 1)
