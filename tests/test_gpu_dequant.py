"""FP4 -> bf16 dequantisation on the GPU against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import synthetic as syn
from helpers import bf16_tensor_bits

pytestmark = pytest.mark.gpu
NV, MX = 0, 1


def _run(qgpu, w, s, g, fmt):
    dw = torch.from_numpy(w).cuda()
    ds = torch.from_numpy(s).cuda()
    dg = None if g is None else torch.from_numpy(g).cuda()
    out = qgpu.dequant(dw, ds, dg, fmt)
    torch.cuda.synchronize()
    return bf16_tensor_bits(out)


def _same(got, ref):
    nan_g, nan_r = (got & 0x7FFF) > 0x7F80, (ref & 0x7FFF) > 0x7F80
    assert np.array_equal(nan_g, nan_r)
    bad = np.argwhere((got != ref) & ~nan_r)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:5].tolist()}"


@pytest.mark.parametrize("fmt", [NV, MX])
@pytest.mark.parametrize("E,N,K", [(1, 64, 64), (3, 128, 192), (2, 192, 128), (1, 64, 2880), (1, 2880, 64)])
def test_dequant_bit_exact_small(qgpu, oracle, fmt, E, N, K):
    rng = syn.rng_for(E * N + K, fmt)
    w, s, g = syn.expert_weights(rng, fmt, E, K, N)
    _same(_run(qgpu, w, s, g, fmt), oracle.dequant(w, s, g, fmt))


@pytest.mark.parametrize("fmt", [NV, MX])
def test_dequant_every_code_and_scale(qgpu, oracle, fmt):
    """All 16 codes against all 256 scale bytes (NaN codes, subnormals, zero)."""
    bs = 16 if fmt == NV else 32
    E, N, K = 2, 256, 16 * bs
    rng = syn.rng_for(99, fmt)
    w = syn.uniform_bytes(rng, (E, K, N // 2))
    s = np.tile(np.arange(256, dtype=np.uint8)[:, None], (E, 1, K // bs))   # row n -> scale byte n
    g = np.array([1.0, 0.125], np.float32) if fmt == NV else None
    _same(_run(qgpu, w, s, g, fmt), oracle.dequant(w, s, g, fmt))


def test_dequant_non_power_of_two_global_scale(qgpu, oracle):
    """An arbitrary fp32 global scale takes the exact-product path."""
    E, N, K = 4, 128, 128
    rng = syn.rng_for(5, 5)
    w, s, _ = syn.expert_weights(rng, NV, E, K, N)
    s[:, :, :] = syn.uniform_bytes(rng, s.shape)           # every E4M3 code
    g = np.array([0.3, 1.7e-3, 1234.567, 3.0e-39], np.float32)
    _same(_run(qgpu, w, s, g, NV), oracle.dequant(w, s, g, NV))


def test_dequant_mxfp4_with_global_scale(qgpu, oracle):
    E, N, K = 3, 64, 256
    rng = syn.rng_for(6, 6)
    w = syn.uniform_bytes(rng, (E, K, N // 2))
    s = syn.uniform_bytes(rng, (E, N, K // 32))            # every E8M0 code incl. 0 and 255
    g = np.array([1.0, 0.5, 2.5], np.float32)
    _same(_run(qgpu, w, s, g, MX), oracle.dequant(w, s, g, MX))


@pytest.mark.parametrize("fc", ["fc1", "fc2"])
def test_dequant_prefill_size_whole_tensor(qgpu, oracle, fc):
    """The prefill workload's dequantisations at full size, in the launch
    configuration the benchmark uses, compared with the oracle bit for bit over
    the whole tensor: FC1 [128, 2048, 1536] -> [128, 3072, 2048] and FC2
    [128, 1536, 1024] -> [128, 2048, 1536]."""
    wl = syn.WORKLOADS["nvfp4_prefill"]
    K, N = (wl.H, 2 * wl.I) if fc == "fc1" else (wl.I, wl.H)
    rng = syn.rng_for(0, 7 if fc == "fc1" else 8)
    w, s, g = syn.expert_weights(rng, NV, wl.E, K, N)
    got = _run(qgpu, w, s, g, NV)
    assert got.shape == (wl.E, N, K)
    ref = oracle.dequant(w, s, g, NV)
    _same(got, ref)
