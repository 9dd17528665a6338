"""Pins of the oracle's dequantisation: the [E,K,N/2] -> [E,N,K] index map and
the [E,N,K/bs] scale map by brute force on tiny one-hot inputs, exactness of
the products (power-of-two scales only shift exponents), and the rounding bound
for a non-power-of-two global scale."""
import math

import numpy as np
import pytest
import torch

import synthetic as syn

NV, MX = 0, 1
ONE_E4M3, TWO_E4M3 = 0x38, 0x40     # 1.0 and 2.0 in E4M3FN
ONE_E8M0, TWO_E8M0 = 127, 128


def _f(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("fmt", [NV, MX])
def test_index_map_one_hot(oracle, fmt):
    E, K, N = 2, 64, 64
    bs = 16 if fmt == NV else 32
    scales = np.full((E, N, K // bs), ONE_E4M3 if fmt == NV else ONE_E8M0, np.uint8)
    g = np.ones(E, np.float32) if fmt == NV else None
    rng = np.random.default_rng(11)
    positions = [(e, k, n) for e in range(E) for k in (0, 1, 17, 63) for n in range(N)]
    positions += [(int(rng.integers(E)), int(rng.integers(K)), int(rng.integers(N)))
                  for _ in range(64)]
    for e, k, n in positions:
        packed = np.zeros((E, K, N // 2), np.uint8)
        packed[e, k, n // 2] = 2 << (4 * (n % 2))           # code 2 = 1.0 at (e, k, n)
        out = _f(oracle.dequant(packed, scales, g, fmt))    # [E, N, K]
        nz = np.argwhere(out != 0.0)
        assert nz.tolist() == [[e, n, k]], (e, k, n, nz[:4])
        assert out[e, n, k] == 1.0


@pytest.mark.parametrize("fmt", [NV, MX])
def test_scale_map_one_hot(oracle, fmt):
    E, K, N = 2, 128, 8
    bs = 16 if fmt == NV else 32
    one, two = (ONE_E4M3, TWO_E4M3) if fmt == NV else (ONE_E8M0, TWO_E8M0)
    packed = np.full((E, K, N // 2), 0x22, np.uint8)        # every code = 1.0
    for e, n, b in [(0, 0, 0), (1, 7, K // bs - 1), (0, 3, 1), (1, 4, 2)]:
        scales = np.full((E, N, K // bs), one, np.uint8)
        scales[e, n, b] = two
        out = _f(oracle.dequant(packed, scales, None, fmt))
        expect = np.ones((E, N, K))
        expect[e, n, b * bs:(b + 1) * bs] = 2.0
        assert np.array_equal(out, expect), (e, n, b)


def test_global_scale_per_expert(oracle):
    E, K, N = 3, 32, 4
    packed = np.full((E, K, N // 2), 0x7F, np.uint8)        # codes 15 (-6) and 7 (6)
    scales = np.full((E, N, K // 16), ONE_E4M3, np.uint8)
    g = np.array([1.0, 0.5, 0.0625], np.float32)
    out = _f(oracle.dequant(packed, scales, g, NV))
    # byte 0x7F: low nibble 0xF (-6) is the even n, high nibble 0x7 (+6) the odd n
    for e in range(E):
        assert np.all(out[e, 0::2] == -6.0 * g[e])
        assert np.all(out[e, 1::2] == 6.0 * g[e])


def test_hand_worked_block(oracle):
    """One NVFP4 block worked by hand from the format definitions.
    k-row 0 bytes (0x21, 0xF8): n0 = code 1 (0.5), n1 = code 2 (1.0),
    n2 = code 8 (-0.0), n3 = code 15 (-6.0).  Scales: n0 0x38 = 1.0,
    n1 0x3C = 1.5, n2 0x08 = 2^-6, n3 0x41 = 2.25.  Global scale 0.5.
    Products: 0.25, 0.75, -0.0, -6.75 -- all exact bf16 values."""
    packed = np.zeros((1, 16, 2), np.uint8)
    packed[0, 0] = [0x21, 0xF8]
    scales = np.array([[[0x38], [0x3C], [0x08], [0x41]]], np.uint8)
    out = oracle.dequant(packed, scales, np.array([0.5], np.float32), NV)
    assert [hex(v) for v in out[0, :, 0]] == ["0x3e80", "0x3f40", "0x8000", "0xc0d8"]
    # every other k has code 0 -> +0.0
    assert np.all(out[0, :, 1:] == 0)


def _exact_products(w1, s1, g1, fmt, e, n, k):
    """Exact product from independent decoders: the printed E2M1 table and
    torch's float8 casts."""
    table = {0: 0.0, 1: 0.5, 2: 1.0, 3: 1.5, 4: 2.0, 5: 3.0, 6: 4.0, 7: 6.0}
    code = (int(w1[e, k, n // 2]) >> (4 * (n % 2))) & 15
    v = table[code & 7] * (-1.0 if code & 8 else 1.0)
    bs = 16 if fmt == NV else 32
    sb = torch.tensor([int(s1[e, n, k // bs])], dtype=torch.uint8)
    sdt = torch.float8_e4m3fn if fmt == NV else torch.float8_e8m0fnu
    s = float(sb.view(sdt).to(torch.float64))
    g = 1.0 if g1 is None else float(g1[e])
    return v * s * g


@pytest.mark.parametrize("fmt", [NV, MX])
def test_config_products_are_exact_bf16(oracle, fmt):
    """With the workloads' scales (power-of-two global / E8M0, 4-bit E4M3)
    every dequantised weight is the exact product: bf16 rounding is a no-op."""
    rng = syn.rng_for(5, 9)
    E, K, N = 4, 64, 32
    w, s, g = syn.expert_weights(rng, fmt, E, K, N)
    out = _f(oracle.dequant(w, s, g, fmt))
    for e in range(E):
        for n in range(N):
            for k in range(0, K, 3):
                assert out[e, n, k] == _exact_products(w, s, g, fmt, e, n, k)


def test_non_power_of_two_global_scale_rounds_once(oracle):
    """With an arbitrary fp32 global scale the value is the exact product
    rounded to the nearest bf16 (within half a bf16 ulp, and a bf16 value)."""
    rng = syn.rng_for(6, 9)
    E, K, N = 3, 32, 16
    w, s, _ = syn.expert_weights(rng, NV, E, K, N)
    g = np.array([0.3, 1.7e-3, 1234.567], np.float32)
    out = oracle.dequant(w, s, g, NV)
    vals = _f(out)
    for e in range(E):
        for n in range(N):
            for k in range(K):
                exact = _exact_products(w, s, g, NV, e, n, k)
                got = vals[e, n, k]
                if exact == 0.0:
                    assert got == 0.0
                    continue
                ulp = 2.0 ** (math.frexp(abs(exact))[1] - 8)
                assert abs(got - exact) <= ulp / 2, (e, n, k, got, exact)
                # the result is a bf16 value (low 16 bits of its float are zero)
                assert np.float32(got).view(np.uint32) & 0xFFFF == 0


def test_nan_scale_gives_nan(oracle):
    packed = np.full((1, 16, 1), 0x21, np.uint8)
    out = oracle.dequant(packed, np.array([[[0x7F], [0x38]]], np.uint8), None, NV)
    assert np.all(out[0, 0] == 0x7FC0) and np.all(_f(out[0, 1]) == 1.0)
    out = oracle.dequant(np.full((1, 32, 1), 0x21, np.uint8),
                         np.array([[[0xFF], [127]]], np.uint8), None, MX)
    assert np.all(out[0, 0] == 0x7FC0) and np.all(_f(out[0, 1]) == 1.0)


def test_scales_kmajor_hand_example(oracle):
    # two experts, three columns, two blocks, written out by hand:
    # column n of expert e holds blocks (b0, b1); k-major puts block rows first
    s = np.array([[[1, 2], [3, 4], [5, 6]],
                  [[7, 8], [9, 10], [11, 12]]], np.uint8)
    want = np.array([[[1, 3, 5], [2, 4, 6]],
                     [[7, 9, 11], [8, 10, 12]]], np.uint8)
    assert np.array_equal(oracle.scales_kmajor(s), want)


def test_scales_kmajor_keeps_dequant(oracle):
    # dequantising through the k-major copy (read back at [e, k // bs, n])
    # gives the same bf16 weights as the page layout
    rng = np.random.default_rng(5)
    E, K, N = 2, 64, 64
    packed = rng.integers(0, 256, (E, K, N // 2), dtype=np.uint8)
    scales = syn.block_scales(rng, NV, (E, N, K // 16))
    km = oracle.scales_kmajor(scales)
    back = np.ascontiguousarray(km.transpose(0, 2, 1))
    assert np.array_equal(oracle.dequant(packed, back, None, NV), oracle.dequant(packed, scales, None, NV))
    # and every scale byte appears once at its transposed place
    assert km.shape == (E, K // 16, N)
    assert np.array_equal(np.sort(km.ravel()), np.sort(scales.ravel()))
