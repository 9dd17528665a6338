"""Pins of the oracle's element codecs against things other than the oracle:
the printed E2M1 value table, torch's float8 casts (a library decoder), torch's
float32 -> bf16 cast, closed-form ties, and special cases."""
import math
import os

import numpy as np
import pytest
import torch

from conftest import GOLDEN


def _golden_e2m1():
    vals = {}
    with open(os.path.join(GOLDEN, "e2m1_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                c, v = line.split()
                vals[int(c)] = float(v)
    return vals


def test_e2m1_matches_printed_table(oracle):
    g = _golden_e2m1()
    assert sorted(g) == list(range(16))
    for c, v in g.items():
        got = oracle.e2m1(c)
        assert got == v, (c, got, v)
        assert math.copysign(1.0, got) == math.copysign(1.0, v), c  # code 8 is -0.0


def test_e2m1_sign_is_bit3(oracle):
    for c in range(8):
        assert oracle.e2m1(c | 8) == -oracle.e2m1(c)
        assert math.copysign(1.0, oracle.e2m1(c | 8)) == -1.0


def _torch_f8(dtype):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(dtype).to(torch.float64).numpy()


def test_e4m3fn_exhaustive_vs_torch(oracle):
    ref = _torch_f8(torch.float8_e4m3fn)
    got = np.array([oracle.e4m3fn(b) for b in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_e4m3fn_special_values(oracle):
    assert oracle.e4m3fn(0x00) == 0.0
    assert math.copysign(1.0, oracle.e4m3fn(0x80)) == -1.0
    assert oracle.e4m3fn(0x7E) == 448.0          # largest finite
    assert math.isnan(oracle.e4m3fn(0x7F)) and math.isnan(oracle.e4m3fn(0xFF))
    assert oracle.e4m3fn(0x01) == 2.0 ** -9      # smallest subnormal
    assert oracle.e4m3fn(0x08) == 2.0 ** -6      # smallest normal
    assert oracle.e4m3fn(0x38) == 1.0
    assert oracle.e4m3fn(0x78) == 256.0          # no infinity at exponent 15
    # the generator's scale range [0.25, 4): exponent fields 5..8
    assert oracle.e4m3fn(5 << 3) == 0.25 and oracle.e4m3fn((8 << 3) | 7) == 3.75


def test_e8m0_exhaustive_vs_torch(oracle):
    ref = _torch_f8(torch.float8_e8m0fnu)
    got = np.array([oracle.e8m0(b) for b in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_e8m0_special_values(oracle):
    assert oracle.e8m0(127) == 1.0
    assert oracle.e8m0(120) == 2.0 ** -7 and oracle.e8m0(134) == 2.0 ** 7
    assert oracle.e8m0(0) == 2.0 ** -127
    assert math.isnan(oracle.e8m0(255))


def test_bf16_rne_matches_torch_on_floats(oracle):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    # add ties, near-ties, subnormals, overflow edges
    extra = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 2 ** -130, 3 * 2 ** -134, 2 ** -149,
                      3.3895313892515355e38, 3.4e38, -0.0, 65504.0, 1.00390625],
                     dtype=np.float32)
    vals = np.concatenate([vals, extra])
    vals = vals[~np.isnan(vals)]
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_rne(float(v)) for v in vals], dtype=np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(vals[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_bf16_rne_rounds_doubles_once(oracle):
    # exact ties go to the even neighbour
    assert oracle.bf16_rne(1.0 + 2 ** -8) == 0x3F80
    assert oracle.bf16_rne(1.0 + 3 * 2 ** -8) == 0x3F82
    # a hair above a tie rounds up -- a float32 intermediate would lose the hair
    assert oracle.bf16_rne(1.0 + 2 ** -8 + 2 ** -40) == 0x3F81
    assert oracle.bf16_rne(-(1.0 + 2 ** -8 + 2 ** -40)) == 0xBF81
    # subnormal bf16 (spacing 2^-133)
    assert oracle.bf16_rne(2.0 ** -133) == 0x0001
    assert oracle.bf16_rne(2.0 ** -134) == 0x0000          # tie -> even (zero)
    assert oracle.bf16_rne(1.5 * 2.0 ** -133) == 0x0002    # tie -> even
    assert oracle.bf16_rne(float("inf")) == 0x7F80
    assert oracle.bf16_rne(2.0 ** 128) == 0x7F80
    assert oracle.bf16_rne(float("nan")) == 0x7FC0
    assert oracle.bf16_rne(-0.0) == 0x8000


def test_swiglu_standard_is_silu_times_value(oracle):
    rng = np.random.default_rng(3)
    g = rng.standard_normal(200) * 4
    v = rng.standard_normal(200) * 4
    ref = (torch.nn.functional.silu(torch.from_numpy(g)) * torch.from_numpy(v)).numpy()
    got = np.array([oracle.swiglu(a, b) for a, b in zip(g, v)])
    np.testing.assert_allclose(got, ref, rtol=1e-14, atol=1e-300)


def test_swiglu_clamps(oracle):
    a, b, lim = 1.702, 1.0, 7.0
    rng = np.random.default_rng(4)
    for gate, val in zip(rng.uniform(-6.5, 6.5, 50), rng.uniform(-6.5, 5.5, 50)):
        # gate is clamped from above only, value on both sides
        assert oracle.swiglu(50.0, val, a, b, lim) == oracle.swiglu(7.0, val, a, b, lim)
        assert oracle.swiglu(gate, 50.0, a, b, lim) == oracle.swiglu(gate, 7.0, a, b, lim)
        assert oracle.swiglu(gate, -50.0, a, b, lim) == oracle.swiglu(gate, -7.0, a, b, lim)
        # below the limit the clamp is inactive and beta shifts the value
        assert oracle.swiglu(gate, val, a, b, lim) == pytest.approx(
            oracle.swiglu(gate, val + b, a, 0.0, math.inf), rel=1e-15, abs=1e-300)
    # a very negative gate is not clamped (min only applies above)
    assert oracle.swiglu(-50.0, 1.0, 1.0, 0.0, 7.0) < 0.0
    # alpha -> large makes the gate a hard ReLU
    assert oracle.swiglu(2.0, 3.0, 1e6, 0.0, math.inf) == pytest.approx(6.0)
    assert oracle.swiglu(-2.0, 3.0, 1e6, 0.0, math.inf) == pytest.approx(0.0, abs=1e-300)
