"""Pins for oracle.fp8 (OCP E4M3 decode, RNE saturating encode, per-tensor scale)."""
import math

import numpy as np
import pytest
import torch

from oracle import fp8

# Closed-form values from the OCP E4M3 definition (bias 7, 3 mantissa bits).
KNOWN = {
    0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
    0x30: 0.5, 0x38: 1.0, 0x3C: 1.5, 0x3F: 1.875, 0x40: 2.0, 0x48: 4.0,
    0x77: 240.0, 0x78: 256.0, 0x7E: 448.0,
    0xB8: -1.0, 0xFE: -448.0, 0x81: -(2.0 ** -9),
}


def test_decode_closed_form():
    vals = fp8.decode_e4m3(np.arange(256, dtype=np.uint8))
    for c, v in KNOWN.items():
        assert vals[c] == v, hex(c)
    assert math.isnan(vals[0x7F]) and math.isnan(vals[0xFF])
    assert np.signbit(vals[0x80]) and vals[0x80] == 0.0
    finite = ~np.isnan(vals)
    assert finite.sum() == 254
    assert np.nanmax(np.abs(vals)) == 448.0
    # monotone over the positive codes
    pos = vals[0:0x7F]
    assert np.all(np.diff(pos) > 0)


def test_decode_matches_torch_for_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = fp8.decode_e4m3(np.arange(256, dtype=np.uint8))
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    m = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[m], ref[m])


def test_encode_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    np.testing.assert_array_equal(fp8.encode_e4m3(fp8.decode_e4m3(codes)), codes)


def test_encode_matches_torch_rne():
    g = np.random.default_rng(0)
    v = np.concatenate([
        g.standard_normal(200000) * 50.0,
        g.standard_normal(50000) * 1e-2,          # subnormal and small normals
        g.uniform(-447.0, 447.0, 50000),
    ]).astype(np.float32)
    # exact midpoints between neighbouring codes exercise ties-to-even
    pos = fp8.decode_e4m3(np.arange(0, 0x7F, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(fp8.encode_e4m3(v), ref)


def test_encode_saturates():
    v = np.array([448.0, 449.0, 463.9, 464.0, 1e4, 1e30, -500.0, -1e30])
    out = fp8.encode_e4m3(v)
    np.testing.assert_array_equal(out, [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE])


def test_quantize_per_tensor():
    g = np.random.default_rng(1)
    w = (g.standard_normal((64, 96)) * 0.02).astype(np.float32)
    q, s = fp8.quantize_per_tensor(w)
    assert s.dtype == np.float32
    assert s == np.float32(np.max(np.abs(w)) / np.float32(448.0))
    i = np.unravel_index(np.argmax(np.abs(w)), w.shape)
    assert q[i] in (0x7E, 0xFE)
    # error bound: half a quantum of the code's binade (relative 2^-4 for normals)
    deq = fp8.dequantize(q, s)
    v = np.abs(w.astype(np.float64) / s)
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -6)))
    bound = 0.5 * 2.0 ** (e - 3) * s * (1 + 1e-6)
    assert np.all(np.abs(deq - w) <= bound)
    z, sz = fp8.quantize_per_tensor(np.zeros((4, 4), np.float32))
    assert sz == 1.0 and not z.any()


def test_quantize_activation_inverted_scale():
    g = np.random.default_rng(4)
    x = (g.standard_normal((2, 50, 96)) * np.exp(g.uniform(-6, 3, (2, 50, 96)))).astype(np.float32)
    q, s = fp8.quantize_activation(x)
    # same scale rule as the weights
    assert s == fp8.quantize_per_tensor(x)[1]
    # codes of x * (1/s), both rounded to fp32, against torch's E4M3 cast
    r = np.float32(1.0) / s
    v = torch.from_numpy(x) * torch.tensor(r, dtype=torch.float32)
    ref = v.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(q, ref)
    # with a power-of-two scale the product is the quotient: the weights' codes
    y = x / np.float32(np.max(np.abs(x))) * np.float32(448.0 * 2.0 ** -5)
    y = y.astype(np.float32)
    qa, sa = fp8.quantize_activation(y)
    qw, sw = fp8.quantize_per_tensor(y)
    assert sa == sw == np.float32(2.0 ** -5)
    np.testing.assert_array_equal(qa, qw)
    # half a quantum of error, plus the reciprocal's rounding
    deq = fp8.dequantize(q, s)
    a = np.abs(x.astype(np.float64) / s)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    bound = (0.5 * 2.0 ** (e - 3) + a * 2.0 ** -21) * s
    assert np.all(np.abs(deq - x) <= bound)
