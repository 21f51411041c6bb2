"""OCP FP8 E4M3 decode and per-tensor quantiser -- oracle (test infrastructure only).

The per-tensor FP8 linears are those of "Distributed Layerwise Offload",
Feature compatibility table, row "Per-tensor online FP8 linears": one weight
tensor and one scale per linear, finalised before streaming.  The pages do
not fix the scale rule or the rounding; the reading used here is the common
per-tensor one:
  s = amax(|W|) / 448   (float32; s = 1 when amax = 0)
  q = e4m3(W / s)       (W / s in float32, then round-to-nearest-even to
                         E4M3 with saturation to +-448)
Activations of the W8A8 linears (an extension the pages do not describe)
are quantised per tensor with the same scale rule and the inverted-scale
form of dynamic FP8 activation quantisers:
  s = amax(|x|) / 448   (float32; 1 when amax = 0),  r = 1 / s  (float32)
  q = e4m3(x * r)       (x * r in float32, then as above)
E4M3 per the OCP 8-bit floating point specification: 1 sign bit, 4 exponent
bits with bias 7, 3 mantissa bits, subnormals, no infinities, S.1111.111 is
NaN, largest finite magnitude 448.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """float64 value of each E4M3 byte."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7 == 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = np.ldexp(m / 8.0, -6)
    nrm = np.ldexp(1.0 + m / 8.0, e - 7)
    val = np.where(e == 0, sub, nrm) * sign
    nan = (e == 15) & (m == 7)
    return np.where(nan, np.nan, val)


def _encode_magnitude(a: np.ndarray) -> np.ndarray:
    """E4M3 code (without sign) of non-negative float64 magnitudes a < 448 + ..."""
    a = np.asarray(a, dtype=np.float64)
    code = np.zeros(a.shape, dtype=np.int64)
    sat = a >= E4M3_MAX
    code[sat] = 0x7E
    # subnormal range: quantum 2^-9
    sub = (~sat) & (a < 2.0 ** -6)
    r = np.rint(a[sub] / 2.0 ** -9).astype(np.int64)          # 0..8, ties to even
    code[sub] = np.where(r == 8, 1 << 3, r)
    # normal range: exponent e = floor(log2 a), quantum 2^(e-3)
    nrm = (~sat) & (~sub)
    an = a[nrm]
    _, ex = np.frexp(an)                                        # an = f * 2^ex, f in [0.5, 1)
    e = ex - 1
    r = np.rint(an / np.ldexp(1.0, e - 3)).astype(np.int64)   # 8..16, ties to even
    carry = r == 16
    e = np.where(carry, e + 1, e)
    r = np.where(carry, 8, r)
    c = ((e + 7) << 3) | (r - 8)
    c = np.where(c > 0x7E, 0x7E, c)                             # saturate past 448
    code[nrm] = c
    return code


def encode_e4m3(v: np.ndarray) -> np.ndarray:
    """Round float values to E4M3 (nearest, ties to even, saturating)."""
    v = np.asarray(v, dtype=np.float64)
    mag = _encode_magnitude(np.abs(v))
    sign = np.signbit(v).astype(np.int64) << 7
    return (mag | sign).astype(np.uint8)


def quantize_per_tensor(w: np.ndarray):
    """(codes uint8, scale float32) of one weight tensor."""
    w32 = np.asarray(w, dtype=np.float32)
    amax = np.float32(np.max(np.abs(w32))) if w32.size else np.float32(0.0)
    s = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(E4M3_MAX))
    v = (w32 / s).astype(np.float32)
    return encode_e4m3(v), s


def quantize_activation(x: np.ndarray):
    """(codes uint8, scale float32) of one activation tensor (W8A8 inputs):
    the weight quantiser's scale, codes of x times the float32 reciprocal."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0.0)
    s = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(E4M3_MAX))
    r = np.float32(np.float32(1.0) / s)
    v = (x32 * r).astype(np.float32)
    return encode_e4m3(v), s


def dequantize(codes: np.ndarray, s) -> np.ndarray:
    """float64 weight s * decode(codes) (exact in float64)."""
    return decode_e4m3(codes) * np.float64(s)
