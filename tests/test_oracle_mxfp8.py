"""Pins of the MXFP8 oracle (oracle/mxfp8.py) against what the FP8 E4M3 and
MX definitions fix on their own: code values from the bit layout (bias 7,
subnormals m * 2^-9, 448 the largest finite, S.1111.111 NaN), round to
nearest with ties to the even mantissa, saturation past 448, the shared
exponent floor(log2 amax) - 8, and exact round trips of representable blocks.
Page: "SGLang and Miles Add Day-0 Support for Inkling", section "Relative
Logits Optimization", paragraph "MXFP8 Support" (K/V stored in MXFP8, Q K^T
in MXFP8, P V in bf16)."""
import math

import numpy as np
import pytest

from oracle import mxfp8 as M


def test_code_values_from_the_bit_layout():
    # value = (1 + m/8) 2^(e-7) for e > 0, m 2^-9 for e == 0
    known = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x78: 256.0, 0x79: 288.0, 0x7E: 448.0,
             0xB8: -1.0, 0xFE: -448.0}
    for code, val in known.items():
        assert M.e4m3_decode(np.uint8(code)) == val, hex(code)
    assert math.isnan(M.e4m3_decode(np.uint8(0x7F)))
    assert math.isnan(M.e4m3_decode(np.uint8(0xFF)))


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(M.e4m3_encode(M.e4m3_decode(codes)), codes)


def test_ties_go_to_the_even_mantissa():
    # spacing 32 in [256, 512): 272 lies between 256 (m=0) and 288 (m=1)
    assert M.e4m3_encode(272.0) == 0x78
    assert M.e4m3_encode(304.0) == 0x7A          # between 288 (m=1) and 320 (m=2)
    assert M.e4m3_encode(2.0 ** -10) == 0x00     # between 0 and the smallest subnormal
    assert M.e4m3_encode(3 * 2.0 ** -10) == 0x02  # between m=1 and m=2 subnormals
    assert M.e4m3_encode(-272.0) == 0xF8
    assert M.e4m3_encode(-2.0 ** -11) == 0x80        # rounds to zero, keeps its sign
    # just off a tie goes to the nearer neighbour
    assert M.e4m3_encode(272.0001) == 0x79
    assert M.e4m3_encode(271.9999) == 0x78


def test_saturation_past_448():
    for x in (448.0, 449.0, 463.99, 464.0, 1000.0, 1e30):
        assert M.e4m3_encode(x) == 0x7E
    assert M.e4m3_encode(-500.0) == 0xFE


def test_shared_exponent():
    amax = np.array([1.0, 1.9, 2.0, 0.75, 448.0, 0.0, 2.0 ** -140, 3e38])
    assert list(M.block_exponent(amax)) == [-8, -8, -7, -9, 0, -127, -127, 119]


def test_single_block_quantise():
    x = np.zeros(32)
    x[0] = 1.0
    x[5] = -0.5
    codes, scales = M.quantize(x)
    assert scales[0] == 119                      # 2^-8
    assert codes[0] == 0x78 and codes[5] == 0xF0  # 256 and -128 in units of 2^-8
    assert np.all(codes[[i for i in range(32) if i not in (0, 5)]] == 0)
    assert np.array_equal(M.dequantize(codes, scales), x)
    # amax 1.9 -> 486.4 units of 2^-8 -> saturates to 448 -> 1.75
    y = np.full(32, 0.25)
    y[3] = 1.9
    cy, sy = M.quantize(y)
    assert sy[0] == 119 and cy[3] == 0x7E
    assert M.dequantize(cy, sy)[3] == 1.75


def test_zero_block():
    codes, scales = M.quantize(np.zeros((2, 64)))
    assert np.all(codes == 0) and np.all(scales == 0)
    assert np.all(M.dequantize(codes, scales) == 0)


def test_representable_blocks_round_trip_exactly():
    rng = np.random.default_rng(3)
    for _ in range(200):
        e = int(rng.integers(-60, 60))
        codes = rng.integers(0, 0x7F, 32).astype(np.uint8)          # finite, non-negative
        codes[rng.integers(0, 32)] = rng.integers(0x78, 0x7F)        # amax in [256, 448] units
        codes = np.where(rng.random(32) < 0.5, codes | 0x80, codes).astype(np.uint8)
        x = M.e4m3_decode(codes) * 2.0 ** e
        c2, s2 = M.quantize(x)
        assert s2[0] == e + 127
        assert np.array_equal(c2, codes)
        assert np.array_equal(M.dequantize(c2, s2), x)


def test_scales_follow_blocks_of_the_last_dimension():
    x = np.concatenate([np.full(32, 3.0), np.full(32, 0.001)])[None, :].repeat(2, 0)
    x[1] *= 1024.0
    codes, scales = M.quantize(x)
    assert scales.shape == (2, 2)
    assert list(scales[0]) == [127 + 1 - 8, 127 + math.floor(math.log2(0.001)) - 8]
    assert list(scales[1]) == [127 + 11 - 8, 127 + math.floor(math.log2(1.024)) - 8]
    d = M.dequantize(codes, scales)
    assert np.allclose(d, x, rtol=2 ** -4)


def test_rounding_error_bound():
    # normal results: |x - q(x)| <= half a 3-bit-mantissa ulp of x / 2^e,
    # unless saturated; subnormal results: <= 2^-10 units of 2^e
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 128)) * np.exp(rng.uniform(-8, 8, (64, 1)))
    codes, scales = M.quantize(x)
    d = M.dequantize(codes, scales)
    unit = np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)
    a = np.abs(x) / unit
    sat = a > 448
    ulp = np.where(a >= 2.0 ** -6, np.ldexp(1.0, np.floor(np.log2(np.maximum(a, 2.0 ** -6))).astype(int) - 3),
                   2.0 ** -9)
    err = np.abs(x - d) / unit
    assert np.all(err[~sat] <= ulp[~sat] / 2)
    assert np.all(np.abs(d[sat]) == 448 * unit[sat])


def test_decode_reference_on_representable_inputs_is_the_forward():
    import oracle
    rng = np.random.default_rng(7)
    Tq, Tk, Hq, Hkv, rd, E = 3, 40, 4, 2, 4, 16
    def repr_tensor(shape):
        codes = rng.integers(0, 0x7F, shape).astype(np.uint8)
        codes = np.where(rng.random(shape) < 0.5, codes | 0x80, codes).astype(np.uint8)
        codes[..., ::32] = 0x7A                                  # a 320-unit element per block
        e = rng.integers(-12, -6, shape[:-1] + (shape[-1] // 32,))
        return codes, (e + 127).astype(np.uint8), M.dequantize(codes, (e + 127).astype(np.uint8))
    qc, qs, qv = repr_tensor((Tq, Hq, 128))
    kc, ks, kv = repr_tensor((Tk, Hkv, 128))
    vc, vs, vv = repr_tensor((Tk, Hkv, 128))
    r = rng.standard_normal((Tq, Hq, rd))
    P = rng.standard_normal((rd, E)) * 0.02
    cq = np.array([0, Tq], dtype=np.int32)
    ck = np.array([0, Tk], dtype=np.int32)
    o1, l1 = M.decode_reference(qv, kc, ks, vc, vs, r, P, cq, ck, alpha=0.088)
    o2, l2 = oracle.forward(qv, kv, vv, r, P, cq, ck, alpha=0.088)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # and a q that is not representable is rounded first
    qn = qv * (1 + 1e-3)
    o3, _ = M.decode_reference(qn, kc, ks, vc, vs, r, P, cq, ck, alpha=0.088)
    o4, _ = oracle.forward(M.roundtrip(qn), kv, vv, r, P, cq, ck, alpha=0.088)
    assert np.array_equal(o3, o4)
