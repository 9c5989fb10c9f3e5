"""MXFP8 quantise / dequantise and the MXFP8 decode reference -- TEST
INFRASTRUCTURE ONLY (only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline may import it).

The page "SGLang and Miles Add Day-0 Support for Inkling", section "Relative
Logits Optimization", paragraph "MXFP8 Support", stores K and V in MXFP8 and
runs Q K^T as an MXFP8 product while P V stays in bf16 with V dequantised on
the fly.  The pages do not spell out the format; MXFP8 is the OCP
Microscaling (MX) format, read here as follows:

  * elements are FP8 E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
    bits; exponent field 0 holds the subnormals m * 2^-9; no infinities; the
    one NaN pattern per sign is S.1111.111; the largest finite value is 448;
  * a block is 32 consecutive elements of the last dimension and shares one
    E8M0 scale: an unsigned byte b meaning 2^(b - 127) (255 is NaN, unused);
  * quantising a block: with amax its largest magnitude, the shared exponent
    is floor(log2(amax)) - 8 (8 = the exponent of the largest power of two
    E4M3 holds), clamped to [-127, 127]; an all-zero block takes -127;
    each element is x / 2^e rounded to the nearest E4M3 value, ties to even,
    magnitudes beyond 448 saturating to 448, the sign kept (a negative value
    that rounds to zero is the code S=1, -0, as in IEEE rounding);
  * dequantising: element value * 2^e, exact.

The MXFP8 decode reference is the fp64 forward of the relative attention on
the dequantised operands: q quantised per 32 head dims of each row (the Q K^T
product runs in MXFP8), K and V dequantised from their MXFP8 storage.

Plain numpy, exact integer / power-of-two arithmetic.
"""
from __future__ import annotations

import numpy as np

BLOCK = 32          # elements per shared scale
E4M3_MAX = 448.0
E4M3_EMAX = 8       # exponent of the largest power of two in E4M3
SCALE_BIAS = 127


def e4m3_decode(bits):
    """Value of E4M3 codes (uint8 array) as float64; NaN for S.1111.111."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    s = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return s * val


def _e4m3_table():
    """The 127 non-negative finite E4M3 values in code order (code = index)."""
    codes = np.arange(0x7F, dtype=np.uint8)   # 0x00 .. 0x7E
    return e4m3_decode(codes)


_POS = _e4m3_table()


def e4m3_encode(x):
    """Nearest E4M3 code of each float64 (ties to the even code, i.e. the
    even mantissa), magnitudes past 448 saturating to 448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    # lower neighbour in the sorted table of non-negative values
    lo = np.clip(np.searchsorted(_POS, a, side="right") - 1, 0, len(_POS) - 1)
    hi = np.minimum(lo + 1, len(_POS) - 1)
    dlo = a - _POS[lo]
    dhi = _POS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi != lo) & ((hi & 1) == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


def block_exponent(amax):
    """Shared exponent of blocks with these largest magnitudes."""
    amax = np.asarray(amax, dtype=np.float64)
    e = np.full(amax.shape, -SCALE_BIAS, dtype=np.int64)
    nz = amax > 0
    # floor(log2(amax)) exactly: frexp gives amax = f * 2^k with f in [0.5, 1)
    _, k = np.frexp(amax[nz])
    e[nz] = k.astype(np.int64) - 1 - E4M3_EMAX
    return np.clip(e, -SCALE_BIAS, SCALE_BIAS)


def quantize(x):
    """MXFP8 of x (last dimension a multiple of 32): (codes uint8 with x's
    shape, scales uint8 with the last dimension divided by 32)."""
    x = np.asarray(x, dtype=np.float64)
    assert x.shape[-1] % BLOCK == 0, "last dimension must be a multiple of 32"
    blk = x.reshape(*x.shape[:-1], x.shape[-1] // BLOCK, BLOCK)
    e = block_exponent(np.abs(blk).max(axis=-1))
    codes = e4m3_encode(blk / np.ldexp(1.0, e)[..., None])
    return codes.reshape(x.shape), (e + SCALE_BIAS).astype(np.uint8)


def dequantize(codes, scales):
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8).astype(np.int64)
    blk = codes.reshape(*codes.shape[:-1], codes.shape[-1] // BLOCK, BLOCK)
    val = e4m3_decode(blk) * np.ldexp(1.0, scales - SCALE_BIAS)[..., None]
    return val.reshape(codes.shape)


def roundtrip(x):
    return dequantize(*quantize(x))


def decode_reference(q, k8, k_scale, v8, v_scale, r, P, cu_seqlens_q, cu_seqlens_k, *,
                     alpha, window=0, log_scale_base=0.0):
    """fp64 MXFP8 decode: the relative-attention forward oracle on q rounded
    through MXFP8 per 32 head dims and on K, V dequantised from their MXFP8
    storage.  Returns (out, lse) like the forward oracle."""
    import oracle

    def _np(t):
        if hasattr(t, "detach"):
            t = t.detach().cpu()
            if str(t.dtype) == "torch.bfloat16":
                t = t.float()
            return t.numpy()
        return np.asarray(t)

    qd = roundtrip(_np(q).astype(np.float64))
    kd = dequantize(_np(k8), _np(k_scale))
    vd = dequantize(_np(v8), _np(v_scale))
    return oracle.forward(qd, kd, vd, _np(r).astype(np.float64), _np(P).astype(np.float64),
                          _np(cu_seqlens_q), _np(cu_seqlens_k), alpha=alpha, window=window,
                          log_scale_base=log_scale_base)
