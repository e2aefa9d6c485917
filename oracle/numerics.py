"""Element formats used by the oracle: bfloat16 and FP8 E4M3.

Test infrastructure only (see the package docstring).

bfloat16: 1 sign, 8 exponent, 7 mantissa bits; the top half of an IEEE
binary32. Decoding is exact.

E4M3 ("fn" flavour, as used for FP8 attention in the block-sparse prefill
survey page, FlashPrefill V2 FP8 figures): 1 sign bit, 4 exponent bits with
bias 7, 3 mantissa bits; no infinities; the all-ones code ``S.1111.111`` is
NaN, so the largest finite magnitude is ``1.75 * 2**8 = 448``; exponent field
0 holds subnormals ``m * 2**-9``.

The per-head quantiser follows the FP8 variant's reading: one scale per head,
``scale = absmax / 448`` in float32 (``1.0`` for an all-zero head), codes
``e4m3(x / scale)`` with the division in float32, round to nearest even and
saturation to ``±448``.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bfloat16 bit patterns, as float64."""
    w = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return w.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Exact value of E4M3 codes (uint8), as float64 (NaN for 0x7F/0xFF)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to E4M3 codes: nearest, ties to even, saturating.

    For ``|x|`` in ``[2**e, 2**(e+1))`` with ``e >= -6`` the spacing of E4M3
    values is ``2**(e-3)``; below ``2**-6`` (subnormals) it is ``2**-9``.
    Rounding ``|x| / spacing`` to the nearest even integer and scaling back
    gives the nearest representable value (a carry into the next binade is
    itself representable). Magnitudes above 448 saturate to 448.
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    if np.isnan(x).any():
        raise ValueError("NaN input")
    a = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    spacing = np.exp2(e - 3.0)
    r = np.rint(a / spacing) * spacing          # np.rint: ties to even
    r = np.minimum(r, E4M3_MAX)
    # encode the (now exactly representable) magnitude
    out = np.zeros(x.shape, np.uint8)
    sub = r < 2.0 ** -6
    m_sub = np.rint(r / 2.0 ** -9).astype(np.int64)
    with np.errstate(divide="ignore"):
        er = np.floor(np.log2(np.where(r > 0, r, 1.0))).astype(np.int64)
    m_norm = np.rint((r / np.exp2(er.astype(np.float64)) - 1.0) * 8.0).astype(np.int64)
    code = np.where(sub, m_sub, ((er + 7) << 3) | m_norm)
    code = np.where(r == 0, 0, code)
    out[...] = (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)
    return out


def per_head_scale(bits: np.ndarray) -> np.ndarray:
    """float32 ``absmax / 448`` per head of bf16 ``[tokens, H, d]`` (1.0 if all zero)."""
    x = (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    absmax = np.zeros(x.shape[1], np.float32)
    for t0 in range(0, x.shape[0], 8192):
        absmax = np.maximum(absmax, np.abs(x[t0:t0 + 8192]).max(axis=(0, 2)))
    return np.where(absmax > 0, absmax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)


def quantize_with_scale(bits: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """E4M3 codes of bf16 ``[tokens, H, d]`` divided (float32) by the per-head scale."""
    x = (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    y = (x / np.asarray(scale, np.float32)[None, :, None]).astype(np.float32)
    return e4m3_from_f32(y)


def quantize_per_head(bits: np.ndarray):
    """Quantise bf16 ``[tokens, H, d]`` to E4M3 with one scale per head.

    Returns ``(codes uint8 [tokens, H, d], scale float32 [H])``.
    """
    scale = per_head_scale(bits)
    return quantize_with_scale(bits, scale), scale
