"""Number formats, written from their public definitions (oracle side).

* FP8 E4M3 — OCP 8-bit Floating Point Specification (OFP8), format "E4M3":
  1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
  encodes subnormals m * 2**-9; S.1111.111 is NaN; there are no infinities;
  the largest finite magnitude is S.1111.110 = 448.
* E8M0 — OCP Microscaling Formats (MX) v1.0, the shared-scale format: an
  unsigned biased exponent (bias 127) encoding 2**(code-127) for codes 0..254
  and NaN for 0xFF.
* bf16 — 1 sign, 8 exponent, 7 mantissa bits (the top half of an fp32).
* FP4 E2M1 — OCP Microscaling Formats (MX) v1.0, element format "FP4 E2M1":
  1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit; exponent field 0
  encodes the subnormal m * 0.5; no NaN or infinity; magnitudes 0, 0.5, 1,
  1.5, 2, 3, 4, 6 for the codes 0..7, bit 3 the sign.

Conversion rules the kernels must reproduce (the page on TransformerEngine's
normalization extension names the formats only; these are the plainest
readings):
* to E4M3: round to nearest, ties to the even code; magnitudes at or above
  448 saturate to 448 ("satfinite"); NaN becomes 0x7F; the sign bit follows
  the sign of the input, so -0 and negative values that round to zero give
  0x80.
* MX shared exponent of a block: e = floor(log2(amax)) - 8, where 8 is the
  exponent of E4M3's largest normal (448 = 1.75 * 2**8); e is clamped to
  [-127, 127] and stored as e + 127.  amax = 0 gives code 0; amax = NaN gives
  0xFF.  amax = +inf is read as the value its fp32 exponent field encodes,
  2**128, giving e = 120 (code 247).
* to E2M1: round to nearest, ties to the even code (the one whose mantissa
  bit is 0); magnitudes above 6 saturate to 6; the sign bit follows the
  input's sign, so negative values that round to zero give 0x8.  Two codes
  share a byte, the element with the lower index in the low nibble.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_NAN = 0x7F


def _e4m3_value(code: int) -> float:
    """Value of one E4M3 code, from the bit fields (NaN for S.1111.111)."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * m * 2.0 ** -9          # subnormal: (m/8) * 2**(1-7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_DECODE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_decode(codes) -> np.ndarray:
    """uint8 E4M3 codes -> fp64 values (exact)."""
    return _DECODE[np.asarray(codes, dtype=np.uint8)]


def e4m3_magnitudes() -> np.ndarray:
    """The 127 finite non-negative E4M3 magnitudes, codes 0x00..0x7E in order."""
    return _DECODE[:0x7F].copy()


_MAGS = e4m3_magnitudes()


def e4m3_encode(v) -> np.ndarray:
    """Round values (taken exactly, as fp64) to E4M3 codes.

    Nearest representable magnitude, ties to the even code, saturating at 448;
    NaN -> 0x7F; sign from the input's sign bit.  The finite magnitudes are
    increasing in the code, so the two neighbours of |v| are found by a sorted
    search and the nearer one is taken.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    nan = np.isnan(v)
    a_clean = np.where(nan, 0.0, a)
    idx = np.searchsorted(_MAGS, a_clean, side="left")
    idx = np.clip(idx, 1, 0x7E)
    lo = _MAGS[idx - 1]
    hi = _MAGS[idx]
    dlo = a_clean - lo
    dhi = hi - a_clean
    take_hi = dhi < dlo
    tie = dhi == dlo
    # on a tie the even code wins; codes idx-1 and idx differ in parity
    take_hi = np.where(tie, (idx % 2) == 0, take_hi)
    code = np.where(take_hi, idx, idx - 1)
    code = np.where(a_clean >= E4M3_MAX, 0x7E, code)
    code = code.astype(np.uint8)
    code = np.where(np.signbit(v), code | 0x80, code).astype(np.uint8)
    code = np.where(nan, E4M3_NAN, code).astype(np.uint8)
    return code


def e8m0_from_amax(amax) -> np.ndarray:
    """MX shared-scale code (uint8) of blocks with absolute maxima ``amax``.

    e = floor(log2 amax) - 8, clamped to [-127, 127], code = e + 127.
    floor(log2 amax) is read exactly from frexp (amax = f * 2**k with
    0.5 <= f < 1 gives floor(log2 amax) = k - 1, subnormals included).
    """
    a = np.asarray(amax, dtype=np.float32).astype(np.float64)
    nan = np.isnan(a)
    inf = np.isinf(a)
    zero = a == 0
    safe = np.where(nan | inf | zero, 1.0, a)
    _, k = np.frexp(safe)
    e = np.clip(k.astype(np.int64) - 1 - 8, -127, 127)
    code = e + 127
    code = np.where(zero, 0, code)
    code = np.where(inf, 128 - 8 + 127, code)
    code = np.where(nan, 0xFF, code)
    return code.astype(np.uint8)


def e8m0_exponent(code) -> np.ndarray:
    """Unbiased exponent e of an E8M0 code (code - 127); NaN code -> 128."""
    return np.asarray(code, dtype=np.int64) - 127


def round_to_bf16(v) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value, ties to even (one rounding).

    The spacing of bf16 values in [2**k, 2**(k+1)) is 2**(k-7); below the
    smallest normal 2**-126 it is 2**-133.  Values beyond the largest finite
    bf16 (2 - 2**-7) * 2**127, once rounded, become +-inf.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.array(v, copy=True)
    fin = np.isfinite(v) & (v != 0)
    if fin.any():
        a = np.abs(v[fin])
        _, k = np.frexp(a)                 # a in [2**(k-1), 2**k)
        expo = np.maximum(k - 1, -126)
        q = np.ldexp(1.0, (expo - 7).astype(np.int32))
        r = np.round(a / q) * q            # np.round: half to even, exact here
        big = (2.0 - 2.0 ** -7) * 2.0 ** 127
        r = np.where(r > big, np.inf, r)
        out[fin] = np.copysign(r, v[fin])
    return out


def bf16_bits(v) -> np.ndarray:
    """uint16 bit patterns of round_to_bf16(v)."""
    r = round_to_bf16(v).astype(np.float32)   # exact: r is a bf16 value
    bits = (r.view(np.uint32) >> 16).astype(np.uint16)
    bits = np.where(np.isnan(r), np.uint16(0x7FC0), bits)
    return bits.astype(np.uint16)


# ------------------------------------------------------------- FP4 E2M1
E2M1_MAX = 6.0


def _e2m1_value(code: int) -> float:
    """Value of one 4-bit E2M1 code, from the bit fields."""
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * m * 0.5                 # subnormal: (m/2) * 2**(1-1)
    return s * (1.0 + m / 2.0) * 2.0 ** (e - 1)


_E2M1_DECODE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)


def e2m1_decode(codes) -> np.ndarray:
    """4-bit E2M1 codes (0..15, any integer dtype) -> fp64 values (exact)."""
    return _E2M1_DECODE[np.asarray(codes, dtype=np.int64) & 0xF]


def e2m1_magnitudes() -> np.ndarray:
    """The 8 non-negative E2M1 magnitudes, codes 0..7 in order."""
    return _E2M1_DECODE[:8].copy()


_E2M1_MAGS = e2m1_magnitudes()


def e2m1_encode(v) -> np.ndarray:
    """Round values (taken exactly, as fp64) to 4-bit E2M1 codes (uint8 0..15).

    Nearest magnitude, ties to the even code, saturating at 6; sign from the
    input's sign bit.  The magnitudes increase with the code, so the two
    neighbours of |v| come from a sorted search.  NaN has no E2M1 code: the
    caller must not pass one.
    """
    v = np.asarray(v, dtype=np.float64)
    if np.isnan(v).any():
        raise ValueError("E2M1 has no NaN")
    a = np.abs(v)
    idx = np.clip(np.searchsorted(_E2M1_MAGS, a, side="left"), 1, 7)
    lo = _E2M1_MAGS[idx - 1]
    hi = _E2M1_MAGS[idx]
    dlo = a - lo
    dhi = hi - a
    take_hi = np.where(dhi == dlo, (idx % 2) == 0, dhi < dlo)
    code = np.where(take_hi, idx, idx - 1)
    code = np.where(a >= E2M1_MAX, 7, code)
    code = np.where(np.signbit(v), code | 0x8, code)
    return code.astype(np.uint8)


def e2m1_pack(codes) -> np.ndarray:
    """[..., 2k] 4-bit codes -> [..., k] bytes: element 2j low, 2j+1 high."""
    c = np.asarray(codes, dtype=np.uint8)
    assert c.shape[-1] % 2 == 0
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def e2m1_unpack(packed) -> np.ndarray:
    """Inverse of e2m1_pack: [..., k] bytes -> [..., 2k] 4-bit codes."""
    b = np.asarray(packed, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0xF
    out[..., 1::2] = b >> 4
    return out
