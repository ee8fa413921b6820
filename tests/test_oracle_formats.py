"""CPU pins of the oracle's number formats (E4M3, E8M0, bf16).

Each check compares the oracle with something other than itself: values read
by hand off the format definitions (tests/golden), a brute-force nearest
search over all 256 codes, and integer bit-field arithmetic.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import formats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_sections(name):
    sec, out = None, {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                sec = line.strip("[]")
                out[sec] = []
                continue
            out.setdefault(sec, []).append(line.split())
    return out


def _val(s):
    return float(s)


def test_e4m3_decode_golden():
    rows = _read_sections("e4m3_codes.txt")["decode"]
    for code, val in rows:
        got = oracle.e4m3_decode(np.uint8(int(code, 16)))
        want = _val(val)
        if math.isnan(want):
            assert math.isnan(got), code
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, got, want)


def test_e4m3_encode_golden():
    rows = _read_sections("e4m3_codes.txt")["encode"]
    for val, code in rows:
        got = int(oracle.e4m3_encode(np.float64(_val(val))))
        assert got == int(code, 16), (val, hex(got), code)


def test_e4m3_table_structure():
    mags = oracle.e4m3_magnitudes()
    assert mags.shape == (127,)
    assert np.all(np.diff(mags) > 0)            # strictly increasing in the code
    assert mags[0] == 0 and mags[-1] == 448
    # negative codes mirror the positive ones
    dec = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.array_equal(dec[0x80:0xFF], -dec[:0x7F])
    assert np.isnan(dec[0x7F]) and np.isnan(dec[0xFF])
    assert np.sum(~np.isnan(dec)) == 254


def _brute_force_e4m3(v):
    """Nearest of all 256 codes by exhaustive distance; ties -> even code."""
    dec = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    out = np.empty(v.shape, dtype=np.uint8)
    for i, x in enumerate(v.ravel()):
        if math.isnan(x):
            out.ravel()[i] = 0x7F
            continue
        a = min(abs(x), 448.0)                   # saturation to the largest finite
        best, bestd = None, None
        for c in range(0x7F):                    # non-negative finite codes
            d = abs(a - dec[c])
            if bestd is None or d < bestd or (d == bestd and c % 2 == 0):
                best, bestd = c, d
        if math.copysign(1.0, x) < 0:
            best |= 0x80
        out.ravel()[i] = best
    return out


def test_e4m3_encode_vs_brute_force():
    rng = np.random.default_rng(1)
    mags = oracle.e4m3_magnitudes()
    mids = (mags[:-1] + mags[1:]) / 2
    pts = [mags, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
           np.nextafter(mags, 0), np.nextafter(mags, 1e9)]
    pts.append(np.array([0.0, 447.9, 448.0, 463.9, 464.0, 465.0, 1e30, np.inf, 2.0 ** -12]))
    # random fp32 bit patterns over the whole E4M3 range and a bit beyond
    bits = rng.integers(0, 2 ** 32, size=4000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32).astype(np.float64)
    f = f[np.isfinite(f)]
    logu = rng.uniform(-14, 10, size=3000)
    pts.append(np.exp2(logu))
    pts.append(f[np.abs(f) < 1e4])
    v = np.concatenate(pts)
    v = np.concatenate([v, -v, [np.nan]])
    assert np.array_equal(oracle.e4m3_encode(v), _brute_force_e4m3(v))


def test_e8m0_golden():
    with open(os.path.join(GOLDEN, "e8m0_scales.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, code = line.split()
            got = int(oracle.e8m0_from_amax(np.float32(float(a))))
            assert got == int(code, 16), (a, hex(got), code)


def test_e8m0_vs_bit_fields():
    """Normal fp32 amax: code = clamp(exponent field - 8, 0, 254) (bits, not frexp)."""
    rng = np.random.default_rng(2)
    bits = rng.integers(0x00800000, 0x7F800000, size=200000, dtype=np.int64).astype(np.uint32)
    a = bits.view(np.float32)
    field = (bits >> 23).astype(np.int64)
    want = np.clip(field - 127 - 8, -127, 127) + 127
    assert np.array_equal(oracle.e8m0_from_amax(a).astype(np.int64), want)
    # every exponent value once, at the bottom and at the top of the binade
    for fe in range(1, 255):
        for m in (0, 0x7FFFFF):
            b = np.array([(fe << 23) | m], dtype=np.uint32)
            assert int(oracle.e8m0_from_amax(b.view(np.float32))[0]) == min(max(fe - 135, -127), 127) + 127


def test_e8m0_block_max_lands_in_top_binade():
    """With e = floor(log2 A) - 8, A * 2**-e lies in [256, 512): the block max
    maps to 256..448 after saturation (the MX rule, not a ceil rule)."""
    rng = np.random.default_rng(3)
    A = np.exp2(rng.uniform(-100, 100, 10000)).astype(np.float32)
    e = oracle.e8m0_from_amax(A).astype(np.int64) - 127
    s = A.astype(np.float64) * np.exp2(-e.astype(np.float64))
    assert np.all((s >= 256) & (s < 512))


def test_bf16_rounding_vs_bit_truncation():
    """round_to_bf16 (one rounding from fp64) against an integer RNE on fp32
    bits, for values that are exactly fp32 (so the two must agree)."""
    rng = np.random.default_rng(4)
    f = (rng.standard_normal(100000) * np.exp2(rng.uniform(-30, 30, 100000))).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    want = r.astype(np.uint32).view(np.float32).astype(np.float64)
    got = oracle.round_to_bf16(f.astype(np.float64))
    assert np.array_equal(got, want)
    # a value that is not an fp32: one rounding from fp64 differs from two
    v = 1.0 + 2.0 ** -8 + 2.0 ** -30          # just above a bf16 midpoint
    assert oracle.round_to_bf16(np.float64(v)) == 1.0 + 2.0 ** -7
    # ties to even
    assert oracle.round_to_bf16(np.float64(1.0 + 2.0 ** -8)) == 1.0
    assert oracle.round_to_bf16(np.float64(1.0 + 3 * 2.0 ** -8)) == 1.0 + 2.0 ** -6
    assert np.isinf(oracle.round_to_bf16(np.float64(3.4e38)))


def test_bf16_bits_roundtrip():
    x = np.array([1.0, -2.5, 2.0 ** -133, 0.0, -0.0, 448.0])
    b = oracle.bf16_bits(x)
    # 2**-133 is the smallest bf16 subnormal (mantissa field 1)
    assert [int(t) for t in b] == [0x3F80, 0xC020, 0x0001, 0x0000, 0x8000, 0x43E0]


@pytest.mark.parametrize("mode", ["fp8_delayed", "fp8_current"])
def test_fp8_stage_small_by_hand(mode):
    y = np.array([[1.0, -2.0, 0.5, 4.0]], dtype=np.float32)
    if mode == "fp8_delayed":
        r = oracle.quantize(y, mode, scale=112.0)
        # 112, -224, 56, 448 are all E4M3 values
        assert list(r["data"][0]) == [0x6E, 0xF6, 0x66, 0x7E]
        assert r["amax"] == 4.0
        assert r["scale_inv"] == np.float32(1.0) / np.float32(112.0)
    else:
        r = oracle.quantize(y, mode)
        assert r["amax"] == 4.0 and r["scale"] == 112.0
        assert list(r["data"][0]) == [0x6E, 0xF6, 0x66, 0x7E]


def test_fp8_current_zero_tensor():
    r = oracle.quantize(np.zeros((2, 32), np.float32), "fp8_current")
    assert r["amax"] == 0 and r["scale"] == 1.0 and np.all(r["data"] == 0)


# ------------------------------------------------------------- FP4 E2M1
def test_e2m1_decode_golden():
    for code, val in _read_sections("e2m1_codes.txt")["decode"]:
        got = float(oracle.e2m1_decode(int(code, 16)))
        want = _val(val)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, got, want)


def test_e2m1_encode_golden():
    for val, code in _read_sections("e2m1_codes.txt")["encode"]:
        got = int(oracle.e2m1_encode(np.float64(_val(val))))
        assert got == int(code, 16), (val, hex(got), code)


def _brute_force_e2m1(x):
    """Nearest of the 8 magnitudes by exhaustive distance (ties -> the code
    with mantissa bit 0), saturating at 6, sign from the sign bit."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    a = min(abs(x), 6.0)
    best = min(range(8), key=lambda c: (abs(a - mags[c]), c % 2))
    return best | (0x8 if math.copysign(1.0, x) < 0 else 0)


def test_e2m1_encode_vs_brute_force():
    rng = np.random.default_rng(3)
    mags = oracle.e2m1_magnitudes()
    mids = (mags[:-1] + mags[1:]) / 2
    pts = [mags, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9), np.nextafter(mags, 1e9),
           rng.uniform(0, 8, 3000), np.exp2(rng.uniform(-10, 5, 1000)), np.array([1e30, np.inf])]
    v = np.concatenate(pts)
    v = np.concatenate([v, -v])
    want = np.array([_brute_force_e2m1(float(t)) for t in v], dtype=np.uint8)
    assert np.array_equal(oracle.e2m1_encode(v), want)


def test_e2m1_roundtrip_and_packing():
    codes = np.arange(16, dtype=np.uint8)
    dec = oracle.e2m1_decode(codes)
    assert np.array_equal(oracle.e2m1_encode(dec), codes)    # -0 keeps 0x8
    # element 2j in the low nibble: codes (1, 2) -> 0x21
    assert oracle.e2m1_pack(np.array([1, 2], np.uint8))[0] == 0x21
    rng = np.random.default_rng(4)
    c = rng.integers(0, 16, (5, 64)).astype(np.uint8)
    p = oracle.e2m1_pack(c)
    assert p.shape == (5, 32)
    assert np.array_equal(oracle.e2m1_unpack(p), c)
    # byte j of a row is 16 * code[2j+1] + code[2j], by integer arithmetic
    assert np.array_equal(p.astype(int), 16 * c[:, 1::2].astype(int) + c[:, 0::2].astype(int))
