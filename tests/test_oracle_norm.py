"""CPU pins of the oracle's normalization arithmetic.

Pins (none of them re-runs the oracle's own formula):
* closed forms worked by hand (tests/golden/norm_closed_forms.txt);
* exact rational statistics (fractions + 50-digit decimal square roots);
* invariants: mean(xhat) = 0, mean(xhat**2) = var/(var+eps), LayerNorm equal
  to RMSNorm on rows with zero mean, scale invariance;
* central finite differences of L = sum(dz * y) for dx, dgamma, dbeta,
  plus sum_j dx_ij = 0 (LayerNorm) and sum_j dx_ij x_ij = 0 (RMSNorm, eps=0);
* pure-Python loop re-derivations of the MXFP8 blocks (rowwise and the
  transposed columnwise layout) on tiny inputs, with a brute-force E4M3;
* NVFP4: a 4 x 16 tensor worked by hand (tests/golden/nvfp4_blocks.txt),
  properties the scale construction forces (the block holding the tensor
  amax gets the largest E4M3 scale, the largest element of a block with a
  normal scale the largest E2M1 code, the dequantization error bound, exact
  invariance under power-of-two scaling of the input, correct rounding of
  the tensor scale) and a loop re-derivation with brute-force E2M1.
"""
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest

import oracle
import rn_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _floats(s):
    return [float(t) for t in s.split()]


def _closed_forms():
    out = []
    with open(os.path.join(GOLDEN, "norm_closed_forms.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            out.append([t.strip() for t in line.split("|")])
    return out


@pytest.mark.parametrize("row", _closed_forms(), ids=lambda r: r[0] + "-" + r[3].replace(" ", "_"))
def test_closed_forms(row):
    op, zc, eps, x, g, b, mu, rs, y = row
    x = np.array([_floats(x)])
    g = np.array(_floats(g), np.float32)
    zc = bool(int(zc))
    eps = float(eps)
    if op == "ln":
        r = oracle.layernorm_fwd(x, g, np.array(_floats(b), np.float32), eps, zc, "none", "f32")
        assert r["mu"][0] == np.float32(float(mu))
    else:
        r = oracle.rmsnorm_fwd(x, g, eps, zc, "none", "f32")
        assert "mu" not in r
    assert r["rsigma"][0] == np.float32(float(rs))
    np.testing.assert_allclose(r["y"][0], _floats(y), rtol=1e-15, atol=1e-15)


def test_stats_exact_rational():
    """mu and rsigma against exact rational mean/variance and a 50-digit sqrt."""
    getcontext().prec = 50
    rng = np.random.default_rng(5)
    for H in (1, 2, 7, 64, 333):
        x = rn_inputs.bf16_bits_to_f32(rn_inputs.to_bf16_bits(rng.normal(0.5, 2.0, (3, H)))).astype(np.float64)
        eps = 1e-5
        m, r = oracle.layernorm_stats(x, eps)
        rr = oracle.rmsnorm_stats(x, eps)
        e = Fraction(float(np.float32(eps)))
        for i in range(3):
            xs = [Fraction(float(v)) for v in x[i]]
            mean = sum(xs) / H
            var = sum((v - mean) ** 2 for v in xs) / H
            ms = sum(v * v for v in xs) / H
            want_r = 1 / (Decimal(var.numerator) / Decimal(var.denominator) + Decimal(e.numerator) / Decimal(e.denominator)).sqrt()
            want_rr = 1 / (Decimal(ms.numerator) / Decimal(ms.denominator) + Decimal(e.numerator) / Decimal(e.denominator)).sqrt()
            assert abs(m[i] - float(mean)) <= 4 * np.spacing(abs(float(mean)) + 1e-300) + 1e-15 * float(sum(abs(v) for v in xs) / H)
            assert abs(r[i] - float(want_r)) <= 8 * np.spacing(float(want_r))
            assert abs(rr[i] - float(want_rr)) <= 8 * np.spacing(float(want_rr))


def test_invariants_mean_zero_var_ratio():
    rng = np.random.default_rng(6)
    x = rng.normal(0.3, 1.7, (16, 96))
    eps = 1e-3
    m, r = oracle.layernorm_stats(x, eps)
    xhat = oracle.norm_apply(x, m, r, np.ones(96), None, False)
    var = np.var(x, axis=1)                       # numpy's biased variance
    np.testing.assert_allclose(np.mean(xhat, axis=1), 0, atol=1e-14)
    np.testing.assert_allclose(np.mean(xhat ** 2, axis=1), var / (var + np.float32(eps)), rtol=1e-13)


def test_layernorm_equals_rmsnorm_on_zero_mean_rows():
    rng = np.random.default_rng(7)
    a = rng.normal(size=(8, 32))
    x = np.concatenate([a, -a], axis=1)           # every row has mean exactly 0
    g = (1 + 0.1 * rng.normal(size=64)).astype(np.float32)
    ln = oracle.layernorm_fwd(x, g, np.zeros(64, np.float32), 1e-6, False, "none", "f32")
    rms = oracle.rmsnorm_fwd(x, g, 1e-6, False, "none", "f32")
    np.testing.assert_allclose(ln["y"], rms["y"], rtol=1e-14, atol=1e-14)
    assert np.all(np.abs(ln["mu"]) < 1e-15)    # zero up to fp64 summation rounding


def test_scale_invariance_and_zero_centered():
    rng = np.random.default_rng(8)
    x = rng.normal(size=(4, 64))
    g = rng.normal(0, 0.1, 64).astype(np.float32)
    b = rng.normal(0, 0.1, 64).astype(np.float32)
    y1 = oracle.layernorm_fwd(x, g, b, 0.0, True, "none", "f32")["y"]
    y2 = oracle.layernorm_fwd(1000.0 * x + 5.0, g, b, 0.0, True, "none", "f32")["y"]
    np.testing.assert_allclose(y1, y2, rtol=1e-9, atol=1e-12)
    # zero-centered gamma g is the same as plain gamma 1 + g
    y3 = oracle.layernorm_fwd(x, (1.0 + g.astype(np.float64)), b, 0.0, False, "none", "f32")["y"]
    np.testing.assert_allclose(y1, y3, rtol=1e-14, atol=1e-14)


def test_h1_layernorm_is_beta():
    x = np.array([[3.5], [-2.0]])
    r = oracle.layernorm_fwd(x, np.array([2.0], np.float32), np.array([0.25], np.float32), 1e-5, False, "none", "f32")
    np.testing.assert_array_equal(r["y"], [[0.25], [0.25]])


# ----------------------------------------------------------- backward pins
def _loss(x, g, b, dz, eps, zc, ln):
    if ln:
        y = oracle.layernorm_fwd(x, g, b, eps, zc, "none", "f32")["y"]
    else:
        y = oracle.rmsnorm_fwd(x, g, eps, zc, "none", "f32")["y"]
    return float(np.sum(dz * y))


@pytest.mark.parametrize("ln", [True, False])
@pytest.mark.parametrize("zc", [False, True])
@pytest.mark.parametrize("H", [8, 40])
def test_backward_finite_differences(ln, zc, H):
    rng = np.random.default_rng(9 + H)
    N = 3
    x = rng.normal(0.2, 1.3, (N, H))
    g = rng.normal(0.1 if zc else 1.0, 0.3, H)
    b = rng.normal(0, 0.3, H)
    dz = rng.normal(size=(N, H))
    eps = 1e-2
    if ln:
        m, r = oracle.layernorm_stats(x, eps)
        res = oracle.layernorm_bwd(dz, x, m, r, g, zc, "f32")
    else:
        r = oracle.rmsnorm_stats(x, eps)
        res = oracle.rmsnorm_bwd(dz, x, r, g, zc, "f32")
    h = 1e-6
    fd_x = np.zeros_like(x)
    for i in range(N):
        for j in range(H):
            xp = x.copy(); xp[i, j] += h
            xm = x.copy(); xm[i, j] -= h
            fd_x[i, j] = (_loss(xp, g, b, dz, eps, zc, ln) - _loss(xm, g, b, dz, eps, zc, ln)) / (2 * h)
    fd_g = np.zeros(H)
    fd_b = np.zeros(H)
    for j in range(H):
        gp = g.copy(); gp[j] += h
        gm = g.copy(); gm[j] -= h
        fd_g[j] = (_loss(x, gp, b, dz, eps, zc, ln) - _loss(x, gm, b, dz, eps, zc, ln)) / (2 * h)
        bp = b.copy(); bp[j] += h
        bm = b.copy(); bm[j] -= h
        fd_b[j] = (_loss(x, g, bp, dz, eps, zc, ln) - _loss(x, g, bm, dz, eps, zc, ln)) / (2 * h)
    np.testing.assert_allclose(res["dx64"], fd_x, rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(res["dgamma64"], fd_g, rtol=1e-6, atol=1e-7)
    if ln:
        np.testing.assert_allclose(res["dbeta64"], fd_b, rtol=1e-6, atol=1e-7)
    else:
        assert "dbeta" not in res


def test_backward_row_identities():
    rng = np.random.default_rng(10)
    x = rng.normal(size=(5, 48))
    dz = rng.normal(size=(5, 48))
    g = rng.normal(1, 0.2, 48)
    m, r = oracle.layernorm_stats(x, 1e-5)
    dx = oracle.layernorm_bwd(dz, x, m, r, g, False, "f32")["dx64"]
    np.testing.assert_allclose(dx.sum(axis=1), 0, atol=1e-12)      # shift invariance
    rr = oracle.rmsnorm_stats(x, 0.0)
    dxr = oracle.rmsnorm_bwd(dz, x, rr, g, False, "f32")["dx64"]
    np.testing.assert_allclose((dxr * x).sum(axis=1), 0, atol=1e-11)  # scale invariance


def test_backward_dbeta_is_column_sum_of_dz():
    rng = np.random.default_rng(11)
    x = rng.normal(size=(6, 16))
    dz = rng.normal(size=(6, 16))
    m, r = oracle.layernorm_stats(x, 1e-5)
    res = oracle.layernorm_bwd(dz, x, m, r, np.ones(16), False, "f32")
    for j in range(16):
        assert res["dbeta64"][j] == pytest.approx(math.fsum(dz[:, j]), abs=1e-13)


# -------------------------------------------------------------- MXFP8 pins
def _bf_e4m3(v):
    """Brute-force nearest E4M3 code of one value (ties to even code)."""
    dec = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    a = min(abs(v), 448.0)
    best = min(range(0x7F), key=lambda c: (abs(a - dec[c]), c % 2))
    return best | (0x80 if math.copysign(1.0, v) < 0 else 0)


def _loop_mx_scale(block):
    A = max(abs(float(t)) for t in block)
    if A == 0:
        return 0
    _, k = math.frexp(A)
    return max(-127, min(127, k - 1 - 8)) + 127


def test_mxfp8_blocks_by_loops():
    rng = np.random.default_rng(12)
    N, H = 64, 96
    # rows and columns with very different magnitudes so that row and column
    # blocks get different scales (a transposition mistake would show)
    y = (rng.normal(size=(N, H)) * np.exp2(rng.integers(-6, 7, N))[:, None]
         * np.exp2(rng.integers(-5, 6, H))[None, :]).astype(np.float32)
    r = oracle.quantize(y, "mxfp8")
    assert r["data"].shape == (N, H) and r["row_scales"].shape == (N, H // 32)
    assert r["col_data"].shape == (H, N) and r["col_scales"].shape == (H, N // 32)
    for i in range(N):
        for jb in range(H // 32):
            blk = [float(t) for t in y[i, jb * 32:(jb + 1) * 32]]
            code = _loop_mx_scale(blk)
            assert r["row_scales"][i, jb] == code
            for t in range(0, 32, 7):
                assert r["data"][i, jb * 32 + t] == _bf_e4m3(blk[t] * 2.0 ** (127 - code))
    for j in range(H):
        for ib in range(N // 32):
            blk = [float(t) for t in y[ib * 32:(ib + 1) * 32, j]]
            code = _loop_mx_scale(blk)
            assert r["col_scales"][j, ib] == code
            for t in range(0, 32, 5):
                assert r["col_data"][j, ib * 32 + t] == _bf_e4m3(blk[t] * 2.0 ** (127 - code))


def test_mxfp8_dequant_error_bound():
    """decode(q) * 2**e is within half an E4M3 step of y (no block saturates
    beyond 448 * 2**e by more than the top step)."""
    rng = np.random.default_rng(13)
    y = (rng.normal(size=(64, 64)) * 3.0).astype(np.float32)
    r = oracle.quantize(y, "mxfp8")
    e = r["row_scales"].astype(np.int64) - 127
    deq = oracle.e4m3_decode(r["data"]).reshape(64, 2, 32) * np.exp2(e)[..., None]
    yy = y.astype(np.float64).reshape(64, 2, 32)
    scaled = np.abs(yy) * np.exp2(-e)[..., None]
    step = np.where(scaled < 2.0 ** -6, 2.0 ** -9, np.exp2(np.floor(np.log2(np.maximum(scaled, 1e-30))) - 3))
    err = np.abs(deq - yy) * np.exp2(-e)[..., None]
    ok = (err <= step / 2 + 1e-12) | (scaled >= 448)
    assert ok.all()


def test_fp8_pipeline_by_loops():
    """Whole fwd (LayerNorm + delayed FP8) on a tiny case by plain loops."""
    w = rn_inputs.make("ln_delayed", N=3, H=64)
    x = w.x_f64()
    res = oracle.layernorm_fwd(x, w.gamma, w.beta, w.eps, True, "fp8_delayed", scale=w.scale)
    eps = float(np.float32(w.eps))
    amax = 0.0
    for i in range(3):
        row = [float(t) for t in x[i]]
        m = math.fsum(row) / 64
        v = math.fsum((t - m) ** 2 for t in row) / 64
        rs = 1 / math.sqrt(v + eps)
        assert res["mu"][i] == np.float32(m) and res["rsigma"][i] == np.float32(rs)
        for j in range(64):
            y = (row[j] - m) * rs * (1.0 + float(w.gamma[j])) + float(w.beta[j])
            y32 = np.float32(y)
            amax = max(amax, abs(float(y32)))
            p = float(np.float32(y32 * np.float32(w.scale)))
            assert res["data"][i, j] == _bf_e4m3(p)
    assert res["amax"] == np.float32(amax)


# ------------------------------------------------- residual add + norm
def _bf16_exact_rne(fr):
    """Round a Fraction to the nearest bf16 (ties to even) by integer
    arithmetic on the exponent and an 8-bit significand."""
    from fractions import Fraction
    import math
    if fr == 0:
        return 0.0
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = a / Fraction(2) ** (e - 7)          # in [128, 256)
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * float(Fraction(n) * Fraction(2) ** (e - 7))


def test_residual_add_rounds_once_to_nearest_even():
    # ties at the bf16 ulp of 1 (2**-7) and of 256 (2): even wins; just above
    # a tie rounds up
    x = np.array([1.0, 1.0, 256.0, 256.0, -3.0], dtype=np.float64)
    r = np.array([2.0 ** -8, 2.0 ** -8 + 2.0 ** -16, 1.0, 3.0, 2.0 ** -8], dtype=np.float64)
    h = oracle.residual_add(x, r, "bf16")
    assert list(h) == [1.0, 1.0 + 2.0 ** -7, 256.0, 260.0, -3.0]
    # fp32 stream: 1 + 2**-24 is a tie at fp32's ulp of 1 -> 1
    h32 = oracle.residual_add(np.array([1.0]), np.array([2.0 ** -24]), "f32")
    assert h32[0] == 1.0


def test_residual_add_matches_exact_rational_rounding():
    from fractions import Fraction
    rng = np.random.default_rng(11)
    x = oracle.round_to_bf16(rng.normal(0, 4, 400))
    r = oracle.round_to_bf16(rng.normal(0, 1, 400) * np.exp2(rng.integers(-20, 8, 400)))
    h = oracle.residual_add(x, r, "bf16")
    want = [_bf16_exact_rne(Fraction(float(a)) + Fraction(float(b))) for a, b in zip(x, r)]
    assert np.array_equal(h, np.array(want))


def test_residual_add_norm_special_cases():
    rng = np.random.default_rng(12)
    x = oracle.round_to_bf16(rng.normal(0.3, 1.5, (5, 64)))
    g = rng.normal(1.0, 0.1, 64)
    b = rng.normal(0.0, 0.1, 64)
    # residual 0: the plain norms of x, and residual_out = x
    res = oracle.rmsnorm_add_fwd(x, np.zeros_like(x), g, 1e-5)
    ref = oracle.rmsnorm_fwd(x, g, 1e-5)
    assert np.array_equal(res["rsigma"], ref["rsigma"]) and np.array_equal(res["data"], ref["data"])
    assert np.array_equal(res["residual_out"], oracle.bf16_bits(x))
    res = oracle.layernorm_add_fwd(x, np.zeros_like(x), g, b, 1e-5)
    ref = oracle.layernorm_fwd(x, g, b, 1e-5)
    assert np.array_equal(res["mu"], ref["mu"]) and np.array_equal(res["data"], ref["data"])
    # residual -x: h = 0, rsigma = 1/sqrt(eps) exactly (fp32 eps), y = 0 (LN: beta)
    res = oracle.rmsnorm_add_fwd(x, -x, g, 1e-5)
    assert np.all(res["h"] == 0) and np.all(res["y"] == 0)
    assert np.allclose(res["rsigma"], np.float32(1.0 / np.sqrt(float(np.float32(1e-5)))), rtol=0, atol=0)
    res = oracle.layernorm_add_fwd(x, -x, g, b, 1e-5)
    assert np.all(res["mu"] == 0) and np.allclose(res["y"], np.broadcast_to(b, (5, 64)), rtol=0, atol=0)


def test_residual_add_rmsnorm_closed_form():
    # x = [1, 2, 3, 4], r = 1/2 -> h = [3/2, 5/2, 7/2, 9/2] (bf16-exact);
    # mean(h^2) = (9 + 25 + 49 + 81) / 16 = 41/4; with eps 0, rsigma = 2/sqrt(41)
    # and y_j = h_j * 2/sqrt(41) (gamma 1)
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    r = np.full((1, 4), 0.5)
    res = oracle.rmsnorm_add_fwd(x, r, np.ones(4), 0.0, out_dtype="f32")
    rs = 2.0 / np.sqrt(41.0)
    assert abs(float(res["rsigma"][0]) - rs) <= 1e-7 * rs
    assert np.allclose(res["y"], np.array([[1.5, 2.5, 3.5, 4.5]]) * rs, rtol=1e-15, atol=0)


# ------------------------------------------- delayed-scaling history step
def test_amax_history_update_by_hand():
    h, s, si = oracle.amax_history_update([4.0, 5.0, 3.0, 6.0], 2.0, 10.0)
    # shifted down, the new amax first; the oldest value (6) drops out
    assert list(h) == [2.0, 4.0, 5.0, 3.0]
    assert s == np.float32(448.0 / 5.0) and si == np.float32(1.0) / s
    # the new amax is the largest
    h, s, _ = oracle.amax_history_update([1.0, 1.0], 7.0, 3.0)
    assert list(h) == [7.0, 1.0] and s == np.float32(64.0)
    # length 1: the history is just the new amax
    h, s, _ = oracle.amax_history_update([9.0], 0.5, 3.0)
    assert list(h) == [0.5] and s == np.float32(896.0)


def test_amax_history_update_keeps_scale_without_a_usable_maximum():
    for hist, amax in (([0.0, 0.0, 0.0], 0.0), ([np.inf, 1.0], 2.0), ([1.0, 2.0], np.nan)):
        h, s, si = oracle.amax_history_update(hist, amax, 12.5)
        assert s == np.float32(12.5) and si == np.float32(0.08)
    # an infinity that has just dropped out no longer matters
    h, s, _ = oracle.amax_history_update([1.0, np.inf], 4.0, 12.5)
    assert list(h) == [4.0, 1.0] and s == np.float32(112.0)


def test_amax_history_update_matches_the_workload_scale():
    # the ln_delayed workload's scale is 448 / max(history): one step with a
    # new amax below that maximum leaves the maximum (unless it drops out)
    w = rn_inputs.make("ln_delayed", N=8, H=64)
    hist = w.amax_history
    h, s, _ = oracle.amax_history_update(hist, 1.0, w.scale)
    assert s == np.float32(np.float32(448.0) / np.max(hist[:-1]))


# -------------------------------------------------------------- NVFP4 pins
def _sections(name):
    sec, out = None, {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                sec = line.strip("[]")
                out[sec] = []
            else:
                out[sec].append(line.split())
    return out


def test_nvfp4_golden_by_hand():
    g = _sections("nvfp4_blocks.txt")
    y = np.array([[float(t) for t in r] for r in g["input"]], dtype=np.float32)
    r = oracle.quantize(y, "nvfp4")
    assert float(r["amax"]) == float(g["amax"][0][0])
    assert float(r["scale"]) == float(g["scale"][0][0])
    # scale_inv: 1/1536 correctly rounded to fp32 (within half an fp32 ulp)
    assert abs(float(r["scale_inv"]) - 1.0 / 1536.0) <= 2.0 ** -24 * (1.0 / 1536.0)
    assert [int(c) for c in r["row_scales"][:, 0]] == [int(t, 16) for t in g["row_scales"][0]]
    want = np.array([[int(t, 16) for t in row] for row in g["data"]], dtype=np.uint8)
    assert np.array_equal(r["data"], want)


def _nvfp4_case(seed, N=48, H=128):
    rng = np.random.default_rng(seed)
    # blocks of very different magnitudes, some zero blocks, some outliers
    y = rng.standard_normal((N, H)) * np.exp2(rng.integers(-12, 4, (N, H // 16)))[..., None].repeat(16, -1).reshape(N, H)
    y[rng.random((N, H)) < 0.02] *= 40.0
    y[:3, :16] = 0.0
    return y.astype(np.float32)


def test_nvfp4_scale_construction_properties():
    y = _nvfp4_case(30)
    N, H = y.shape
    r = oracle.quantize(y, "nvfp4")
    amax = float(np.max(np.abs(y)))
    assert float(r["amax"]) == amax
    S = float(r["scale"])
    assert abs(S - 2688.0 / amax) <= 2.0 ** -24 * (2688.0 / amax)        # one correct rounding
    sc = r["row_scales"]
    assert sc.shape == (N, H // 16) and r["data"].shape == (N, H // 2)
    codes = oracle.e2m1_unpack(r["data"]).reshape(N, H // 16, 16)
    yb = y.astype(np.float64).reshape(N, H // 16, 16)
    A = np.abs(yb).max(axis=-1)
    # the block that holds the tensor amax: A * S / 6 = 448 -> the top scale
    i, j = np.unravel_index(np.argmax(A), A.shape)
    assert sc[i, j] == 0x7E
    # scale codes are non-negative; zero blocks get scale 0 and codes 0
    assert np.all(sc < 0x80)
    zero = A == 0
    assert np.all(sc[zero] == 0) and np.all(codes[zero] == 0)
    v = oracle.e4m3_decode(sc)
    # blocks with a normal E4M3 scale: the largest element maps to +-6
    normal = v >= 2.0 ** -6
    top = np.take_along_axis(codes, np.abs(yb).argmax(axis=-1)[..., None], -1)[..., 0]
    assert np.all((top[normal] & 0x7) == 7)
    # dequantization: value = E2M1 * v / S; the E2M1 grid's largest half-step
    # is 1 (between 4 and 6), and v <= (A * S / 6) * (1 + 2**-4) for normal v
    deq = oracle.e2m1_decode(codes) * (v / S)[..., None]
    err = np.abs(deq - yb)
    bound = (A * 1.0625 / 6.0)[..., None] * (1 + 1e-6) + 1e-30
    assert np.all(err[normal] <= bound[normal])
    # signs: a nonzero code carries the sign of its element
    nz = (codes & 0x7) != 0
    assert np.all(((codes & 0x8) != 0)[nz] == (yb < 0)[nz])


def test_nvfp4_power_of_two_invariance():
    """Scaling the tensor by 2**j scales S by 2**-j exactly and leaves every
    code unchanged (all products shift exponent only), barring underflow."""
    y = _nvfp4_case(31)
    r0 = oracle.quantize(y, "nvfp4")
    for j in (-20, -3, 5, 30):
        r = oracle.quantize((y * np.float32(2.0 ** j)).astype(np.float32), "nvfp4")
        assert float(r["scale"]) == float(r0["scale"]) * 2.0 ** -j
        assert np.array_equal(r["row_scales"], r0["row_scales"])
        assert np.array_equal(r["data"], r0["data"])


def test_nvfp4_zero_and_tiny_tensors():
    r = oracle.quantize(np.zeros((2, 32), np.float32), "nvfp4")
    assert float(r["amax"]) == 0 and float(r["scale"]) == 1.0 and float(r["scale_inv"]) == 1.0
    assert not r["data"].any() and not r["row_scales"].any()
    # amax = 2**-140 (fp32 subnormal): 2688 / amax overflows fp32 -> capped
    y = np.zeros((1, 16), np.float32)
    y[0, 3] = np.float32(2.0 ** -140)
    r = oracle.quantize(y, "nvfp4")
    assert float(r["scale"]) == float(np.finfo(np.float32).max)


def _loop_nvfp4(y):
    """Row by row, block by block, element by element with fp32 scalars, a
    brute-force E4M3 for the scale and a brute-force E2M1 for the elements."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    amax = np.float32(max(abs(float(t)) for t in y.ravel()))
    S = np.float32(1.0) if amax == 0 else np.float32(np.float32(2688.0) / amax)
    k = np.float32(S / np.float32(6.0))
    N, H = y.shape
    scales = np.zeros((N, H // 16), np.uint8)
    codes = np.zeros((N, H), np.uint8)
    for i in range(N):
        for b in range(H // 16):
            blk = y[i, 16 * b:16 * b + 16]
            A = np.float32(max(abs(float(t)) for t in blk))
            c = _bf_e4m3(float(np.float32(A * k)))
            scales[i, b] = c
            vv = np.float32(oracle.e4m3_decode(np.uint8(c)))
            e = np.float32(0.0) if vv == 0 else np.float32(S / vv)
            for t in range(16):
                p = float(np.float32(blk[t] * e))
                a = min(abs(p), 6.0)
                m = min(range(8), key=lambda q: (abs(a - mags[q]), q % 2))
                codes[i, 16 * b + t] = m | (8 if math.copysign(1.0, p) < 0 else 0)
    packed = np.zeros((N, H // 2), np.uint8)
    for i in range(N):
        for jj in range(H // 2):
            packed[i, jj] = codes[i, 2 * jj] + 16 * codes[i, 2 * jj + 1]
    return packed, scales


def test_nvfp4_by_loops():
    y = _nvfp4_case(32, N=6, H=64)
    r = oracle.quantize(y, "nvfp4")
    packed, scales = _loop_nvfp4(y)
    assert np.array_equal(r["row_scales"], scales)
    assert np.array_equal(r["data"], packed)


def test_nvfp4_fused_forward_is_norm_then_quantize():
    """The NVFP4 forward quantizes fp32(y) of the same norm with the tensor
    amax of that y (the norm+amax then quantize path)."""
    w = rn_inputs.make("rms_current", N=8, H=256)
    x = w.x_f64()
    res = oracle.rmsnorm_fwd(x, w.gamma, w.eps, False, "nvfp4")
    y32 = res["y"].astype(np.float32)
    assert float(res["amax"]) == float(np.max(np.abs(y32)))
    packed, scales = _loop_nvfp4(y32)
    assert np.array_equal(res["data"], packed) and np.array_equal(res["row_scales"], scales)
