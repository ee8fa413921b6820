"""CPU pins of the oracle's scaled activations (oracle/act.py).

Pins (none re-runs the oracle's own formula):
* values worked by hand: SReLU on a few points, sigmoid(0) = 1/2 and
  sigmoid(ln 3) = 3/4 (so silu(ln 3) = (3/4) ln 3), SwiGLU with a zero gate;
* identities between the forms: clamped SwiGLU with an infinite limit and
  alpha = 1 equals SwiGLU with the linear half shifted by one; inside the
  bounds the clamps do nothing; beyond them the output no longer depends on
  the input; sigmoid(z) + sigmoid(-z) = 1 and no overflow at |z| = 800;
* central finite differences of L = sum(dy * s * act(x)) for dx (every
  form, both halves of the GLU gradient) and of L with respect to the row
  scales for dscales;
* the quantized outputs are the normalization quantizer applied to fp32(y).
"""
import math

import numpy as np
import pytest

import oracle
from oracle import act as A


def test_srelu_by_hand():
    x = np.array([[-2.0, -0.5, 0.0, 0.5, 3.0]])
    assert np.array_equal(A.act_value(x, "srelu"), [[0.0, 0.0, 0.0, 0.25, 9.0]])
    assert np.array_equal(A.act_grad(x, "srelu")[0], [[0.0, 0.0, 0.0, 1.0, 6.0]])


def test_sigmoid_and_silu_by_hand():
    assert A.sigmoid(0.0) == 0.5
    l3 = math.log(3.0)
    assert A.sigmoid(l3) == pytest.approx(0.75, rel=1e-15)
    assert A.sigmoid(-l3) == pytest.approx(0.25, rel=1e-15)
    # swiglu(a = ln 3, b = 2) = (3/4) ln 3 * 2; a zero gate gives 0 for any b
    x = np.array([[l3, 0.0, 2.0, 123.0]])
    y = A.act_value(x, "swiglu")
    assert y[0, 0] == pytest.approx(1.5 * l3, rel=1e-15) and y[0, 1] == 0.0
    # d/da silu(a) * b at a = 0 is b / 2; d/db = silu(0) = 0
    da, db = A.act_grad(np.array([[0.0, 4.0]]), "swiglu")
    assert da[0, 0] == 2.0 and db[0, 0] == 0.0


def test_sigmoid_symmetry_and_range():
    z = np.linspace(-800, 800, 20001)
    s = A.sigmoid(z)
    assert np.all(np.isfinite(s)) and s[0] == 0.0 and s[-1] == 1.0
    assert np.max(np.abs(s + A.sigmoid(-z) - 1.0)) <= 4.5e-16   # two ulps of 1


def test_clamped_swiglu_identities():
    rng = np.random.default_rng(50)
    a = rng.normal(0, 3, (16, 64))
    b = rng.normal(0, 3, (16, 64))
    x = np.concatenate([a, b], axis=1)
    # no clamp, alpha 1: silu(a) * (b + 1) = swiglu(a, b + 1)
    c = A.act_value(x, "clamped_swiglu", limit=np.inf, alpha=1.0)
    s = A.act_value(np.concatenate([a, b + 1.0], axis=1), "swiglu")
    assert np.max(np.abs(c - s)) <= 1e-13 * np.max(np.abs(s))
    # inside the bounds the clamps are inactive; beyond them the output is flat
    L = 7.0
    inside = (a <= L) & (np.abs(b) <= L)
    c7 = A.act_value(x, "clamped_swiglu", limit=L, alpha=1.702)
    cinf = A.act_value(x, "clamped_swiglu", limit=np.inf, alpha=1.702)
    assert np.array_equal(c7[inside], cinf[inside])
    x2 = x.copy()
    x2[:, :64] = np.where(a > L, a + 5.0, a)
    x2[:, 64:] = np.where(np.abs(b) > L, b * 2.0, b)
    assert np.array_equal(A.act_value(x2, "clamped_swiglu", limit=L), c7)
    da, db = A.act_grad(x2, "clamped_swiglu", limit=L)
    assert np.all(da[a > L] == 0) and np.all(db[np.abs(b) > L] == 0)


@pytest.mark.parametrize("act", A.ACTS)
def test_backward_finite_differences(act):
    rng = np.random.default_rng(51)
    n, h = 3, 8
    w = h if act == "srelu" else 2 * h
    x = rng.normal(0, 2.5, (n, w))
    if act == "clamped_swiglu":
        # keep every input away from the clamp bounds (kinks) by more than the step
        x = np.where(np.abs(np.abs(x) - 7.0) < 0.05, x + 0.2, x)
    if act == "srelu":
        x = np.where(np.abs(x) < 0.05, 0.3, x)
    dy = rng.normal(size=(n, h))
    s = rng.uniform(0.1, 1.0, n)
    res = A.scaled_act_bwd(dy, x, s, act, "f32")

    def loss(xx, ss):
        return np.sum(dy * ss[:, None] * A.act_value(xx, act))

    eps = 1e-6
    fd = np.zeros_like(x)
    for i in range(n):
        for j in range(w):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += eps
            xm[i, j] -= eps
            fd[i, j] = (loss(xp, s) - loss(xm, s)) / (2 * eps)
    assert np.max(np.abs(fd - res["dx64"])) <= 1e-6 * max(1.0, np.max(np.abs(fd)))
    fs = np.zeros(n)
    for i in range(n):
        sp, sm = s.copy(), s.copy()
        sp[i] += eps
        sm[i] -= eps
        fs[i] = (loss(x, sp) - loss(x, sm)) / (2 * eps)
    assert np.max(np.abs(fs - res["dscales64"])) <= 1e-6 * max(1.0, np.max(np.abs(fs)))


def test_clamped_swiglu_gradient_next_to_the_bounds():
    """Inputs just inside and just outside the limit: the finite-difference
    gradient is the clamped one (zero only outside)."""
    a = np.array([[6.5, 6.95, 7.05, 8.0, -3.0, -7.05]])
    b = np.array([[6.95, -6.95, 7.05, -7.05, 0.5, 2.0]])
    x = np.concatenate([a, b], axis=1)
    dy = np.ones((1, 6))
    res = A.scaled_act_bwd(dy, x, None, "clamped_swiglu", "f32")
    eps = 1e-6
    for j in range(12):
        xp, xm = x.copy(), x.copy()
        xp[0, j] += eps
        xm[0, j] -= eps
        fd = (A.act_value(xp, "clamped_swiglu").sum() - A.act_value(xm, "clamped_swiglu").sum()) / (2 * eps)
        assert res["dx64"][0, j] == pytest.approx(fd, abs=1e-6), j
    assert np.count_nonzero(res["dx64"][0, :6]) == 4 and np.count_nonzero(res["dx64"][0, 6:]) == 4


def test_no_scales_is_unit_scales_and_rounding():
    rng = np.random.default_rng(52)
    x = rng.normal(size=(4, 64))
    r1 = A.scaled_act_fwd(x, None, "swiglu", "none", "f32")
    r2 = A.scaled_act_fwd(x, np.ones(4), "swiglu", "none", "f32")
    assert np.array_equal(r1["data"], r2["data"])
    # the unquantized output is y rounded once
    rb = A.scaled_act_fwd(x, None, "swiglu", "none", "bf16")
    assert np.array_equal(rb["data"], oracle.bf16_bits(r1["y"]))


def test_quantized_outputs_are_the_norm_quantizer_on_fp32_y():
    rng = np.random.default_rng(53)
    x = rng.normal(0, 2, (64, 128))
    s = rng.uniform(0, 1, 64)
    r = A.scaled_act_fwd(x, s, "swiglu", "fp8_current")
    y32 = r["y"].astype(np.float32)
    assert float(r["amax"]) == float(np.max(np.abs(y32)))
    assert float(r["scale"]) == float(np.float32(448.0) / np.float32(r["amax"]))
    assert np.array_equal(r["data"], oracle.e4m3_encode((y32 * r["scale"]).astype(np.float64)))
    m = A.scaled_act_fwd(x, s, "swiglu", "mxfp8")
    assert m["data"].shape == (64, 64) and m["row_scales"].shape == (64, 2)
    assert "col_data" not in m
