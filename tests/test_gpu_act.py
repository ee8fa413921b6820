"""GPU parity of the scaled activations (rn_scaled_act_fwd / _bwd) against
the oracle (oracle/act.py), through the C ABI.

Tolerances (the arithmetic is a few fp32 products, one hardware exponential
-- relative error at most 2 + 1.17 |z| ulp, under 2**-18 for the |z| <= 25
these inputs stay within (x ~ N(0, 2), alpha * x for the clamped form) -- and
one 2-ulp division per element, so the kernel's y32 lies within a few tens
of fp32 ulps of the oracle's y; w is the magnitude of the product of terms
that forms a value, which also covers the bc + 1 of the clamped form):
* bf16 outputs within one bf16 ulp of the oracle's rounded value plus
  2**-18 * w; fp32 outputs within 2**-18 * w;
* FP8 and MXFP8 codes as for the normalization (one-step misses only
  within 1e-6 * scale * w of a rounding boundary, at most 0.1 %);
* amax within 1e-6 * max(w);
* dx as the outputs, with w the magnitude of s * dy * (the derivative's
  terms); dscales within 1e-5 * sum_j |dy * act| of the oracle's sum.
"""
import numpy as np
import pytest
import torch

import mxfp8_quantization_gb300 as rn
import oracle
import rn_inputs
from oracle import act as A
from parity import bf16_ulp, check_fp8_codes, check_mx
from test_gpu_parity import bf16_bits, to_dev

pytestmark = pytest.mark.gpu
LIM, ALPHA = 7.0, 1.702


@pytest.fixture(autouse=True)
def _no_device_error():
    yield
    assert rn.device_error() == 0


def _inputs(act, N, H, dtype, with_scales=True, seed=0):
    w = rn_inputs.make("moe_act", N=N, H=H, seed=seed)
    x64 = w.x_f64()
    dy64 = w.dz_f64()
    x, dy = w.x, w.dz
    if act == "srelu":                       # H inputs a row: the gate half
        x64 = np.ascontiguousarray(x64[:, :H])
        x = np.ascontiguousarray(x[:, :H])
    if dtype == "f32":
        x = x64.astype(np.float32)
        dy = dy64.astype(np.float32)
    s = w.scales if with_scales else None
    return x, x64, dy, dy64, s


def _split(x64, act):
    h = x64.shape[1] if act == "srelu" else x64.shape[1] // 2
    return x64[:, :h], (None if act == "srelu" else x64[:, h:])


def _w_fwd(x64, s, act):
    """Magnitude of the product of terms that forms y."""
    a, b = _split(x64, act)
    sc = np.ones(a.shape[0]) if s is None else s.astype(np.float64)
    if act == "srelu":
        w = np.maximum(a, 0) ** 2
    elif act == "swiglu":
        w = np.abs(a * A.sigmoid(a) * b)
    else:
        ac = np.minimum(a, LIM)
        bc = np.clip(b, -LIM, LIM)
        w = np.abs(ac * A.sigmoid(ALPHA * ac)) * (np.abs(bc) + 1.0)
    return w * np.abs(sc)[:, None]


def _w_bwd(x64, dy64, s, act):
    a, b = _split(x64, act)
    sd = np.abs(dy64) * (1.0 if s is None else np.abs(s.astype(np.float64))[:, None])
    if act == "srelu":
        return sd * 2 * np.maximum(a, 0)
    if act == "swiglu":
        sg = A.sigmoid(a)
        return np.concatenate([sd * np.abs(b) * sg * (1 + np.abs(a) * (1 - sg)), sd * np.abs(a) * sg], 1)
    ac = np.minimum(a, LIM)
    bc = np.clip(b, -LIM, LIM)
    sg = A.sigmoid(ALPHA * ac)
    return np.concatenate([sd * (np.abs(bc) + 1) * sg * (1 + ALPHA * np.abs(ac) * (1 - sg)),
                           sd * np.abs(ac) * sg], 1)


def _check_values(got64, ref64, w, dtype, what):
    if dtype == "bf16":
        ref = oracle.round_to_bf16(ref64)
        tol = bf16_ulp(ref) + 2.0 ** -18 * w
    else:
        ref = ref64
        tol = 2.0 ** -18 * w + 1e-38
    err = np.abs(got64 - ref)
    bad = err > tol
    assert not bad.any(), f"{what}: {bad.sum()} off, max err/tol {np.max(err / tol):.3f}"


def _dev(a, dtype):
    return to_dev(a, dtype)


FWD = [
    # (act, dtype, mode, N, H, scales)
    ("swiglu", "bf16", "none", 203, 1024, True),
    ("swiglu", "bf16", "none", 37, 2056, True),      # a second, one-chunk slice per row
    ("swiglu", "bf16", "none", 9, 4096, False),      # two full slices, no scales
    ("srelu", "bf16", "fp8_delayed", 203, 1024, True),
    ("clamped_swiglu", "bf16", "fp8_current", 150, 2048, True),
    ("swiglu", "f32", "none", 67, 1000, True),
    ("clamped_swiglu", "f32", "fp8_delayed", 67, 512, True),
    ("swiglu", "bf16", "mxfp8", 64, 256, True),
    ("srelu", "f32", "mxfp8", 40, 96, True),          # blocks over 8 lanes
    ("clamped_swiglu", "bf16", "mxfp8", 33, 2080, False),
]


@pytest.mark.parametrize("case", FWD, ids=lambda c: f"{c[0]}-{c[1]}-{c[2]}-{c[3]}x{c[4]}")
def test_scaled_act_forward(case):
    act, dtype, mode, N, H, with_s = case
    x, x64, _, _, s = _inputs(act, N, H, dtype, with_s)
    sd = None if s is None else torch.from_numpy(s).cuda()
    scale = float(np.float32(448.0) / np.float32(30.0)) if mode == "fp8_delayed" else None
    out = rn.scaled_act_fwd(_dev(x, dtype), act, sd, quant=mode, limit=LIM, alpha=ALPHA, scale=scale)
    ref = A.scaled_act_fwd(x64, s, act, mode, dtype, LIM, ALPHA, scale=scale)
    w = _w_fwd(x64, s, act)
    y32 = ref["y"].astype(np.float32)
    if mode == "none":
        got = (bf16_bits(out).astype(np.uint32) << 16).view(np.float32) if dtype == "bf16" \
            else out.cpu().numpy()
        _check_values(got.astype(np.float64), ref["y"], w, dtype, act)
    elif mode == "mxfp8":
        assert out.col_data is None
        check_mx(out.data.cpu().numpy(), out.row_scales.cpu().numpy(), y32, w, "act-mx")
    else:
        am = float(out.amax.item())
        assert abs(am - float(ref["amax"])) <= 1e-6 * w.max()
        if mode == "fp8_current":
            s_gpu = np.float32(out.scale.item())
            assert s_gpu == np.float32(448.0) / np.float32(am)
            s_ref = float(ref["scale"])
        else:
            s_gpu = s_ref = float(np.float32(scale))
        p = (y32 * np.float32(s_ref)).astype(np.float64)
        win = 1e-6 * s_ref * w + np.abs(p) * abs(float(s_gpu) / s_ref - 1.0)
        check_fp8_codes(out.data.cpu().numpy(), ref["data"], p, win, f"act {mode}")


BWD = [
    ("swiglu", "bf16", 203, 1024, True),
    ("swiglu", "bf16", 37, 2056, False),
    ("srelu", "bf16", 203, 1024, True),
    ("clamped_swiglu", "bf16", 150, 2048, True),
    ("swiglu", "f32", 67, 1000, True),
    ("srelu", "f32", 33, 4100, True),
    ("clamped_swiglu", "f32", 67, 512, False),
]


@pytest.mark.parametrize("case", BWD, ids=lambda c: f"{c[0]}-{c[1]}-{c[2]}x{c[3]}")
def test_scaled_act_backward(case):
    act, dtype, N, H, with_s = case
    x, x64, dy, dy64, s = _inputs(act, N, H, dtype, with_s)
    sd = None if s is None else torch.from_numpy(s).cuda()
    dx, ds = rn.scaled_act_bwd(_dev(dy, dtype), _dev(x, dtype), act, sd, limit=LIM, alpha=ALPHA)
    ref = A.scaled_act_bwd(dy64, x64, s, act, dtype, LIM, ALPHA)
    got = (bf16_bits(dx).astype(np.uint32) << 16).view(np.float32) if dtype == "bf16" \
        else dx.cpu().numpy()
    _check_values(got.astype(np.float64), ref["dx64"], _w_bwd(x64, dy64, s, act), dtype, "dx")
    bound = 1e-5 * np.sum(np.abs(dy64 * A.act_value(x64, act, LIM, ALPHA)), axis=1) + 1e-30
    err = np.abs(ds.cpu().numpy().astype(np.float64) - ref["dscales64"])
    assert np.all(err <= bound), f"dscales: max err/bound {np.max(err / bound):.3f}"
    # without dscales the same dx
    dx2, ds2 = rn.scaled_act_bwd(_dev(dy, dtype), _dev(x, dtype), act, sd, limit=LIM, alpha=ALPHA,
                                 dscales=False)
    assert ds2 is None and torch.equal(dx, dx2)


def test_scaled_act_empty():
    x = torch.empty((0, 512), dtype=torch.bfloat16, device="cuda")
    y = rn.scaled_act_fwd(x, "swiglu")
    assert y.shape == (0, 256)
    r = rn.scaled_act_fwd(x, "swiglu", quant="fp8_current")
    assert r.amax.item() == 0 and r.scale.item() == 1.0
    dx, ds = rn.scaled_act_bwd(torch.empty((0, 256), dtype=torch.bfloat16, device="cuda"), x, "swiglu")
    assert dx.shape == (0, 512) and ds.shape == (0,)


def test_moe_act_65536x2048_sampled():
    """The benchmarked workload at full size: forward bf16 and FP8 current
    scaling (tensor amax over every row), backward, on sampled rows."""
    w = rn_inputs.make("moe_act")
    x = _dev(w.x, "bf16")
    sd = torch.from_numpy(w.scales).cuda()
    dy = _dev(w.dz, "bf16")
    y = rn.scaled_act_fwd(x, "swiglu", sd)
    yq = rn.scaled_act_fwd(x, "swiglu", sd, quant="fp8_current")
    dx, ds = rn.scaled_act_bwd(dy, x, "swiglu", sd)
    amax = np.float32(0)
    wmax = 0.0
    for r0 in range(0, w.N, 4096):
        xb = w.x_f64(slice(r0, r0 + 4096))
        sb = w.scales[r0:r0 + 4096]
        yb = A.act_value(xb, "swiglu") * sb.astype(np.float64)[:, None]
        amax = max(amax, np.float32(np.max(np.abs(yb.astype(np.float32)))))
        wmax = max(wmax, float(_w_fwd(xb, sb, "swiglu").max()))
    assert abs(float(yq.amax.item()) - float(amax)) <= 1e-6 * wmax
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([rng.choice(w.N, 300, replace=False), [0, w.N - 1]]))
    xr = w.x_f64(rows)
    sr = w.scales[rows]
    ref = A.scaled_act_fwd(xr, sr, "swiglu", "fp8_current", amax=amax)
    wr = _w_fwd(xr, sr, "swiglu")
    got = (bf16_bits(y).astype(np.uint32) << 16).view(np.float32)[rows].astype(np.float64)
    _check_values(got, ref["y"], wr, "bf16", "y")
    s_ref = float(ref["scale"])
    p = (ref["y"].astype(np.float32) * np.float32(s_ref)).astype(np.float64)
    win = 1e-6 * s_ref * wr + np.abs(p) * abs(float(yq.scale.item()) / s_ref - 1.0)
    check_fp8_codes(yq.data.cpu().numpy()[rows], ref["data"], p, win, "moe fp8 current")
    dyr = w.dz_f64(rows)
    rb = A.scaled_act_bwd(dyr, xr, sr, "swiglu", "bf16")
    gotdx = (bf16_bits(dx).astype(np.uint32) << 16).view(np.float32)[rows].astype(np.float64)
    _check_values(gotdx, rb["dx64"], _w_bwd(xr, dyr, sr, "swiglu"), "bf16", "dx")
    bound = 1e-5 * np.sum(np.abs(dyr * A.act_value(xr, "swiglu")), axis=1)
    assert np.all(np.abs(ds.cpu().numpy()[rows] - rb["dscales64"]) <= bound)
