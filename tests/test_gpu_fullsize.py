"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (the public entry points, sm_margin 0 unless stated).

The oracle computes every row where the checked quantity needs it (tensor
amax, dgamma / dbeta) and samples rows otherwise (the element-wise outputs),
always including the first and the last row / row tile.
"""
import numpy as np
import pytest
import torch

import mxfp8_quantization_gb300 as rn
import oracle
import rn_inputs
from parity import (bf16_ulp, check_fp8_codes, check_mx, check_nvfp4, check_stats,
                    term_magnitude)
from test_gpu_parity import bf16_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_error():
    yield
    assert rn.device_error() == 0


def _sample_rows(N, n, seed=0, align=1):
    rng = np.random.default_rng(seed)
    units = N // align
    pick = set(rng.choice(units, size=min(n, units), replace=False).tolist()) | {0, units - 1}
    rows = np.concatenate([np.arange(u * align, (u + 1) * align) for u in sorted(pick)])
    return rows


def test_ln_delayed_8192x4096_fwd_and_bwd():
    w = rn_inputs.make("ln_delayed")
    x = to_dev(w.x, "bf16")
    g = to_dev(w.gamma, "f32")
    b = to_dev(w.beta, "f32")
    out, mu, rs = rn.layernorm_fwd(x, g, b, w.eps, quant="fp8_delayed", scale=w.scale,
                                   zero_centered_gamma=True)
    x64 = w.x_f64()
    ref = oracle.layernorm_fwd(x64, w.gamma, w.beta, w.eps, True, "fp8_delayed", scale=w.scale)
    mu_h, rs_h = mu.cpu().numpy(), rs.cpu().numpy()
    check_stats(mu_h, rs_h, x64, ref["mu"], ref["rsigma"])
    wt = term_magnitude(x64, ref["mu"], ref["rsigma"], w.gamma, w.beta, True)
    s = np.float32(w.scale)
    p = (ref["y"].astype(np.float32) * s).astype(np.float64)
    check_fp8_codes(out.data.cpu().numpy(), ref["data"], p, 1e-6 * float(s) * wt, "ln fp8 delayed")
    assert abs(out.amax.item() - float(ref["amax"])) <= 1e-6 * wt.max()
    del wt, p
    # backward from the oracle's saved statistics
    dz = to_dev(w.dz, "bf16")
    dx, dg, db = rn.layernorm_bwd(dz, x, torch.from_numpy(ref["mu"]).cuda(),
                                  torch.from_numpy(ref["rsigma"]).cuda(), g, 0, True)
    rb = oracle.layernorm_bwd(w.dz_f64(), x64, ref["mu"], ref["rsigma"], w.gamma, True, "bf16")
    got = (bf16_bits(dx).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r = oracle.round_to_bf16(rb["dx64"])
    rms = np.sqrt(np.mean(rb["dx64"] ** 2, axis=1, keepdims=True))
    err = np.abs(got - r)
    assert np.all((err <= bf16_ulp(r)) | (err <= 2e-3 * rms))
    xhat = (x64 - ref["mu"][:, None].astype(np.float64)) * ref["rsigma"][:, None].astype(np.float64)
    dz64 = w.dz_f64()
    assert np.all(np.abs(dg.cpu().numpy() - rb["dgamma64"]) <= 1e-3 * np.sum(np.abs(dz64 * xhat), axis=0))
    assert np.all(np.abs(db.cpu().numpy() - rb["dbeta64"]) <= 1e-3 * np.sum(np.abs(dz64), axis=0))


def test_rms_current_16384x8192():
    w = rn_inputs.make("rms_current")
    x = to_dev(w.x, "bf16")
    g = to_dev(w.gamma, "f32")
    out, rs = rn.rmsnorm_fwd(x, g, w.eps, quant="fp8_current")
    rs_h = rs.cpu().numpy()
    # tensor amax over every row, in row blocks
    amax = np.float32(0.0)
    wmax = 0.0
    r_all = np.empty(w.N, np.float64)
    for r0 in range(0, w.N, 2048):
        xb = w.x_f64(slice(r0, r0 + 2048))
        f = oracle.rmsnorm_fwd(xb, w.gamma, w.eps, False, "none", "f32")
        amax = max(amax, oracle.norm.tensor_amax(f["y"].astype(np.float32)))
        r_all[r0:r0 + 2048] = oracle.rmsnorm_stats(xb, w.eps)
        wmax = max(wmax, float(term_magnitude(xb, None, f["rsigma"], w.gamma, None, False).max()))
    assert np.all(np.abs(rs_h - r_all) <= 1e-5 * r_all)
    am_gpu = np.float32(out.amax.item())
    assert abs(float(am_gpu) - float(amax)) <= 1e-6 * wmax
    s_gpu = np.float32(out.scale.item())
    assert s_gpu == np.float32(448.0) / am_gpu
    assert np.float32(out.scale_inv.item()) == np.float32(1.0) / s_gpu
    rows = _sample_rows(w.N, 400, seed=1)
    xr = w.x_f64(rows)
    ref = oracle.rmsnorm_fwd(xr, w.gamma, w.eps, False, "fp8_current", amax=amax)
    s_ref = float(ref["scale"])
    wt = term_magnitude(xr, None, ref["rsigma"], w.gamma, None, False)
    p = (ref["y"].astype(np.float32) * np.float32(s_ref)).astype(np.float64)
    win = 1e-6 * s_ref * wt + np.abs(p) * abs(float(s_gpu) / s_ref - 1.0)
    check_fp8_codes(out.data.cpu().numpy()[rows], ref["data"], p, win, "rms fp8 current")


def test_rms_nvfp4_16384x8192():
    """The NVFP4 path on the current-scaling workload (the bench's NVFP4
    line): tensor amax over every row, codes and block scales on sampled
    rows."""
    w = rn_inputs.make("rms_current")
    x = to_dev(w.x, "bf16")
    g = to_dev(w.gamma, "f32")
    out, rs = rn.rmsnorm_fwd(x, g, w.eps, quant="nvfp4")
    amax = np.float32(0.0)
    wmax = 0.0
    for r0 in range(0, w.N, 2048):
        xb = w.x_f64(slice(r0, r0 + 2048))
        f = oracle.rmsnorm_fwd(xb, w.gamma, w.eps, False, "none", "f32")
        amax = max(amax, oracle.norm.tensor_amax(f["y"].astype(np.float32)))
        wmax = max(wmax, float(term_magnitude(xb, None, f["rsigma"], w.gamma, None, False).max()))
    am_gpu = np.float32(out.amax.item())
    assert abs(float(am_gpu) - float(amax)) <= 1e-6 * wmax
    S = np.float32(out.scale.item())
    assert S == np.float32(2688.0) / am_gpu
    assert np.float32(out.scale_inv.item()) == np.float32(1.0) / S
    rows = _sample_rows(w.N, 400, seed=3)
    xr = w.x_f64(rows)
    ref = oracle.rmsnorm_fwd(xr, w.gamma, w.eps, False, "nvfp4", amax=amax)
    check_stats(None, rs.cpu().numpy()[rows], xr, None, ref["rsigma"])
    wt = term_magnitude(xr, None, ref["rsigma"], w.gamma, None, False)
    check_nvfp4(out.data.cpu().numpy()[rows], out.row_scales.cpu().numpy()[rows],
                ref["y"].astype(np.float32), wt, ref["scale"], S, "rms nvfp4 full")


@pytest.mark.parametrize("ln", [True, False], ids=["ln", "rms"])
def test_mxfp8_65536x2048(ln):
    w = rn_inputs.make("mxfp8")
    x = to_dev(w.x, "bf16")
    g = to_dev(w.gamma, "f32")
    if ln:
        out, mu, rs = rn.layernorm_fwd(x, g, to_dev(w.beta, "f32"), w.eps, quant="mxfp8")
    else:
        out, rs = rn.rmsnorm_fwd(x, g, w.eps, quant="mxfp8")
    rows = _sample_rows(w.N, 24, seed=2, align=32)
    xr = w.x_f64(rows)
    if ln:
        ref = oracle.layernorm_fwd(xr, w.gamma, w.beta, w.eps, False, "none", "f32")
        check_stats(mu.cpu().numpy()[rows], rs.cpu().numpy()[rows], xr, ref["mu"], ref["rsigma"])
        wt = term_magnitude(xr, ref["mu"], ref["rsigma"], w.gamma, w.beta, False)
    else:
        ref = oracle.rmsnorm_fwd(xr, w.gamma, w.eps, False, "none", "f32")
        check_stats(None, rs.cpu().numpy()[rows], xr, None, ref["rsigma"])
        wt = term_magnitude(xr, None, ref["rsigma"], w.gamma, None, False)
    y32 = ref["y"].astype(np.float32)
    check_mx(out.data.cpu().numpy()[rows], out.row_scales.cpu().numpy()[rows], y32, wt, "mx-row")
    # columnwise: each sampled 32-row tile is a set of column blocks
    cd = out.col_data.cpu().numpy()
    cs = out.col_scales.cpu().numpy()
    tiles = rows.reshape(-1, 32)
    for i, tr in enumerate(tiles):
        yt = np.ascontiguousarray(y32[32 * i:32 * (i + 1)].T)
        wtt = np.ascontiguousarray(wt[32 * i:32 * (i + 1)].T)
        check_mx(cd[:, tr[0]:tr[0] + 32], cs[:, tr[0] // 32:tr[0] // 32 + 1], yt, wtt, "mx-col")


@pytest.mark.parametrize("ln", [True, False], ids=["ln", "rms"])
@pytest.mark.parametrize("name", ["bwd_f32", "bwd_bf16"])
def test_backward_full(name, ln):
    w = rn_inputs.make(name)
    N, H = w.N, w.H
    x = to_dev(w.x, w.dtype)
    dz = to_dev(w.dz, w.dtype)
    g = to_dev(w.gamma, "f32")
    # oracle statistics (fp32, as saved by a forward) and the full dgamma /
    # dbeta, accumulated over row blocks in fp64
    mu = np.empty(N, np.float32) if ln else None
    rs = np.empty(N, np.float32)
    dg_ref = np.zeros(H)
    db_ref = np.zeros(H)
    den_g = np.zeros(H)
    den_b = np.zeros(H)
    for r0 in range(0, N, 8192):
        sl = slice(r0, min(N, r0 + 8192))
        xb = w.x_f64(sl)
        dzb = w.dz_f64(sl)
        if ln:
            m, r = oracle.layernorm_stats(xb, w.eps)
            mu[sl], rs[sl] = m.astype(np.float32), r.astype(np.float32)
            b = oracle.layernorm_bwd(dzb, xb, mu[sl], rs[sl], w.gamma, False, w.dtype)
            db_ref += b["dbeta64"]
            xhat = (xb - mu[sl][:, None].astype(np.float64)) * rs[sl][:, None].astype(np.float64)
        else:
            rs[sl] = oracle.rmsnorm_stats(xb, w.eps).astype(np.float32)
            b = oracle.rmsnorm_bwd(dzb, xb, rs[sl], w.gamma, False, w.dtype)
            xhat = xb * rs[sl][:, None].astype(np.float64)
        dg_ref += b["dgamma64"]
        den_g += np.sum(np.abs(dzb * xhat), axis=0)
        den_b += np.sum(np.abs(dzb), axis=0)
    mud = torch.from_numpy(mu).cuda() if ln else None
    rsd = torch.from_numpy(rs).cuda()
    outs = {}
    for margin in (0, 16):
        if ln:
            outs[margin] = rn.layernorm_bwd(dz, x, mud, rsd, g, margin, False)
        else:
            outs[margin] = rn.rmsnorm_bwd(dz, x, rsd, g, margin, False)
    for a, b2 in zip(outs[0], outs[16]):            # sm_margin changes nothing
        assert torch.equal(a, b2)
    res = outs[0]
    assert np.all(np.abs(res[1].cpu().numpy() - dg_ref) <= 1e-3 * den_g)
    if ln:
        assert np.all(np.abs(res[2].cpu().numpy() - db_ref) <= 1e-3 * den_b)
    rows = _sample_rows(N, 300, seed=3)
    xr, dzr = w.x_f64(rows), w.dz_f64(rows)
    if ln:
        rb = oracle.layernorm_bwd(dzr, xr, mu[rows], rs[rows], w.gamma, False, w.dtype)
    else:
        rb = oracle.rmsnorm_bwd(dzr, xr, rs[rows], w.gamma, False, w.dtype)
    dx64 = rb["dx64"]
    rms = np.sqrt(np.mean(dx64 ** 2, axis=1, keepdims=True))
    if w.dtype == "bf16":
        got = (bf16_bits(res[0]).astype(np.uint32) << 16).view(np.float32).astype(np.float64)[rows]
        r = oracle.round_to_bf16(dx64)
        err = np.abs(got - r)
        assert np.all((err <= bf16_ulp(r)) | (err <= 2e-3 * rms))
    else:
        got = res[0].cpu().numpy()[rows].astype(np.float64)
        assert np.all(np.abs(got - dx64) <= 2e-3 * np.maximum(np.abs(dx64), rms))
    rowrel = np.linalg.norm(got - dx64, axis=1) / np.linalg.norm(dx64, axis=1)
    assert np.all(rowrel <= 2e-3)
