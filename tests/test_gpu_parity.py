"""GPU parity: the CUDA kernels (through the C ABI) against the fp64 oracle.

Inputs come from rn_inputs (seeded), identical for both sides.  Sizes here
span several tiles and a ragged tail; the full workload sizes are covered in
test_gpu_fullsize.py.
"""
import numpy as np
import pytest
import torch

import mxfp8_quantization_gb300 as rn
import oracle
import rn_inputs
from parity import (check_bf16, check_fp8_codes, check_mx, check_stats, term_magnitude)

pytestmark = pytest.mark.gpu


def to_dev(a, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def bf16_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.fixture(autouse=True)
def _no_device_error():
    yield
    assert rn.device_error() == 0


# ------------------------------------------------------ quantizer, exact
def _e4m3_class_values():
    """Every fp32 sign/exponent/top-12-mantissa pattern with low bits from a
    covering set: all rounding decisions of fp32 -> E4M3 are represented."""
    s = np.arange(2, dtype=np.uint32)[:, None, None, None] << 31
    e = np.arange(256, dtype=np.uint32)[None, :, None, None] << 23
    m = np.arange(4096, dtype=np.uint32)[None, None, :, None] << 11
    lo = np.array([0, 1, 0x3FF, 0x400, 0x401, 0x7FF], dtype=np.uint32)[None, None, None, :]
    return (s | e | m | lo).reshape(-1).view(np.float32)


def test_quantize_only_e4m3_all_rounding_classes():
    y = _e4m3_class_values().reshape(-1, 4096)          # [3072, 4096]
    yd = to_dev(y, "f32")
    r = rn.quantize_only(yd, "fp8_delayed", scale=1.0)
    got = r.data.cpu().numpy()
    want = oracle.e4m3_encode(y.astype(np.float64))
    bad = got != want
    assert not bad.any(), (f"{bad.sum()} mismatches, e.g. y={y[bad][:6]} gpu={got[bad][:6]} "
                           f"ref={want[bad][:6]}")
    assert np.isnan(r.amax.item())                       # the set holds NaNs: NaN wins
    assert r.scale_inv.item() == 1.0


def test_quantize_only_delayed_and_current_bit_exact():
    rng = np.random.default_rng(20)
    y = (rng.standard_normal((517, 1024)) * np.exp2(rng.uniform(-20, 20, (517, 1)))).astype(np.float32)
    yd = to_dev(y, "f32")
    s = np.float32(448.0) / np.float32(5.3)
    r = rn.quantize_only(yd, "fp8_delayed", scale=float(s))
    ref = oracle.quantize(y, "fp8_delayed", scale=s)
    assert np.array_equal(r.data.cpu().numpy(), ref["data"])
    assert r.amax.cpu().numpy()[0] == ref["amax"]
    assert r.scale_inv.cpu().numpy()[0] == ref["scale_inv"]
    r = rn.quantize_only(yd, "fp8_current")
    ref = oracle.quantize(y, "fp8_current")
    assert r.amax.cpu().numpy()[0] == ref["amax"]
    assert r.scale.cpu().numpy()[0] == ref["scale"]
    assert r.scale_inv.cpu().numpy()[0] == ref["scale_inv"]
    assert np.array_equal(r.data.cpu().numpy(), ref["data"])


def test_quantize_only_current_all_zero():
    yd = torch.zeros((64, 256), dtype=torch.float32, device="cuda")
    r = rn.quantize_only(yd, "fp8_current")
    assert r.amax.item() == 0 and r.scale.item() == 1.0 and r.scale_inv.item() == 1.0
    assert int(r.data.max()) == 0


def _mx_sweep_values():
    """Blocks whose maxima sweep every fp32 exponent (plus zero blocks and
    subnormal blocks); within a block the values span 2**-12 .. 1 of the max."""
    rng = np.random.default_rng(21)
    rows = []
    for field in range(0, 255):
        for mant in (0, 0x400000, 0x7FFFFF, int(rng.integers(0, 1 << 23))):
            amax = np.array([(field << 23) | mant], dtype=np.uint32).view(np.float32)[0]
            blk = (rng.uniform(-1, 1, 32) * np.exp2(rng.integers(-12, 1, 32))).astype(np.float32) * amax
            blk[rng.integers(0, 32)] = amax * (1 if rng.random() < 0.5 else -1)
            rows.append(blk)
    rows.append(np.zeros(32, np.float32))
    rows.append((rng.uniform(-1, 1, 32) * 2.0 ** -140).astype(np.float32))   # subnormal block
    arr = np.concatenate(rows)
    H = 256
    arr = np.concatenate([arr, np.zeros((-arr.size) % (32 * H), np.float32)])
    return arr.reshape(-1, H)                     # [128, 256]: N and H multiples of 32


def test_quantize_only_mxfp8_bit_exact():
    y = _mx_sweep_values()
    assert y.shape[0] % 32 == 0 and y.shape[0] >= 32
    r = rn.quantize_only(to_dev(y, "f32"), "mxfp8")
    ref = oracle.quantize(y, "mxfp8")
    for k in ("data", "row_scales", "col_data", "col_scales"):
        got = getattr(r, k).cpu().numpy()
        bad = got != ref[k]
        assert not bad.any(), f"{k}: {bad.sum()} mismatches"


def test_quantize_only_mxfp8_single_direction():
    rng = np.random.default_rng(22)
    y = rng.standard_normal((64, 256)).astype(np.float32)
    ref = oracle.quantize(y, "mxfp8")
    r = rn.quantize_only(to_dev(y, "f32"), "mxfp8", colwise=False)
    assert r.col_data is None and np.array_equal(r.data.cpu().numpy(), ref["data"])
    r = rn.quantize_only(to_dev(y, "f32"), "mxfp8", rowwise=False)
    assert r.data is None and np.array_equal(r.col_data.cpu().numpy(), ref["col_data"])
    assert np.array_equal(r.col_scales.cpu().numpy(), ref["col_scales"])


# -------------------------------------------------------- fused forward
def _run_fwd(w, ln, mode, sm_margin=0, out_dtype=None, rowwise=True, colwise=True):
    x = to_dev(w.x, w.dtype)
    g = to_dev(w.gamma, "f32")
    kw = dict(quant=mode, sm_margin=sm_margin, zero_centered_gamma=w.zero_centered_gamma,
              out_dtype=out_dtype)
    if mode == "fp8_delayed":
        kw["scale"] = w.scale
    if mode == "mxfp8":
        kw.update(rowwise=rowwise, colwise=colwise)
    if ln:
        b = to_dev(w.beta, "f32") if w.beta is not None else None
        out, mu, rs = rn.layernorm_fwd(x, g, b, w.eps, **kw)
        return out, mu.cpu().numpy(), rs.cpu().numpy()
    out, rs = rn.rmsnorm_fwd(x, g, w.eps, **kw)
    return out, None, rs.cpu().numpy()


def _oracle_fwd(w, ln, mode, amax=None):
    x = w.x_f64()
    if ln:
        return oracle.layernorm_fwd(x, w.gamma, w.beta, w.eps, w.zero_centered_gamma, mode,
                                    scale=w.scale, amax=amax)
    return oracle.rmsnorm_fwd(x, w.gamma, w.eps, w.zero_centered_gamma, mode, scale=w.scale,
                              amax=amax)


def _terms(w, ref, ln):
    return term_magnitude(w.x_f64(), ref.get("mu") if ln else None, ref["rsigma"], w.gamma,
                          w.beta if ln else None, w.zero_centered_gamma)


FWD_CASES = [
    # (workload, N, H, ln, mode)
    ("rms_small", None, None, False, "none"),
    ("rms_small", None, None, False, "fp8_delayed"),
    ("rms_small", 203, 1024, False, "fp8_current"),
    ("ln_delayed", 75, None, True, "fp8_delayed"),
    ("ln_delayed", 75, None, True, "none"),
    ("ln_delayed", 45, 1000, True, "none"),
    ("rms_current", 203, None, False, "fp8_current"),
    ("rms_current", 67, 2048, True, "fp8_current"),
    ("mxfp8", 96, None, True, "mxfp8"),
    ("mxfp8", 96, None, False, "mxfp8"),
    ("mxfp8", 64, 512, True, "mxfp8"),
    # rows of whole 128-byte column blocks take the box kernel (bf16 H a
    # multiple of 64, every fp32 row); other bf16 widths the ring kernel
    ("mxfp8", 160, 256, False, "mxfp8"),
    ("mxfp8", 96, 1024, True, "mxfp8"),
    ("mxfp8", 96, 1024, False, "mxfp8"),
    ("mxfp8", 64, 768, True, "mxfp8"),
    ("mxfp8", 64, 800, False, "mxfp8"),
    ("mxfp8", 32, 3072, True, "mxfp8"),
    ("mxfp8", 64, 4096, True, "mxfp8"),
    ("mxfp8", 32, 4096, False, "mxfp8"),
    # wide rows, both directions (the box kernel holds no whole tile)
    ("mxfp8", 32, 8192, True, "mxfp8"),
    ("mxfp8", 64, 8192, True, "mxfp8"),
    ("mxfp8", 32, 8192, False, "mxfp8"),
    ("mxfp8", 32, 16384, True, "mxfp8"),
    ("mxfp8", 96, 2112, True, "mxfp8"),     # a last box of one column block
    ("bwd_f32", 64, 2048, True, "mxfp8"),
    ("bwd_f32", 32, 4096, False, "mxfp8"),
    ("bwd_f32", 64, 1056, True, "mxfp8"),   # fp32: a last sub-tile of 32 columns
    ("bwd_f32", 67, 1024, True, "none"),
    ("bwd_f32", 67, 1024, False, "fp8_delayed"),
    ("bwd_f32", 64, 1024, True, "mxfp8"),
    ("ln_delayed", 9, 16384, True, "fp8_delayed"),
    ("rms_small", 1, 8, False, "none"),
    ("rms_small", 3, 8, True, "fp8_current"),
    # rows of < 8 KB with many rows go several to a ring slot (one copy):
    # 4 KB rows two a slot, 2 KB four, 1 KB eight; N leaves a short last group
    ("ln_delayed", 1301, 2048, True, "fp8_delayed"),
    ("ln_delayed", 1301, 2048, True, "none"),
    ("rms_current", 2437, 1024, False, "fp8_current"),
    ("rms_current", 2437, 1024, True, "fp8_current"),
    ("bwd_f32", 4900, 256, True, "fp8_delayed"),
    ("bwd_f32", 4900, 256, False, "none"),
]


@pytest.mark.parametrize("case", FWD_CASES, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}-{'ln' if c[3] else 'rms'}-{c[4]}")
def test_fused_forward_parity(case):
    name, N, H, ln, mode = case
    w = rn_inputs.make(name, N=N, H=H)
    if mode == "fp8_delayed" and w.scale is None:
        w.scale = float(np.float32(448.0) / np.float32(4.0))
    if ln and w.beta is None:
        w.beta = (np.random.default_rng(1).normal(0, 0.1, w.H)).astype(np.float32)
    out, mu, rs = _run_fwd(w, ln, mode)
    ref = _oracle_fwd(w, ln, mode)
    check_stats(mu, rs, w.x_f64(), ref.get("mu"), ref["rsigma"])
    wt = _terms(w, ref, ln)
    y32 = ref["y"].astype(np.float32)
    if mode == "none":
        if w.dtype == "bf16":
            check_bf16(bf16_bits(out), ref["y"], wt)
        else:
            got = out.cpu().numpy().astype(np.float64)
            assert np.all(np.abs(got - ref["y"]) <= 2.0 ** -20 * wt)
    elif mode in ("fp8_delayed", "fp8_current"):
        amax = float(out.amax.item())
        assert abs(amax - float(ref["amax"])) <= 1e-6 * wt.max()
        s_ref = np.float32(ref["scale"]) if mode == "fp8_current" else np.float32(w.scale)
        s_gpu = np.float32(out.scale.item())
        if mode == "fp8_current":
            assert s_gpu == np.float32(448.0) / np.float32(amax)      # IEEE division
            assert abs(float(s_gpu) - float(s_ref)) <= 1e-5 * float(s_ref)
        assert np.float32(out.scale_inv.item()) == np.float32(1.0) / s_gpu
        p = (y32 * s_ref).astype(np.float64)
        win = 1e-6 * float(s_ref) * wt + np.abs(p) * abs(float(s_gpu) / float(s_ref) - 1.0)
        check_fp8_codes(out.data.cpu().numpy(), ref["data"], p, win, mode)
    else:
        check_mx(out.data.cpu().numpy(), out.row_scales.cpu().numpy(), y32, wt, "mx-row")
        check_mx(out.col_data.cpu().numpy(), out.col_scales.cpu().numpy(),
                 np.ascontiguousarray(y32.T), np.ascontiguousarray(wt.T), "mx-col")


def test_forward_out_f32_is_y32():
    w = rn_inputs.make("ln_delayed", N=40, H=512)
    out, mu, rs = _run_fwd(w, True, "none", out_dtype=torch.float32)
    ref = _oracle_fwd(w, True, "none")
    wt = _terms(w, ref, True)
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref["y"]) <= 2.0 ** -20 * wt)


def test_forward_sm_margin_and_repeat_bit_identical():
    w = rn_inputs.make("ln_delayed", N=333, H=4096)
    a = _run_fwd(w, True, "fp8_delayed", sm_margin=0)
    b = _run_fwd(w, True, "fp8_delayed", sm_margin=16)
    c = _run_fwd(w, True, "fp8_delayed", sm_margin=0)
    for o in (b, c):
        assert torch.equal(a[0].data, o[0].data) and torch.equal(a[0].amax, o[0].amax)
        assert np.array_equal(a[1], o[1]) and np.array_equal(a[2], o[2])


@pytest.mark.parametrize("H", [256, 2048])
def test_mxfp8_columnwise_only_and_margin(H):
    """Columnwise-only MXFP8 equals the columnwise half of the two-direction
    call (the same kernel) for any sm_margin."""
    w = rn_inputs.make("mxfp8", N=192, H=H)
    both = _run_fwd(w, True, "mxfp8")
    col = _run_fwd(w, True, "mxfp8", sm_margin=100, rowwise=False)
    assert col[0].data is None
    assert torch.equal(both[0].col_data, col[0].col_data)
    assert torch.equal(both[0].col_scales, col[0].col_scales)
    assert np.array_equal(both[1], col[1]) and np.array_equal(both[2], col[2])


ROW_ONLY = [
    # (workload, N, H, ln, sm_margin): rowwise-only MXFP8 takes the one-pass row kernel
    ("mxfp8", 192, 2048, True, 0),
    ("mxfp8", 96, 256, False, 5),
    ("mxfp8", 64, 800, True, 0),       # lanes with a ragged share of the row
    ("mxfp8", 32, 8192, True, 0),      # four warps a row
    ("bwd_f32", 64, 1024, True, 0),    # fp32: a block spans 8 lanes
    ("bwd_f32", 32, 96, False, 0),
    ("mxfp8", 1312, 2048, True, 0),    # two rows a ring slot
    ("mxfp8", 4896, 512, False, 0),    # eight rows a ring slot
]


@pytest.mark.parametrize("case", ROW_ONLY, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}-{'ln' if c[3] else 'rms'}-m{c[4]}")
def test_mxfp8_rowwise_only(case):
    name, N, H, ln, margin = case
    w = rn_inputs.make(name, N=N, H=H)
    if ln and w.beta is None:
        w.beta = (np.random.default_rng(1).normal(0, 0.1, w.H)).astype(np.float32)
    out, mu, rs = _run_fwd(w, ln, "mxfp8", sm_margin=margin, colwise=False)
    assert out.col_data is None and out.col_scales is None
    ref = _oracle_fwd(w, ln, "none")
    check_stats(mu, rs, w.x_f64(), ref.get("mu"), ref["rsigma"])
    check_mx(out.data.cpu().numpy(), out.row_scales.cpu().numpy(), ref["y"].astype(np.float32),
             _terms(w, ref, ln), "mx-row-only")


def test_forward_empty():
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(256, device="cuda")
    out, rs = rn.rmsnorm_fwd(x, g, 1e-6)
    assert out.shape == (0, 256)
    out, rs = rn.rmsnorm_fwd(x, g, 1e-6, quant="fp8_current")
    assert out.amax.item() == 0 and out.scale.item() == 1.0


# --------------------------------------------------------------- backward
BWD_CASES = [
    ("rms_small", None, None, False),
    ("ln_delayed", 75, None, True),
    ("bwd_f32", 203, None, True),
    ("bwd_f32", 203, None, False),
    ("bwd_bf16", 45, None, True),
    ("bwd_bf16", 45, None, False),
    ("bwd_bf16", 1, 5120, True),
    ("bwd_f32", 3, 8, True),
    # the wide stats-warp kernel in both of its builds: 512 threads (2 and 4
    # chunks a thread) and 576 threads (4 chunks a thread; 14336 and 16384,
    # the widest bf16 row)
    ("bwd_bf16", 24, 8192, True),
    ("bwd_bf16", 16, 10240, False),
    ("bwd_bf16", 8, 14336, True),
    ("bwd_bf16", 8, 16384, False),
    ("bwd_f32", 5, 8192, True),
]


def _run_bwd(w, ln, mu, rs, sm_margin=0):
    x = to_dev(w.x, w.dtype)
    dz = to_dev(w.dz, w.dtype)
    g = to_dev(w.gamma, "f32")
    rsd = torch.from_numpy(rs).cuda()
    if ln:
        return rn.layernorm_bwd(dz, x, torch.from_numpy(mu).cuda(), rsd, g, sm_margin,
                                w.zero_centered_gamma)
    return rn.rmsnorm_bwd(dz, x, rsd, g, sm_margin, w.zero_centered_gamma)


def _bwd_reference(w, ln):
    """Oracle backward fed with the oracle forward's fp32 mu / rsigma."""
    x = w.x_f64()
    if ln:
        f = oracle.layernorm_fwd(x, w.gamma, w.beta, w.eps, w.zero_centered_gamma, "none")
        b = oracle.layernorm_bwd(w.dz_f64(), x, f["mu"], f["rsigma"], w.gamma,
                                 w.zero_centered_gamma, w.dtype)
        return f["mu"], f["rsigma"], b
    f = oracle.rmsnorm_fwd(x, w.gamma, w.eps, w.zero_centered_gamma, "none")
    b = oracle.rmsnorm_bwd(w.dz_f64(), x, f["rsigma"], w.gamma, w.zero_centered_gamma, w.dtype)
    return None, f["rsigma"], b


def check_bwd(w, ln, got, mu, rs, ref):
    dx = got[0]
    dx64 = ref["dx64"]
    rms = np.sqrt(np.mean(dx64 ** 2, axis=1, keepdims=True))
    if w.dtype == "bf16":
        g = (bf16_bits(dx).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        r = oracle.round_to_bf16(dx64)
        from parity import bf16_ulp
        err = np.abs(g - r)
        assert np.all((err <= bf16_ulp(r)) | (err <= 2e-3 * rms)), f"dx max err {err.max()}"
        g_f = g
    else:
        g_f = dx.cpu().numpy().astype(np.float64)
        err = np.abs(g_f - dx64)
        assert np.all(err <= 2e-3 * np.maximum(np.abs(dx64), rms)), f"dx max err {err.max()}"
    rowrel = np.linalg.norm(g_f - dx64, axis=1) / np.maximum(np.linalg.norm(dx64, axis=1), 1e-300)
    assert np.all(rowrel <= 2e-3), rowrel.max()
    x = w.x_f64()
    xhat = ((x - mu[:, None]) if ln else x) * rs.astype(np.float64)[:, None]
    dz = w.dz_f64()
    denom = np.sum(np.abs(dz * xhat), axis=0)
    dg = got[1].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(dg - ref["dgamma64"]) <= 1e-3 * denom + 1e-30), "dgamma"
    if ln:
        db = got[2].cpu().numpy().astype(np.float64)
        assert np.all(np.abs(db - ref["dbeta64"]) <= 1e-3 * np.sum(np.abs(dz), axis=0) + 1e-30), "dbeta"


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}-{'ln' if c[3] else 'rms'}")
def test_backward_parity(case):
    name, N, H, ln = case
    w = rn_inputs.make(name, N=N, H=H)
    if ln and w.beta is None:
        w.beta = np.zeros(w.H, np.float32)
    mu, rs, ref = _bwd_reference(w, ln)
    got = _run_bwd(w, ln, mu, rs)
    check_bwd(w, ln, got, mu, rs, ref)


@pytest.mark.parametrize("ln", [True, False])
def test_backward_deterministic_across_sm_margin(ln):
    w = rn_inputs.make("bwd_bf16", N=1500, H=5120)
    x = w.x_f64()
    if ln:
        m, r = oracle.layernorm_stats(x, w.eps)
        mu, rs = m.astype(np.float32), r.astype(np.float32)
    else:
        mu, rs = None, oracle.rmsnorm_stats(x, w.eps).astype(np.float32)
    a = _run_bwd(w, ln, mu, rs, sm_margin=0)
    b = _run_bwd(w, ln, mu, rs, sm_margin=16)
    c = _run_bwd(w, ln, mu, rs, sm_margin=0)
    for o in (b, c):
        for t0, t1 in zip(a, o):
            assert torch.equal(t0, t1)


def test_backward_empty():
    x = torch.empty((0, 64), dtype=torch.float32, device="cuda")
    g = torch.ones(64, device="cuda")
    e = torch.empty(0, device="cuda")
    dx, dg, db = rn.layernorm_bwd(x, x, e, e, g)
    assert dx.shape == (0, 64) and float(dg.abs().sum()) == 0 and float(db.abs().sum()) == 0


def test_backward_workspace_too_small():
    w = rn_inputs.make("bwd_f32", N=64, H=256)
    x = to_dev(w.x, "f32")
    rs = torch.ones(64, device="cuda")
    g = torch.ones(256, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(rn.RNError, match="status 3"):
        rn.rmsnorm_bwd(x, x, rs, g, workspace=ws)


@pytest.mark.parametrize("dtype,H,ln,ok", [
    (torch.bfloat16, 41216, True, True), (torch.bfloat16, 41280, True, False),
    (torch.float32, 20608, False, True), (torch.float32, 20640, False, False),
    (torch.bfloat16, 3104, True, True), (torch.bfloat16, 3168, True, False),
    (torch.bfloat16, 3296, False, True), (torch.bfloat16, 3360, False, False),
])
def test_mxfp8_two_direction_width_limits(dtype, H, ln, ok):
    """The two-direction MXFP8 width limits the header states: the widest
    accepted row runs, the next width is refused on the host."""
    x = torch.randn((32, H), device="cuda").to(dtype)
    g = torch.ones(H, device="cuda")
    run = (lambda: rn.layernorm_fwd(x, g, None, 1e-5, quant="mxfp8")) if ln else \
        (lambda: rn.rmsnorm_fwd(x, g, 1e-5, quant="mxfp8"))
    if ok:
        out = run()[0]
        assert out.col_data.shape == (H, 32)
    else:
        with pytest.raises(rn.RNError, match="status 2"):
            run()
