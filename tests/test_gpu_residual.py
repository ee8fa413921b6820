"""GPU parity of the residual add + norm forward (rn_rmsnorm_add_fwd,
rn_layernorm_add_fwd) against the oracle: h = x + residual rounded once to
the stream dtype is compared bit for bit, the outputs of the norm of h with
the tolerances of the plain forward."""
import numpy as np
import pytest
import torch

import mxfp8_quantization_gb300 as rn
import oracle
import rn_inputs
from parity import check_bf16, check_fp8_codes, check_mx, check_stats, term_magnitude

pytestmark = pytest.mark.gpu


def to_dev(a, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.fixture(autouse=True)
def _no_device_error():
    yield
    assert rn.device_error() == 0


def _workload(name, N, H):
    w = rn_inputs.make(name, N=N, H=H)
    if w.residual is None:           # fp32 cases: the workload's dz as the residual
        w.residual = w.dz
    if w.scale is None:
        w.scale = float(np.float32(448.0) / np.float32(8.0))
    return w


def _run(w, ln, mode, sm_margin=0, rowwise=True, colwise=True):
    x, r, g = to_dev(w.x, w.dtype), to_dev(w.residual, w.dtype), to_dev(w.gamma, "f32")
    kw = dict(quant=mode, sm_margin=sm_margin, scale=w.scale if mode == "fp8_delayed" else None,
              rowwise=rowwise, colwise=colwise)
    if ln:
        out, h, mu, rs = rn.layernorm_add_fwd(x, r, g, to_dev(w.beta, "f32"), w.eps, **kw)
        return out, h, mu.cpu().numpy(), rs.cpu().numpy()
    out, h, rs = rn.rmsnorm_add_fwd(x, r, g, w.eps, **kw)
    return out, h, None, rs.cpu().numpy()


def _oracle(w, ln, mode):
    x, r = w.x_f64(), w.residual_f64()
    if ln:
        return oracle.layernorm_add_fwd(x, r, w.gamma, w.beta, w.eps, w.dtype, mode=mode,
                                        scale=w.scale)
    return oracle.rmsnorm_add_fwd(x, r, w.gamma, w.eps, w.dtype, mode=mode, scale=w.scale)


CASES = [
    # (workload, N, H, ln, mode)
    ("rms_add", 75, 4096, False, "fp8_delayed"),
    ("rms_add", 75, 4096, True, "none"),
    ("rms_add", 45, 1000, True, "fp8_current"),
    ("rms_add", 203, 1024, False, "fp8_current"),
    ("rms_add", 9, 16384, False, "fp8_delayed"),
    ("rms_add", 3, 8, True, "none"),
    ("bwd_f32", 67, 1024, False, "none"),
    ("bwd_f32", 67, 1024, True, "fp8_delayed"),
    ("rms_add", 96, 4096, True, "mxfp8"),
    ("rms_add", 64, 2048, False, "mxfp8"),
    ("bwd_f32", 64, 1024, True, "mxfp8"),
    # rows of 4 / 2 KB go two / four to a ring slot (x and residual rows);
    # N leaves a short last group
    ("rms_add", 1301, 2048, False, "fp8_delayed"),
    ("rms_add", 2437, 1024, True, "fp8_current"),
    ("rms_add", 1312, 2048, True, "mxfp8"),
]


def _check(w, ln, mode, got, ref):
    out, h, mu, rs = got
    if w.dtype == "bf16":
        assert np.array_equal(bits(h), ref["residual_out"]), "residual_out differs"
    else:
        assert np.array_equal(h.cpu().numpy(), ref["residual_out"]), "residual_out differs"
    hf = ref["h"]
    check_stats(mu, rs, hf, ref.get("mu"), ref["rsigma"])
    wt = term_magnitude(hf, ref.get("mu") if ln else None, ref["rsigma"], w.gamma,
                        w.beta if ln else None, False)
    if mode == "mxfp8":
        y32 = ref["y"].astype(np.float32)
        if out.data is not None:
            check_mx(out.data.cpu().numpy(), out.row_scales.cpu().numpy(), y32, wt, "residual mx-row")
        if out.col_data is not None:
            # the columnwise copy holds the blocks of y transposed: the
            # rowwise blocks of y.T
            check_mx(out.col_data.cpu().numpy(), out.col_scales.cpu().numpy(),
                     np.ascontiguousarray(y32.T), np.ascontiguousarray(wt.T), "residual mx-col")
        return
    if mode == "none":
        if w.dtype == "bf16":
            check_bf16(bits(out), ref["y"], wt)
        else:
            assert np.all(np.abs(out.cpu().numpy().astype(np.float64) - ref["y"]) <= 2.0 ** -20 * wt)
        return
    amax = float(out.amax.item())
    assert abs(amax - float(ref["amax"])) <= 1e-6 * wt.max()
    s_ref = np.float32(ref["scale"]) if mode == "fp8_current" else np.float32(w.scale)
    s_gpu = np.float32(out.scale.item())
    p = (ref["y"].astype(np.float32) * s_ref).astype(np.float64)
    win = 1e-6 * float(s_ref) * wt + np.abs(p) * abs(float(s_gpu) / float(s_ref) - 1.0)
    check_fp8_codes(out.data.cpu().numpy(), ref["data"], p, win, mode)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}-{'ln' if c[3] else 'rms'}-{c[4]}")
def test_residual_add_forward_parity(case):
    name, N, H, ln, mode = case
    w = _workload(name, N, H)
    _check(w, ln, mode, _run(w, ln, mode), _oracle(w, ln, mode))


def test_residual_add_full_size_and_margin():
    w = _workload("rms_add", None, None)
    a = _run(w, False, "fp8_delayed")
    _check(w, False, "fp8_delayed", a, _oracle(w, False, "fp8_delayed"))
    b = _run(w, False, "fp8_delayed", sm_margin=16)
    assert torch.equal(a[0].data, b[0].data) and torch.equal(a[1], b[1])
    assert np.array_equal(a[3], b[3]) and torch.equal(a[0].amax, b[0].amax)


MX_DIRECTIONS = [
    # (workload, N, H, ln, rowwise, colwise): the box kernel (bf16 H % 64 == 0,
    # fp32), the ring kernel (bf16 H % 64 == 32), each direction alone
    ("rms_add", 96, 2048, True, False, True),
    ("rms_add", 64, 2080, False, True, True),
    ("rms_add", 128, 1024, True, True, False),
    ("bwd_f32", 64, 1056, False, False, True),
]


@pytest.mark.parametrize("case", MX_DIRECTIONS,
                         ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}-{'ln' if c[3] else 'rms'}-r{int(c[4])}c{int(c[5])}")
def test_residual_add_mxfp8_directions(case):
    """MXFP8 after the residual add, each block direction alone and both: the
    stored sum, the statistics and the requested blocks against the oracle;
    the blocks not asked for are not allocated."""
    name, N, H, ln, rowwise, colwise = case
    w = _workload(name, N, H)
    got = _run(w, ln, "mxfp8", rowwise=rowwise, colwise=colwise)
    out = got[0]
    assert (out.data is not None) == rowwise and (out.col_data is not None) == colwise
    _check(w, ln, "mxfp8", got, _oracle(w, ln, "mxfp8"))


def test_residual_add_mxfp8_full_size_and_margin():
    """Both directions after the residual add at 65536 x 2048 (the MXFP8
    workload's shape, the residual drawn as in the residual-add workload):
    the result does not depend on sm_margin, and matches the plain forward of
    the stored sum."""
    w = _workload("rms_add", 65536, 2048)
    x, r, g = to_dev(w.x, "bf16"), to_dev(w.residual, "bf16"), to_dev(w.gamma, "f32")
    a, h, rs = rn.rmsnorm_add_fwd(x, r, g, w.eps, quant="mxfp8")
    b, h2, rs2 = rn.rmsnorm_add_fwd(x, r, g, w.eps, quant="mxfp8", sm_margin=16)
    assert torch.equal(h, h2) and torch.equal(rs, rs2)
    assert torch.equal(a.data, b.data) and torch.equal(a.row_scales, b.row_scales)
    assert torch.equal(a.col_data, b.col_data) and torch.equal(a.col_scales, b.col_scales)
    # the rowwise blocks are the row kernel's, the columnwise ones (and the
    # last rsigma written) the two-direction kernel's, each on the stored sum
    row, _ = rn.rmsnorm_fwd(h, g, w.eps, quant="mxfp8", colwise=False)
    col, rs3 = rn.rmsnorm_fwd(h, g, w.eps, quant="mxfp8", rowwise=False)
    assert torch.equal(a.data, row.data) and torch.equal(a.row_scales, row.row_scales)
    assert torch.equal(a.col_data, col.col_data) and torch.equal(a.col_scales, col.col_scales)
    assert torch.equal(rs, rs3)
