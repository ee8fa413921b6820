"""GPU parity of the NVFP4 output path (norm + amax, then quantize to E2M1
with an E4M3 scale per 16 elements and the tensor scale S = 448*6/amax)
against the oracle, through the C ABI.

* rn_quantize_only on caller-given fp32 values: bit for bit (codes, block
  scales, amax, S, 1/S), on tensors that run every E2M1 rounding class with
  an exact element factor, E4M3 block-scale rounding classes, a wide dynamic
  range (block scales that underflow to E4M3 subnormals and zero), ragged
  row counts and the degenerate tensors (all zero, tiny amax);
* the fused forward (LayerNorm / RMSNorm, bf16 / fp32 input, rows from one
  block to 16384 elements, zero-centred gamma, sm_margin, residual add)
  with the tolerances of ``parity.check_nvfp4``.
"""
import numpy as np
import pytest
import torch

import mxfp8_quantization_gb300 as rn
import oracle
import rn_inputs
from parity import check_nvfp4, check_stats, term_magnitude
from test_gpu_parity import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _no_device_error():
    yield
    assert rn.device_error() == 0


def _assert_exact(r, ref):
    assert np.array_equal(r.row_scales.cpu().numpy(), ref["row_scales"]), "block scales differ"
    got, want = r.data.cpu().numpy(), ref["data"]
    bad = got != want
    assert not bad.any(), (f"{bad.sum()} code bytes differ, e.g. gpu={got[bad][:6]} "
                           f"ref={want[bad][:6]}")
    assert np.float32(r.amax.item()) == ref["amax"]
    assert np.float32(r.scale.item()) == ref["scale"]
    assert np.float32(r.scale_inv.item()) == ref["scale_inv"]


def _e2m1_class_tensor():
    """Row 0 holds the tensor amax 1.75 (S = 1536, S/6 = 256).  Every other
    block has its maximum 3/256, so A * S/6 = 3 (an E4M3 value) and the
    element factor is S/3 = 512, a power of two: y * 512 = p exactly, and
    the p values run through every E2M1 value, midpoint (tie) and their
    fp32 neighbours, with both signs."""
    mags = oracle.e2m1_magnitudes()
    mids = (mags[:-1] + mags[1:]) / 2
    rng = np.random.default_rng(40)
    p = np.concatenate([mags, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                        np.nextafter(mids.astype(np.float32), np.float32(7)),
                        np.nextafter(mags[1:].astype(np.float32), np.float32(0)),
                        np.nextafter(mags[:-1].astype(np.float32), np.float32(7)),
                        rng.uniform(0, 6, 400).astype(np.float32)]).astype(np.float32)
    p = np.concatenate([p, -p])
    per = 15
    nblk = -(-p.size // per)
    p = np.concatenate([p, np.zeros(nblk * per - p.size, np.float32)]).reshape(nblk, per)
    blocks = np.concatenate([np.full((nblk, 1), 6.0, np.float32), p], axis=1)   # max |p| = 6
    H = 256
    nb = H // 16
    rows = -(-nblk // nb)
    blocks = np.concatenate([blocks, np.zeros((rows * nb - nblk, 16), np.float32)])
    y = (blocks / np.float32(512.0)).astype(np.float32).reshape(rows, H)
    top = np.zeros((1, H), np.float32)
    top[0, 5] = 1.75
    return np.concatenate([top, y])


def _scale_class_tensor():
    """Block maxima a / 256 with a sweeping E4M3 rounding classes (each
    binade from 2**-12 to 2**8: the 3-bit mantissa grid, its midpoints and
    their fp32 neighbours), so that A * S/6 = a exactly; the other elements
    of a block are random below its maximum."""
    rng = np.random.default_rng(41)
    a = []
    for e in range(-12, 9):
        for m in range(16):
            base = np.float32((1.0 + m / 16.0) * 2.0 ** e)
            a += [base, np.nextafter(base, np.float32(0)), np.nextafter(base, np.float32(1e9))]
    a = np.array([t for t in a if t <= 448.0], np.float32)
    A = (a / np.float32(256.0)).astype(np.float32)
    blocks = rng.uniform(-1, 1, (A.size, 16)).astype(np.float32) * A[:, None]
    blocks[:, 3] = A * np.where(rng.random(A.size) < 0.5, -1, 1)
    H = 512
    nb = H // 16
    rows = -(-A.size // nb)
    blocks = np.concatenate([blocks, np.zeros((rows * nb - A.size, 16), np.float32)])
    y = blocks.reshape(rows, H)
    y[0, 0] = 1.75                       # the tensor amax (A * S/6 = 448 there)
    return y


@pytest.mark.parametrize("make", [_e2m1_class_tensor, _scale_class_tensor],
                         ids=["e2m1_classes", "e4m3_scale_classes"])
def test_quantize_only_nvfp4_rounding_classes(make):
    y = make()
    r = rn.quantize_only(to_dev(y, "f32"), "nvfp4")
    _assert_exact(r, oracle.quantize(y, "nvfp4"))


@pytest.mark.parametrize("shape", [(517, 1024), (3, 16), (64, 48), (129, 4112)])
def test_quantize_only_nvfp4_wide_range(shape):
    N, H = shape
    rng = np.random.default_rng(42 + N)
    y = (rng.standard_normal((N, H)) * np.exp2(rng.uniform(-20, 20, (N, 1)))).astype(np.float32)
    r = rn.quantize_only(to_dev(y, "f32"), "nvfp4")
    ref = oracle.quantize(y, "nvfp4")
    _assert_exact(r, ref)
    # most rows sit far below the tensor amax: their blocks underflow to
    # E4M3 subnormal or zero scales, which this case must reach
    sc = ref["row_scales"]
    if N >= 64:
        assert (sc == 0).any() and ((sc > 0) & (sc < 8)).any()


def test_quantize_only_nvfp4_degenerate():
    r = rn.quantize_only(torch.zeros((32, 64), dtype=torch.float32, device="cuda"), "nvfp4")
    assert r.amax.item() == 0 and r.scale.item() == 1.0 and r.scale_inv.item() == 1.0
    assert int(r.data.max()) == 0 and int(r.row_scales.max()) == 0
    y = np.zeros((2, 32), np.float32)
    y[1, 17] = np.float32(2.0 ** -140)
    y[0, 2] = -np.float32(2.0 ** -142)
    r = rn.quantize_only(to_dev(y, "f32"), "nvfp4")
    _assert_exact(r, oracle.quantize(y, "nvfp4"))
    # N == 0: only the scalars
    r = rn.quantize_only(torch.empty((0, 64), dtype=torch.float32, device="cuda"), "nvfp4")
    assert r.amax.item() == 0 and r.scale.item() == 1.0


# ------------------------------------------------------------ fused forward
FWD = [
    # (workload, N, H, ln, sm_margin)
    ("rms_current", 203, 1024, False, 0),
    ("rms_current", 67, 2064, True, 0),      # lanes hold a ragged share of the row
    ("rms_current", 45, 1008, False, 3),     # short rows (4 chunks a lane), sm_margin
    ("ln_delayed", 75, 4096, True, 0),       # zero-centred gamma
    ("ln_delayed", 9, 16384, True, 0),       # four warps a row
    ("bwd_f32", 67, 1024, True, 0),          # fp32 input: a block spans four lanes
    ("bwd_f32", 33, 8192, False, 0),
    ("rms_small", 3, 16, False, 0),          # one block a row
    ("rms_current", 2437, 1024, False, 0),   # four rows a ring slot, short last group
    ("ln_delayed", 1301, 2048, True, 0),     # two rows a ring slot
]


def _terms(w, ref, ln, x64):
    return term_magnitude(x64, ref.get("mu") if ln else None, ref["rsigma"], w.gamma,
                          w.beta if ln else None, w.zero_centered_gamma)


@pytest.mark.parametrize("case", FWD, ids=lambda c: f"{c[0]}-{c[1]}x{c[2]}-{'ln' if c[3] else 'rms'}-m{c[4]}")
def test_fused_forward_nvfp4(case):
    name, N, H, ln, margin = case
    w = rn_inputs.make(name, N=N, H=H)
    if ln and w.beta is None:
        w.beta = (np.random.default_rng(1).normal(0, 0.1, w.H)).astype(np.float32)
    x, g = to_dev(w.x, w.dtype), to_dev(w.gamma, "f32")
    kw = dict(quant="nvfp4", sm_margin=margin, zero_centered_gamma=w.zero_centered_gamma)
    x64 = w.x_f64()
    if ln:
        out, mu, rs = rn.layernorm_fwd(x, g, to_dev(w.beta, "f32"), w.eps, **kw)
        ref = oracle.layernorm_fwd(x64, w.gamma, w.beta, w.eps, w.zero_centered_gamma, "nvfp4")
        check_stats(mu.cpu().numpy(), rs.cpu().numpy(), x64, ref["mu"], ref["rsigma"])
    else:
        out, rs = rn.rmsnorm_fwd(x, g, w.eps, **kw)
        ref = oracle.rmsnorm_fwd(x64, w.gamma, w.eps, w.zero_centered_gamma, "nvfp4")
        check_stats(None, rs.cpu().numpy(), x64, None, ref["rsigma"])
    wt = _terms(w, ref, ln, x64)
    am = np.float32(out.amax.item())
    assert abs(float(am) - float(ref["amax"])) <= 1e-6 * wt.max()
    S = np.float32(out.scale.item())
    assert S == np.float32(2688.0) / am                      # one IEEE division
    assert np.float32(out.scale_inv.item()) == np.float32(1.0) / S
    assert out.data.shape == (N, H // 2) and out.row_scales.shape == (N, H // 16)
    check_nvfp4(out.data.cpu().numpy(), out.row_scales.cpu().numpy(), ref["y"].astype(np.float32),
                wt, ref["scale"], S, name)


@pytest.mark.parametrize("ln", [False, True], ids=["rms", "ln"])
def test_residual_add_nvfp4(ln):
    w = rn_inputs.make("rms_add", N=75, H=4096)
    x, r, g = to_dev(w.x, "bf16"), to_dev(w.residual, "bf16"), to_dev(w.gamma, "f32")
    if ln:
        out, h, mu, rs = rn.layernorm_add_fwd(x, r, g, to_dev(w.beta, "f32"), w.eps, quant="nvfp4")
        ref = oracle.layernorm_add_fwd(w.x_f64(), w.residual_f64(), w.gamma, w.beta, w.eps, "bf16",
                                       mode="nvfp4")
    else:
        out, h, rs = rn.rmsnorm_add_fwd(x, r, g, w.eps, quant="nvfp4")
        ref = oracle.rmsnorm_add_fwd(w.x_f64(), w.residual_f64(), w.gamma, w.eps, "bf16",
                                     mode="nvfp4")
    assert np.array_equal(h.contiguous().view(torch.int16).cpu().numpy().view(np.uint16),
                          ref["residual_out"])
    hf = ref["h"]
    wt = term_magnitude(hf, ref.get("mu"), ref["rsigma"], w.gamma, w.beta if ln else None, False)
    am = np.float32(out.amax.item())
    assert abs(float(am) - float(ref["amax"])) <= 1e-6 * wt.max()
    check_nvfp4(out.data.cpu().numpy(), out.row_scales.cpu().numpy(), ref["y"].astype(np.float32),
                wt, ref["scale"], np.float32(out.scale.item()), "residual nvfp4")


def test_fused_nvfp4_empty():
    x = torch.empty((0, 1024), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(1024, dtype=torch.float32, device="cuda")
    out, rs = rn.rmsnorm_fwd(x, g, 1e-6, quant="nvfp4")
    assert out.amax.item() == 0 and out.scale.item() == 1.0 and rs.numel() == 0
