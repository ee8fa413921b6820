"""GPU parity of the delayed-scaling history step (rn_delayed_scaling_update)
against the oracle, bit for bit, and the loop it closes around the FP8
delayed-scaling forward."""
import numpy as np
import pytest
import torch

import mxfp8_quantization_gb300 as rn
import oracle
import rn_inputs

pytestmark = pytest.mark.gpu


def _step(hist, amax, scale):
    h = torch.from_numpy(np.asarray(hist, dtype=np.float32).copy()).cuda()
    a = torch.tensor([amax], dtype=torch.float32, device="cuda")
    s = torch.tensor([scale], dtype=torch.float32, device="cuda")
    si = rn.delayed_scaling_update(h, a, s)
    return h.cpu().numpy(), np.float32(s.item()), np.float32(si.item())


def _same(a, b):
    a, b = np.asarray(a, dtype=np.float32), np.asarray(b, dtype=np.float32)
    return np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("L", [1, 2, 16, 100, 1024])
def test_history_step_bit_exact(L):
    rng = np.random.default_rng(L)
    for k in range(4):
        hist = rng.uniform(0.0, 10.0, L).astype(np.float32)
        amax = np.float32(rng.uniform(0.0, 20.0))
        scale = np.float32(rng.uniform(1.0, 100.0))
        got = _step(hist, amax, scale)
        want = oracle.amax_history_update(hist, amax, scale)
        assert _same(got[0], want[0]) and _same(got[1], want[1]) and _same(got[2], want[2])


@pytest.mark.parametrize("hist,amax", [([0.0, 0.0, 0.0], 0.0), ([np.inf, 1.0], 2.0),
                                       ([1.0, 2.0], np.nan), ([1.0, np.inf], 4.0),
                                       ([-1.0, -2.0], -0.5)])
def test_history_step_special_values(hist, amax):
    got = _step(hist, amax, 12.5)
    want = oracle.amax_history_update(hist, amax, 12.5)
    assert _same(got[0], want[0]) and _same(got[1], want[1]) and _same(got[2], want[2])


def test_history_step_closes_the_delayed_scaling_loop():
    w = rn_inputs.make("ln_delayed", N=96, H=1024)
    x = torch.from_numpy(w.x.view(np.int16)).view(torch.bfloat16).cuda()
    g = torch.from_numpy(w.gamma).cuda()
    b = torch.from_numpy(w.beta).cuda()
    hist = torch.from_numpy(w.amax_history.copy()).cuda()
    scale = torch.tensor([w.scale], dtype=torch.float32, device="cuda")
    h_ref, s_ref = w.amax_history.copy(), np.float32(w.scale)
    for _ in range(3):
        out, mu, rs = rn.layernorm_fwd(x, g, b, w.eps, quant="fp8_delayed", scale=scale,
                                       zero_centered_gamma=True)
        rn.delayed_scaling_update(hist, out.amax, scale)
        h_ref, s_ref, _ = oracle.amax_history_update(h_ref, np.float32(out.amax.item()), s_ref)
        assert _same(hist.cpu().numpy(), h_ref) and _same(scale.cpu().numpy()[0], s_ref)
    assert rn.device_error() == 0
