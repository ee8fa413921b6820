"""rn_layernorm_bwd_noalloc: the LayerNorm backward for callers that cannot
allocate device memory where they run it.  It keeps its dgamma/dbeta partial
sums in the library's fixed per-device scratch array instead of a workspace.

Called here through the C ABI (ctypes, raw device pointers) and compared with
the regular rn_layernorm_bwd on the same inputs, on two calls in a row with
different shapes, so that whatever the first call left in the shared array
cannot leak into the second.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import mxfp8_quantization_gb300 as rn
import oracle
import rn_inputs

pytestmark = pytest.mark.gpu


def _dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _case(N, H, seed):
    w = rn_inputs.make("bwd_bf16", N=N, H=H, seed=seed)
    m, r = oracle.layernorm_stats(w.x_f64(), w.eps)
    return (_dev_bf16(w.x), _dev_bf16(w.dz), torch.from_numpy(w.gamma).cuda(),
            torch.from_numpy(m.astype(np.float32)).cuda(), torch.from_numpy(r.astype(np.float32)).cuda())


def _noalloc(lib, x, dz, g, mu, rs):
    N, H = x.shape
    dx = torch.empty_like(x)
    dg = torch.empty(H, dtype=torch.float32, device="cuda")
    db = torch.empty(H, dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.rn_layernorm_bwd_noalloc(p(dz), p(x), 0, p(mu), p(rs), p(g), N, H, 0, 0, p(dx), p(dg),
                                      p(db), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.rn_status_str(st)
    return dx, dg, db


def _bf16_to_f64(t):
    return (t.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32) << 16
            ).view(np.float32).astype(np.float64)


def test_noalloc_backward_matches_regular_on_two_calls():
    lib = rn._load()
    for N, H, seed in ((1000, 2048, 5), (3000, 5120, 6)):
        x, dz, g, mu, rs = _case(N, H, seed)
        ref = rn.layernorm_bwd(dz, x, mu, rs, g)
        got = _noalloc(lib, x, dz, g, mu, rs)
        torch.cuda.synchronize()
        # the parity tests' tolerances: dx within one bf16 ulp, dgamma and
        # dbeta within 1e-3 of the summed magnitudes of their terms
        a, b = _bf16_to_f64(got[0]), _bf16_to_f64(ref[0])
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(b), 2.0 ** -126))) - 7)
        assert np.all(np.abs(a - b) <= ulp)
        xh = (x.float() - mu[:, None]) * rs[:, None]
        den_g = (dz.float() * xh).abs().sum(0).cpu().numpy().astype(np.float64)
        den_b = dz.float().abs().sum(0).cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got[1].cpu().numpy() - ref[1].cpu().numpy()) <= 1e-3 * den_g)
        assert np.all(np.abs(got[2].cpu().numpy() - ref[2].cpu().numpy()) <= 1e-3 * den_b)
    assert rn.device_error() == 0


def test_noalloc_backward_rejects_problems_beyond_its_scratch():
    lib = rn._load()
    x = torch.zeros((8192, 4096), dtype=torch.bfloat16, device="cuda")   # partials need 32 MiB
    g = torch.ones(4096, device="cuda")
    v = torch.ones(8192, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.rn_layernorm_bwd_noalloc(p(x), p(x), 0, p(v), p(v), p(g), 8192, 4096, 0, 0, p(x), p(g),
                                      p(g), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 3                                       # RN_ERR_WORKSPACE, nothing enqueued
