"""rn_layernorm_bwd_noalloc: the LayerNorm backward for callers that cannot
allocate device memory where they run it.  It keeps its dgamma/dbeta partial
sums in the library's fixed per-device scratch array instead of a workspace.

Called here through the C ABI (ctypes, raw device pointers) and compared with
the regular rn_layernorm_bwd on the same inputs: both run the same kernels
with the same chunking, so the results must be bit-identical.  Each call is
also checked against the fp64 oracle.  The calls run back to back on the
shared array, the largest problem first, so that a smaller call that read
partials past its own chunk count would pick up the larger call's leftovers
and fail.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import mxfp8_quantization_gb300 as rn
import oracle
import rn_inputs
from parity import bf16_ulp

pytestmark = pytest.mark.gpu


def _dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _case(N, H, seed, zcg):
    w = rn_inputs.make("bwd_bf16", N=N, H=H, seed=seed)
    x64, dz64 = w.x_f64(), w.dz_f64()
    m, r = oracle.layernorm_stats(x64, w.eps)
    mu, rs = m.astype(np.float32), r.astype(np.float32)
    ref = oracle.layernorm_bwd(dz64, x64, mu, rs, w.gamma, zcg, "bf16")
    xhat = (x64 - mu[:, None].astype(np.float64)) * rs[:, None].astype(np.float64)
    den = (np.sum(np.abs(dz64 * xhat), axis=0), np.sum(np.abs(dz64), axis=0))
    dev = (_dev_bf16(w.x), _dev_bf16(w.dz), torch.from_numpy(w.gamma).cuda(),
           torch.from_numpy(mu).cuda(), torch.from_numpy(rs).cuda())
    return dev, ref, den


def _noalloc(lib, x, dz, g, mu, rs, zcg, margin):
    N, H = x.shape
    dx = torch.empty_like(x)
    dg = torch.empty(H, dtype=torch.float32, device="cuda")
    db = torch.empty(H, dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.rn_layernorm_bwd_noalloc(p(dz), p(x), 0, p(mu), p(rs), p(g), N, H, zcg, margin, p(dx),
                                      p(dg), p(db),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.rn_status_str(st)
    return dx, dg, db


def _bf16_to_f64(t):
    return (t.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32) << 16
            ).view(np.float32).astype(np.float64)


def _check_oracle(got, ref, den):
    # the parity tolerances: dx within one bf16 ulp of the oracle's rounded
    # value (or 2e-3 of the row's rms), dgamma / dbeta within 1e-3 of the
    # summed magnitudes of their terms
    dx64 = ref["dx64"]
    r = oracle.round_to_bf16(dx64)
    rms = np.sqrt(np.mean(dx64 ** 2, axis=1, keepdims=True))
    err = np.abs(_bf16_to_f64(got[0]) - r)
    assert np.all((err <= bf16_ulp(r)) | (err <= 2e-3 * rms))
    assert np.all(np.abs(got[1].cpu().numpy() - ref["dgamma64"]) <= 1e-3 * den[0])
    assert np.all(np.abs(got[2].cpu().numpy() - ref["dbeta64"]) <= 1e-3 * den[1])


def test_noalloc_backward_matches_regular_on_calls_in_a_row():
    lib = rn._load()
    # largest first: 375 chunks of partials (15 MB of the 16 MiB), then 125,
    # then a zero-centered call with 16 SMs left free
    for N, H, seed, zcg, margin in ((3000, 5120, 6, 0, 0), (1000, 2048, 5, 0, 0),
                                    (1000, 2048, 7, 1, 16)):
        (x, dz, g, mu, rs), ref, den = _case(N, H, seed, bool(zcg))
        want = rn.layernorm_bwd(dz, x, mu, rs, g, margin, bool(zcg))
        got = _noalloc(lib, x, dz, g, mu, rs, zcg, margin)
        torch.cuda.synchronize()
        for a, b in zip(got, want):
            assert torch.equal(a, b)
        _check_oracle(got, ref, den)
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
