"""CPU-only checks of the C ABI: the library builds, loads and exports every
entry point include/rn.h declares, and the host-side argument checks answer
before any device work (no GPU is touched)."""
import ctypes
import os
import re

import pytest

import mxfp8_quantization_gb300 as rn
from mxfp8_quantization_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rn.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return rn._load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(rn_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for f in ("rn_layernorm_fwd", "rn_rmsnorm_fwd", "rn_layernorm_bwd", "rn_rmsnorm_bwd",
              "rn_quantize_only", "rn_status_str", "rn_device_error", "rn_abi_version"):
        assert f in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_only_api_symbols_are_exported(lib):
    out = os.popen(f"nm -D --defined-only {rn.lib_path()}").read().split("\n")
    syms = [l.split()[-1] for l in out if l.strip()]
    assert syms and all(s.startswith("rn_") for s in syms), syms[:10]


def test_status_strings(lib):
    assert lib.rn_status_str(0) == b"ok"
    assert lib.rn_status_str(3) == b"workspace missing or too small"
    assert lib.rn_abi_version() == 1


def _out(**kw):
    o = rn._Output()
    for k, v in kw.items():
        setattr(o, k, v)
    return o


def test_forward_rejects_bad_arguments_on_host(lib):
    x = ctypes.c_void_p(0x1000)
    g = ctypes.c_void_p(0x2000)
    rs = ctypes.c_void_p(0x3000)
    mu = ctypes.c_void_p(0x4000)
    o = _out(data=0x5000, out_dtype=0)
    # NULL x
    assert lib.rn_rmsnorm_fwd(None, 0, g, 4, 1024, 1e-5, 0, 0, 0, ctypes.byref(o), rs, None) == 1
    # LayerNorm needs mu
    assert lib.rn_layernorm_fwd(x, 0, g, None, 4, 1024, 1e-5, 0, 0, 0, ctypes.byref(o), None, rs, None) == 1
    # bad dtype, bad mode, negative N
    assert lib.rn_rmsnorm_fwd(x, 7, g, 4, 1024, 1e-5, 0, 0, 0, ctypes.byref(o), rs, None) == 1
    assert lib.rn_rmsnorm_fwd(x, 0, g, 4, 1024, 1e-5, 0, 0, 9, ctypes.byref(o), rs, None) == 1
    assert lib.rn_rmsnorm_fwd(x, 0, g, -1, 1024, 1e-5, 0, 0, 0, ctypes.byref(o), rs, None) == 1
    # a field the mode does not use must be NULL
    o2 = _out(data=0x5000, amax=0x6000, out_dtype=0)
    assert lib.rn_rmsnorm_fwd(x, 0, g, 4, 1024, 1e-5, 0, 0, 0, ctypes.byref(o2), rs, None) == 1
    # FP8_DELAYED without its scale
    o3 = _out(data=0x5000, amax=0x6000, scale_inv=0x7000)
    assert lib.rn_rmsnorm_fwd(x, 0, g, 4, 1024, 1e-5, 0, 0, 1, ctypes.byref(o3), rs, None) == 1
    # bf16 rows must be a multiple of 8 elements; misaligned x
    assert lib.rn_rmsnorm_fwd(x, 0, g, 4, 1020, 1e-5, 0, 0, 0, ctypes.byref(o), rs, None) == 2
    assert lib.rn_rmsnorm_fwd(ctypes.c_void_p(0x1002), 0, g, 4, 1024, 1e-5, 0, 0, 0, ctypes.byref(o), rs, None) == 2
    # MXFP8 needs N and H multiples of 32
    om = _out(data=0x5000, row_scales=0x6000)
    assert lib.rn_layernorm_fwd(x, 0, g, None, 40, 1024, 1e-5, 0, 0, 3, ctypes.byref(om), mu, rs, None) == 2
    # quantize_only takes only the quantizing modes
    assert lib.rn_quantize_only(x, 4, 1024, 0, ctypes.byref(o), None) == 1


def test_nvfp4_forward_rejects_bad_arguments_on_host(lib):
    x = ctypes.c_void_p(0x1000)
    g = ctypes.c_void_p(0x2000)
    rs = ctypes.c_void_p(0x3000)
    full = dict(data=0x5000, row_scales=0x6000, scale_out=0x7000, scale_inv=0x7010, amax=0x7020)
    # every NVFP4 output is required; the FP8 / MX-only fields must be NULL
    for drop in full:
        o = _out(**{k: v for k, v in full.items() if k != drop})
        assert lib.rn_rmsnorm_fwd(x, 0, g, 4, 1024, 1e-5, 0, 0, 4, ctypes.byref(o), rs, None) == 1, drop
    for extra in ("col_data", "col_scales", "scale"):
        o = _out(**full, **{extra: 0x8000})
        assert lib.rn_rmsnorm_fwd(x, 0, g, 4, 1024, 1e-5, 0, 0, 4, ctypes.byref(o), rs, None) == 1, extra
    # rows must hold whole 16-element blocks (H = 1032 is a valid bf16 row)
    o = _out(**full)
    assert lib.rn_rmsnorm_fwd(x, 0, g, 4, 1032, 1e-5, 0, 0, 4, ctypes.byref(o), rs, None) == 2
    assert lib.rn_quantize_only(x, 4, 1028, 4, ctypes.byref(o), None) == 2
    # misaligned packed output
    o = _out(**dict(full, data=0x5008))
    assert lib.rn_rmsnorm_fwd(x, 0, g, 4, 1024, 1e-5, 0, 0, 4, ctypes.byref(o), rs, None) == 2


def test_backward_workspace_query_needs_no_device(lib):
    n = ctypes.c_size_t(0)
    # bf16 8192 x 4096: chunks of 8 rows -> 1024 partial rows of dgamma, dbeta
    assert lib.rn_layernorm_bwd(None, None, 0, None, None, None, 8192, 4096, 0, 0, None, None,
                                None, None, ctypes.byref(n), None) == 0
    assert n.value == 1024 * 2 * 4096 * 4
    # fp32 131072 x 1024: chunks of 128 rows
    assert lib.rn_rmsnorm_bwd(None, None, 1, None, None, 131072, 1024, 0, 0, None, None, None,
                              ctypes.byref(n), None) == 0
    assert n.value == 1024 * 1 * 1024 * 4
    # 3000 rows (ragged): 375 chunks
    assert lib.rn_rmsnorm_bwd(None, None, 0, None, None, 3000, 5120, 0, 0, None, None, None,
                              ctypes.byref(n), None) == 0
    assert n.value == 375 * 5120 * 4
    # query without a size pointer
    assert lib.rn_rmsnorm_bwd(None, None, 0, None, None, 64, 64, 0, 0, None, None, None, None, None) == 1


def test_backward_width_limits_on_host(lib):
    """The backward's widest rows (the header's conventions): bf16 H = 16384,
    fp32 H = 8192; the next width is refused at the workspace query."""
    n = ctypes.c_size_t(0)
    for dt, ok, bad in ((0, 16384, 16392), (1, 8192, 8196)):
        assert lib.rn_layernorm_bwd(None, None, dt, None, None, None, 64, ok, 0, 0, None, None,
                                    None, None, ctypes.byref(n), None) == 0
        assert n.value == 8 * 2 * ok * 4
        assert lib.rn_rmsnorm_bwd(None, None, dt, None, None, 64, bad, 0, 0, None, None, None,
                                  ctypes.byref(n), None) == 2


def test_backward_rejects_small_workspace_on_host(lib):
    p = ctypes.c_void_p(0x10000)
    n = ctypes.c_size_t(16)
    st = lib.rn_layernorm_bwd(p, p, 0, p, p, p, 64, 256, 0, 0, p, p, p, p, ctypes.byref(n), None)
    assert st == 3


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(rn, "_lib", None)
    monkeypatch.setattr(rn, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(rn.RNError, match="missing"):
        rn._load()


def test_residual_add_forward_rejects_bad_arguments_on_host(lib):
    x, r, h = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x8000), ctypes.c_void_p(0x9000)
    g, rs, mu = ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000), ctypes.c_void_p(0x4000)
    o = _out(data=0x5000, out_dtype=0)
    # the residual and the stored sum are required
    assert lib.rn_rmsnorm_add_fwd(x, None, 0, g, 4, 1024, 1e-5, 0, 0, 0, ctypes.byref(o), h, rs, None) == 1
    assert lib.rn_rmsnorm_add_fwd(x, r, 0, g, 4, 1024, 1e-5, 0, 0, 0, ctypes.byref(o), None, rs, None) == 1
    # MXFP8 with the columnwise copy after the residual add: N a multiple of 32
    om = _out(data=0x5000, row_scales=0x6000, col_data=0x7000, col_scales=0x7800)
    assert lib.rn_layernorm_add_fwd(x, r, 0, g, None, 48, 1024, 1e-5, 0, 0, 3, ctypes.byref(om), h, mu,
                                    rs, None) == 2
    # misaligned residual
    assert lib.rn_rmsnorm_add_fwd(x, ctypes.c_void_p(0x8004), 0, g, 4, 1024, 1e-5, 0, 0, 0, ctypes.byref(o),
                                  h, rs, None) == 2


def test_delayed_scaling_update_rejects_bad_arguments_on_host(lib):
    p = ctypes.c_void_p(0x1000)
    assert lib.rn_delayed_scaling_update(p, 0, p, p, p, None) == 1      # empty history
    assert lib.rn_delayed_scaling_update(None, 4, p, p, p, None) == 1
    assert lib.rn_delayed_scaling_update(p, 2048, p, p, p, None) == 2   # longer than 1024


def test_scaled_activation_rejects_bad_arguments_on_host(lib):
    x = ctypes.c_void_p(0x1000)
    o = _out(data=0x5000, out_dtype=0)
    f32 = ctypes.c_float
    # bad activation, NULL x, bad dtype, negative N
    assert lib.rn_scaled_act_fwd(7, x, 0, None, 4, 1024, f32(7), f32(1.702), 0, ctypes.byref(o), None) == 1
    assert lib.rn_scaled_act_fwd(1, None, 0, None, 4, 1024, f32(7), f32(1.702), 0, ctypes.byref(o), None) == 1
    assert lib.rn_scaled_act_fwd(1, x, 5, None, 4, 1024, f32(7), f32(1.702), 0, ctypes.byref(o), None) == 1
    assert lib.rn_scaled_act_fwd(1, x, 0, None, -1, 1024, f32(7), f32(1.702), 0, ctypes.byref(o), None) == 1
    # clamped SwiGLU needs a limit >= 0 and a finite alpha
    assert lib.rn_scaled_act_fwd(2, x, 0, None, 4, 1024, f32(-1), f32(1.702), 0, ctypes.byref(o), None) == 1
    assert lib.rn_scaled_act_fwd(2, x, 0, None, 4, 1024, f32(float("nan")), f32(1.702), 0, ctypes.byref(o), None) == 1
    assert lib.rn_scaled_act_fwd(2, x, 0, None, 4, 1024, f32(7), f32(float("inf")), 0, ctypes.byref(o), None) == 1
    # rows of whole 16-byte chunks, aligned x
    assert lib.rn_scaled_act_fwd(1, x, 0, None, 4, 1020, f32(7), f32(1.702), 0, ctypes.byref(o), None) == 2
    assert lib.rn_scaled_act_fwd(1, ctypes.c_void_p(0x1008), 0, None, 4, 1024, f32(7), f32(1.702), 0, ctypes.byref(o), None) == 2
    # MXFP8 rowwise only; no NVFP4
    om = _out(data=0x5000, row_scales=0x6000, col_data=0x7000, col_scales=0x8000)
    assert lib.rn_scaled_act_fwd(1, x, 0, None, 4, 1024, f32(7), f32(1.702), 3, ctypes.byref(om), None) == 2
    om = _out(data=0x5000, row_scales=0x6000)
    assert lib.rn_scaled_act_fwd(1, x, 0, None, 4, 1040, f32(7), f32(1.702), 3, ctypes.byref(om), None) == 2
    on = _out(data=0x5000, row_scales=0x6000, scale_out=0x7000, scale_inv=0x7010, amax=0x7020)
    assert lib.rn_scaled_act_fwd(1, x, 0, None, 4, 1024, f32(7), f32(1.702), 4, ctypes.byref(on), None) == 2
    # backward: NULL dy / dx, misaligned dx
    assert lib.rn_scaled_act_bwd(1, None, x, 0, None, 4, 1024, f32(7), f32(1.702), x, None, None) == 1
    assert lib.rn_scaled_act_bwd(1, x, x, 0, None, 4, 1024, f32(7), f32(1.702), None, None, None) == 1
    assert lib.rn_scaled_act_bwd(1, x, x, 0, None, 4, 1024, f32(7), f32(1.702), ctypes.c_void_p(0x2004), None, None) == 2


def test_binding_rejects_a_tensor_on_another_device(monkeypatch):
    import torch

    class OnDevice1:
        is_cuda = True
        device = torch.device("cuda", 1)
        dtype = torch.float32
        shape = (4,)

        def is_contiguous(self):
            return True

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    with pytest.raises(rn.RNError, match="current device"):
        rn._need(OnDevice1(), "x")
