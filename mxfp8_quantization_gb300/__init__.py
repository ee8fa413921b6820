"""GB300 fused LayerNorm / RMSNorm with FP8, MXFP8 and NVFP4 output.

Thin Python binding over the C ABI in ``include/rn.h`` (``librn.so``, built
in-tree by ``_build.build()``).  This module only marshals arguments: it
allocates outputs with PyTorch, passes raw device pointers and the current
CUDA stream, and raises on a nonzero status.  Every step of the computation
runs in the library's CUDA kernels; there is no fallback.

Entry points mirror the page "Implementation:NVIDIA TransformerEngine
PyTorch Ext Normalization" (section "Signature"):

    layernorm_fwd(x, gamma, beta, eps, quant, sm_margin, zero_centered_gamma)
        -> (output, mu, rsigma)
    rmsnorm_fwd(x, gamma, eps, quant, sm_margin, zero_centered_gamma)
        -> (output, rsigma)
    layernorm_bwd(dz, x, mu, rsigma, gamma, sm_margin, zero_centered_gamma)
        -> (dx, dgamma, dbeta)
    rmsnorm_bwd(dz, x, rsigma, gamma, sm_margin, zero_centered_gamma)
        -> (dx, dgamma)

``quant`` is one of "none", "fp8_delayed" (needs ``scale``), "fp8_current",
"mxfp8", "nvfp4"; the page's quantizer object becomes this string plus the
scale.  ``scaled_act_fwd`` / ``scaled_act_bwd`` are the scaled SReLU, SwiGLU
and clamped SwiGLU of the page "Activation + GroupedLinear Fusion for MOE
and other MOE optimizations".
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

__all__ = [
    "layernorm_fwd", "rmsnorm_fwd", "layernorm_bwd", "rmsnorm_bwd", "quantize_only",
    "layernorm_bwd_noalloc", "layernorm_add_fwd", "rmsnorm_add_fwd", "delayed_scaling_update",
    "bwd_workspace_bytes", "device_error", "Fp8Output", "MXFP8Output", "NVFP4Output", "lib_path",
    "RNError",
    "QUANT_MODES", "ACTS", "scaled_act_fwd", "scaled_act_bwd",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "librn.so")
QUANT_MODES = {"none": 0, "fp8_delayed": 1, "fp8_current": 2, "mxfp8": 3, "nvfp4": 4}
_BF16, _F32 = 0, 1
ACTS = {"srelu": 0, "swiglu": 1, "clamped_swiglu": 2}


class RNError(RuntimeError):
    pass


class _Output(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("row_scales", ctypes.c_void_p),
        ("col_data", ctypes.c_void_p),
        ("col_scales", ctypes.c_void_p),
        ("scale", ctypes.c_void_p),
        ("scale_out", ctypes.c_void_p),
        ("scale_inv", ctypes.c_void_p),
        ("amax", ctypes.c_void_p),
        ("out_dtype", ctypes.c_int),
    ]


_lib = None


def lib_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RNError(
            f"{_LIB_PATH} is missing: build it first (mxfp8_quantization_gb300._build.build())")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    outp = ctypes.POINTER(_Output)
    szp = ctypes.POINTER(ctypes.c_size_t)
    lib.rn_layernorm_fwd.argtypes = [vp, i32, vp, vp, i64, i64, f32, i32, i32, i32, outp, vp, vp, vp]
    lib.rn_rmsnorm_fwd.argtypes = [vp, i32, vp, i64, i64, f32, i32, i32, i32, outp, vp, vp]
    lib.rn_layernorm_bwd.argtypes = [vp, vp, i32, vp, vp, vp, i64, i64, i32, i32, vp, vp, vp, vp, szp, vp]
    lib.rn_rmsnorm_bwd.argtypes = [vp, vp, i32, vp, vp, i64, i64, i32, i32, vp, vp, vp, szp, vp]
    lib.rn_layernorm_add_fwd.argtypes = [vp, vp, i32, vp, vp, i64, i64, f32, i32, i32, i32, outp,
                                         vp, vp, vp, vp]
    lib.rn_rmsnorm_add_fwd.argtypes = [vp, vp, i32, vp, i64, i64, f32, i32, i32, i32, outp, vp, vp,
                                       vp]
    lib.rn_quantize_only.argtypes = [vp, i64, i64, i32, outp, vp]
    lib.rn_delayed_scaling_update.argtypes = [vp, i64, vp, vp, vp, vp]
    lib.rn_scaled_act_fwd.argtypes = [i32, vp, i32, vp, i64, i64, f32, f32, i32, outp, vp]
    lib.rn_scaled_act_bwd.argtypes = [i32, vp, vp, i32, vp, i64, i64, f32, f32, vp, vp, vp]
    lib.rn_layernorm_bwd_noalloc.argtypes = [vp, vp, i32, vp, vp, vp, i64, i64, i32, i32, vp, vp, vp, vp]
    lib.rn_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    lib.rn_status_str.argtypes = [i32]
    lib.rn_status_str.restype = ctypes.c_char_p
    for f in ("rn_layernorm_fwd", "rn_rmsnorm_fwd", "rn_layernorm_bwd", "rn_rmsnorm_bwd",
              "rn_quantize_only", "rn_device_error", "rn_abi_version", "rn_layernorm_bwd_noalloc",
              "rn_layernorm_add_fwd", "rn_rmsnorm_add_fwd", "rn_delayed_scaling_update",
              "rn_scaled_act_fwd", "rn_scaled_act_bwd"):
        getattr(lib, f).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != 0:
        msg = _load().rn_status_str(status).decode()
        raise RNError(f"{what}: status {status} ({msg})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return _BF16
    if t.dtype == torch.float32:
        return _F32
    raise RNError(f"unsupported dtype {t.dtype}: x must be bfloat16 or float32")


def _need(t, name, dtype=None, shape=None):
    if t is None:
        raise RNError(f"{name} is required")
    if not t.is_cuda or not t.is_contiguous():
        raise RNError(f"{name} must be a contiguous CUDA tensor")
    # the library launches on the current device (and picks its per-device
    # state by it): a tensor on another device would be read through the
    # wrong device's pointers
    if t.device.index != torch.cuda.current_device():
        raise RNError(f"{name} is on {t.device}, but the current device is "
                      f"cuda:{torch.cuda.current_device()}")
    if dtype is not None and t.dtype != dtype:
        raise RNError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise RNError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


@dataclass
class Fp8Output:
    """E4M3 codes with their per-tensor scale (FP8_DELAYED / FP8_CURRENT)."""
    data: torch.Tensor       # uint8 [N, H]
    scale_inv: torch.Tensor  # fp32 [1]
    amax: torch.Tensor       # fp32 [1]
    scale: torch.Tensor      # fp32 [1] (given for delayed, computed for current)


@dataclass
class MXFP8Output:
    """MXFP8: rowwise 1x32 and columnwise 32x1 blocks with E8M0 scales."""
    data: torch.Tensor | None        # uint8 [N, H]
    row_scales: torch.Tensor | None  # uint8 [N, H/32]
    col_data: torch.Tensor | None    # uint8 [H, N] (transposed)
    col_scales: torch.Tensor | None  # uint8 [H, N/32]


@dataclass
class NVFP4Output:
    """NVFP4: E2M1 codes with an E4M3 scale per 1x16 block and a tensor scale."""
    data: torch.Tensor        # uint8 [N, H/2], two codes per byte (even element low)
    row_scales: torch.Tensor  # uint8 [N, H/16] E4M3 block-scale codes
    scale: torch.Tensor       # fp32 [1] S = 448 * 6 / amax
    scale_inv: torch.Tensor   # fp32 [1] 1 / S
    amax: torch.Tensor        # fp32 [1]


def _make_output(x, quant, out_dtype, scale, rowwise=True, colwise=True):
    N, H = x.shape
    dev = x.device
    o = _Output()
    if quant == "none":
        odt = x.dtype if out_dtype is None else out_dtype
        data = torch.empty((N, H), dtype=odt, device=dev)
        o.data = data.data_ptr()
        o.out_dtype = _dtype_code(data)
        return o, data
    if quant in ("fp8_delayed", "fp8_current"):
        data = torch.empty((N, H), dtype=torch.uint8, device=dev)
        res = Fp8Output(data, torch.empty(1, dtype=torch.float32, device=dev),
                        torch.empty(1, dtype=torch.float32, device=dev), None)
        o.data = data.data_ptr()
        o.scale_inv = res.scale_inv.data_ptr()
        o.amax = res.amax.data_ptr()
        if quant == "fp8_delayed":
            if scale is None:
                raise RNError("fp8_delayed needs scale")
            s = scale if isinstance(scale, torch.Tensor) else torch.tensor([float(scale)], dtype=torch.float32)
            s = s.to(device=dev, dtype=torch.float32).reshape(1).contiguous()
            res.scale = s
            o.scale = s.data_ptr()
        else:
            res.scale = torch.empty(1, dtype=torch.float32, device=dev)
            o.scale_out = res.scale.data_ptr()
        return o, res
    if quant == "mxfp8":
        res = MXFP8Output(None, None, None, None)
        if rowwise:
            res.data = torch.empty((N, H), dtype=torch.uint8, device=dev)
            res.row_scales = torch.empty((N, H // 32), dtype=torch.uint8, device=dev)
            o.data = res.data.data_ptr()
            o.row_scales = res.row_scales.data_ptr()
        if colwise:
            res.col_data = torch.empty((H, N), dtype=torch.uint8, device=dev)
            res.col_scales = torch.empty((H, N // 32), dtype=torch.uint8, device=dev)
            o.col_data = res.col_data.data_ptr()
            o.col_scales = res.col_scales.data_ptr()
        return o, res
    if quant == "nvfp4":
        f32 = dict(dtype=torch.float32, device=dev)
        res = NVFP4Output(torch.empty((N, H // 2), dtype=torch.uint8, device=dev),
                          torch.empty((N, H // 16), dtype=torch.uint8, device=dev),
                          torch.empty(1, **f32), torch.empty(1, **f32), torch.empty(1, **f32))
        o.data = res.data.data_ptr()
        o.row_scales = res.row_scales.data_ptr()
        o.scale_out = res.scale.data_ptr()
        o.scale_inv = res.scale_inv.data_ptr()
        o.amax = res.amax.data_ptr()
        return o, res
    raise RNError(f"unknown quant mode {quant!r}")


def layernorm_fwd(x, gamma, beta, eps, quant="none", sm_margin=0, zero_centered_gamma=False,
                  scale=None, out_dtype=None, rowwise=True, colwise=True):
    """LayerNorm forward -> (output, mu, rsigma); output per ``quant``."""
    lib = _load()
    _need(x, "x")
    N, H = x.shape
    _need(gamma, "gamma", torch.float32, (H,))
    if beta is not None:
        _need(beta, "beta", torch.float32, (H,))
    mu = torch.empty(N, dtype=torch.float32, device=x.device)
    rsigma = torch.empty(N, dtype=torch.float32, device=x.device)
    o, res = _make_output(x, quant, out_dtype, scale, rowwise, colwise)
    st = lib.rn_layernorm_fwd(_ptr(x), _dtype_code(x), _ptr(gamma), _ptr(beta), N, H, float(eps),
                              int(bool(zero_centered_gamma)), int(sm_margin), QUANT_MODES[quant],
                              ctypes.byref(o), _ptr(mu), _ptr(rsigma), _stream())
    _check(st, "rn_layernorm_fwd")
    return res, mu, rsigma


def rmsnorm_fwd(x, gamma, eps, quant="none", sm_margin=0, zero_centered_gamma=False, scale=None,
                out_dtype=None, rowwise=True, colwise=True):
    """RMSNorm forward -> (output, rsigma); output per ``quant``."""
    lib = _load()
    _need(x, "x")
    N, H = x.shape
    _need(gamma, "gamma", torch.float32, (H,))
    rsigma = torch.empty(N, dtype=torch.float32, device=x.device)
    o, res = _make_output(x, quant, out_dtype, scale, rowwise, colwise)
    st = lib.rn_rmsnorm_fwd(_ptr(x), _dtype_code(x), _ptr(gamma), N, H, float(eps),
                            int(bool(zero_centered_gamma)), int(sm_margin), QUANT_MODES[quant],
                            ctypes.byref(o), _ptr(rsigma), _stream())
    _check(st, "rn_rmsnorm_fwd")
    return res, rsigma


def layernorm_add_fwd(x, residual, gamma, beta, eps, quant="none", sm_margin=0,
                      zero_centered_gamma=False, scale=None, out_dtype=None, rowwise=True,
                      colwise=True):
    """h = x + residual (rounded to x's dtype), LayerNorm(h) -> (output, h, mu, rsigma);
    output per ``quant`` (MXFP8: the blocks ``rowwise`` / ``colwise`` select)."""
    lib = _load()
    _need(x, "x")
    N, H = x.shape
    _need(residual, "residual", x.dtype, (N, H))
    _need(gamma, "gamma", torch.float32, (H,))
    if beta is not None:
        _need(beta, "beta", torch.float32, (H,))
    h = torch.empty_like(x)
    mu = torch.empty(N, dtype=torch.float32, device=x.device)
    rsigma = torch.empty(N, dtype=torch.float32, device=x.device)
    o, res = _make_output(x, quant, out_dtype, scale, rowwise, colwise)
    st = lib.rn_layernorm_add_fwd(_ptr(x), _ptr(residual), _dtype_code(x), _ptr(gamma), _ptr(beta),
                                  N, H, float(eps), int(bool(zero_centered_gamma)), int(sm_margin),
                                  QUANT_MODES[quant], ctypes.byref(o), _ptr(h), _ptr(mu),
                                  _ptr(rsigma), _stream())
    _check(st, "rn_layernorm_add_fwd")
    return res, h, mu, rsigma


def rmsnorm_add_fwd(x, residual, gamma, eps, quant="none", sm_margin=0,
                    zero_centered_gamma=False, scale=None, out_dtype=None, rowwise=True,
                    colwise=True):
    """h = x + residual (rounded to x's dtype), RMSNorm(h) -> (output, h, rsigma); output per
    ``quant`` (MXFP8: the blocks ``rowwise`` / ``colwise`` select)."""
    lib = _load()
    _need(x, "x")
    N, H = x.shape
    _need(residual, "residual", x.dtype, (N, H))
    _need(gamma, "gamma", torch.float32, (H,))
    h = torch.empty_like(x)
    rsigma = torch.empty(N, dtype=torch.float32, device=x.device)
    o, res = _make_output(x, quant, out_dtype, scale, rowwise, colwise)
    st = lib.rn_rmsnorm_add_fwd(_ptr(x), _ptr(residual), _dtype_code(x), _ptr(gamma), N, H,
                                float(eps), int(bool(zero_centered_gamma)), int(sm_margin),
                                QUANT_MODES[quant], ctypes.byref(o), _ptr(h), _ptr(rsigma),
                                _stream())
    _check(st, "rn_rmsnorm_add_fwd")
    return res, h, rsigma


def delayed_scaling_update(amax_history, amax, scale):
    """One delayed-scaling step on device tensors: shifts `amax` (fp32 [1])
    into `amax_history` (fp32 [L], most recent first) and updates `scale`
    (fp32 [1]) in place; returns scale_inv (fp32 [1])."""
    lib = _load()
    _need(amax_history, "amax_history", torch.float32)
    _need(amax, "amax", torch.float32, (1,))
    _need(scale, "scale", torch.float32, (1,))
    scale_inv = torch.empty(1, dtype=torch.float32, device=scale.device)
    st = lib.rn_delayed_scaling_update(_ptr(amax_history), amax_history.numel(), _ptr(amax),
                                       _ptr(scale), _ptr(scale_inv), _stream())
    _check(st, "rn_delayed_scaling_update")
    return scale_inv


def _act_width(x, act):
    if act not in ACTS:
        raise RNError(f"unknown activation {act!r}")
    return x.shape[1] if act == "srelu" else x.shape[1] // 2


def scaled_act_fwd(x, act, scales=None, quant="none", limit=7.0, alpha=1.702, scale=None,
                   out_dtype=None):
    """y = scales[:, None] * act(x): x [N, H] (srelu) or [N, 2H] (swiglu,
    clamped_swiglu: gate half, then linear half); returns the output in the
    form of the forward norm calls (MXFP8: rowwise blocks only)."""
    lib = _load()
    _need(x, "x")
    N, H = x.shape[0], _act_width(x, act)
    if scales is not None:
        _need(scales, "scales", torch.float32, (N,))
    o, res = _make_output(x[:, :H], quant, out_dtype, scale, True, False)
    st = lib.rn_scaled_act_fwd(ACTS[act], _ptr(x), _dtype_code(x), _ptr(scales), N, H,
                               float(limit), float(alpha), QUANT_MODES[quant], ctypes.byref(o),
                               _stream())
    _check(st, "rn_scaled_act_fwd")
    return res


def scaled_act_bwd(dy, x, act, scales=None, limit=7.0, alpha=1.702, dscales=True):
    """-> (dx shaped like x, dscales fp32 [N] or None)."""
    lib = _load()
    _need(x, "x")
    N, H = x.shape[0], _act_width(x, act)
    _need(dy, "dy", x.dtype, (N, H))
    if scales is not None:
        _need(scales, "scales", torch.float32, (N,))
    dx = torch.empty_like(x)
    ds = torch.empty(N, dtype=torch.float32, device=x.device) if dscales else None
    st = lib.rn_scaled_act_bwd(ACTS[act], _ptr(dy), _ptr(x), _dtype_code(x), _ptr(scales), N, H,
                               float(limit), float(alpha), _ptr(dx), _ptr(ds), _stream())
    _check(st, "rn_scaled_act_bwd")
    return dx, ds


def bwd_workspace_bytes(N, H, dtype, layernorm=True) -> int:
    """Workspace bytes the backward needs (the query step of the protocol)."""
    lib = _load()
    n = ctypes.c_size_t(0)
    code = _BF16 if dtype == torch.bfloat16 else _F32
    if layernorm:
        st = lib.rn_layernorm_bwd(None, None, code, None, None, None, N, H, 0, 0, None, None, None,
                                  None, ctypes.byref(n), None)
    else:
        st = lib.rn_rmsnorm_bwd(None, None, code, None, None, N, H, 0, 0, None, None, None,
                                ctypes.byref(n), None)
    _check(st, "workspace query")
    return int(n.value)


def _workspace(N, H, dtype, layernorm, device, workspace):
    need = bwd_workspace_bytes(N, H, dtype, layernorm)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
    return workspace, ctypes.c_size_t(workspace.numel() * workspace.element_size())


def layernorm_bwd(dz, x, mu, rsigma, gamma, sm_margin=0, zero_centered_gamma=False, workspace=None):
    """LayerNorm backward -> (dx, dgamma, dbeta)."""
    lib = _load()
    _need(x, "x")
    N, H = x.shape
    _need(dz, "dz", x.dtype, (N, H))
    _need(mu, "mu", torch.float32, (N,))
    _need(rsigma, "rsigma", torch.float32, (N,))
    _need(gamma, "gamma", torch.float32, (H,))
    dx = torch.empty_like(x)
    dgamma = torch.empty(H, dtype=torch.float32, device=x.device)
    dbeta = torch.empty(H, dtype=torch.float32, device=x.device)
    ws, n = _workspace(N, H, x.dtype, True, x.device, workspace)
    st = lib.rn_layernorm_bwd(_ptr(dz), _ptr(x), _dtype_code(x), _ptr(mu), _ptr(rsigma), _ptr(gamma),
                              N, H, int(bool(zero_centered_gamma)), int(sm_margin), _ptr(dx),
                              _ptr(dgamma), _ptr(dbeta), _ptr(ws), ctypes.byref(n), _stream())
    _check(st, "rn_layernorm_bwd")
    return dx, dgamma, dbeta


def rmsnorm_bwd(dz, x, rsigma, gamma, sm_margin=0, zero_centered_gamma=False, workspace=None):
    """RMSNorm backward -> (dx, dgamma)."""
    lib = _load()
    _need(x, "x")
    N, H = x.shape
    _need(dz, "dz", x.dtype, (N, H))
    _need(rsigma, "rsigma", torch.float32, (N,))
    _need(gamma, "gamma", torch.float32, (H,))
    dx = torch.empty_like(x)
    dgamma = torch.empty(H, dtype=torch.float32, device=x.device)
    ws, n = _workspace(N, H, x.dtype, False, x.device, workspace)
    st = lib.rn_rmsnorm_bwd(_ptr(dz), _ptr(x), _dtype_code(x), _ptr(rsigma), _ptr(gamma), N, H,
                            int(bool(zero_centered_gamma)), int(sm_margin), _ptr(dx), _ptr(dgamma),
                            _ptr(ws), ctypes.byref(n), _stream())
    _check(st, "rn_rmsnorm_bwd")
    return dx, dgamma


def layernorm_bwd_noalloc(dz, x, mu, rsigma, gamma, sm_margin=0, zero_centered_gamma=False):
    """LayerNorm backward -> (dx, dgamma, dbeta) without a workspace: the
    library's fixed per-device scratch array holds the partial sums (for
    callers that cannot allocate device memory; see include/rn.h for its size
    limit and the rule that overlapping calls race)."""
    lib = _load()
    _need(x, "x")
    N, H = x.shape
    _need(dz, "dz", x.dtype, (N, H))
    _need(mu, "mu", torch.float32, (N,))
    _need(rsigma, "rsigma", torch.float32, (N,))
    _need(gamma, "gamma", torch.float32, (H,))
    dx = torch.empty_like(x)
    dgamma = torch.empty(H, dtype=torch.float32, device=x.device)
    dbeta = torch.empty(H, dtype=torch.float32, device=x.device)
    st = lib.rn_layernorm_bwd_noalloc(_ptr(dz), _ptr(x), _dtype_code(x), _ptr(mu), _ptr(rsigma),
                                      _ptr(gamma), N, H, int(bool(zero_centered_gamma)),
                                      int(sm_margin), _ptr(dx), _ptr(dgamma), _ptr(dbeta), _stream())
    _check(st, "rn_layernorm_bwd_noalloc")
    return dx, dgamma, dbeta


def quantize_only(y, quant, scale=None, rowwise=True, colwise=True):
    """Quantize caller-given fp32 values [N, H] (the unfused quantize step)."""
    lib = _load()
    _need(y, "y", torch.float32)
    N, H = y.shape
    o, res = _make_output(y, quant, None, scale, rowwise, colwise)
    st = lib.rn_quantize_only(_ptr(y), N, H, QUANT_MODES[quant], ctypes.byref(o), _stream())
    _check(st, "rn_quantize_only")
    return res


def device_error() -> int:
    """Read and clear the kernels' device error word (synchronizes)."""
    code = ctypes.c_uint(0)
    _check(_load().rn_device_error(ctypes.byref(code)), "rn_device_error")
    return int(code.value)
