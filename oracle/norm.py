"""LayerNorm / RMSNorm forward and backward with fused output quantization.

Oracle side, fp64, plain numpy.  Source: the page "Implementation:NVIDIA
TransformerEngine PyTorch Ext Normalization":

* Description: forward functions normalize and optionally quantize the
  output (paths UNFUSED, FULLY_FUSED for delayed scaling and MXFP8,
  FUSED_NORM_AMAX_FP8 for current scaling); backward functions return dx,
  dgamma and dbeta; gamma may be zero-centered; sm_margin only tunes
  occupancy (so it has no effect on any value computed here).
* Signature / I/O Contract: layernorm_fwd(input, weight, bias, eps, quantizer,
  sm_margin, zero_centered_gamma) -> (output, mu, rsigma); rmsnorm_fwd has no
  bias and no mu ("Mean (LayerNorm only)"); layernorm_bwd(dz, x, mu, rsigma,
  gamma, ...) -> (dx, dgamma, dbeta); rmsnorm_bwd(dz, x, rsigma, gamma, ...)
  -> (dx, dgamma).

The pages print no formula.  Readings taken (the plainest standard ones):
* variance is the biased one (divide by H); eps is added inside the square
  root for both norms; rsigma = 1 / sqrt(var + eps) (LayerNorm) and
  rsigma = 1 / sqrt(mean(x**2) + eps) (RMSNorm);
* zero-centered gamma means the effective weight is 1 + gamma, and dgamma is
  taken with respect to the stored gamma (same value, since d(1+g)/dg = 1);
* eps reaches the kernels as an fp32 argument, so its fp32 value is used;
* mu and rsigma are returned as fp32 (rounded once from fp64);
* the unquantized output is y rounded once to the output dtype;
* the quantization stage starts from y32 = fp32(y) and then follows exact
  IEEE fp32 steps, so that it can be compared bit for bit:
    delayed  p = fp32(y32 * s), code = E4M3(p), amax = max |y32| over the
             whole tensor, scale_inv = fp32(1 / s);
    current  amax as above, s = fp32(448 / amax) (s = 1 when amax = 0),
             then as delayed;
    MXFP8    per block of 32 (1x32 along a row, and 32x1 down a column):
             A = max |y32|, code_e8m0(A), element code = E4M3(y32 * 2**-e)
             (a power-of-two scaling, exact); the columnwise data is stored
             transposed, [H, N], with scales [H, N/32].
    NVFP4    (the page names this path, FUSED_NORM_AMAX_NVFP4, as the
             current-scaling scheme applied to NVFP4, and defines no format;
             the reading is NVIDIA's published NVFP4 layout: E2M1 elements,
             one E4M3 scale per 16 consecutive elements of a row, and one fp32
             scale for the tensor): amax as for current scaling,
             S = fp32(448 * 6 / amax) (the largest E4M3 times the largest
             E2M1; capped at the largest finite fp32; S = 1 when amax = 0),
             k = fp32(S / 6); per block of 16 along a row A = max |y32|,
             scale code sc = E4M3(fp32(A * k)), with v = its value
             e = fp32(S / v) (e = 0 when v = 0), element code =
             E2M1(fp32(y32 * e)); codes packed two to a byte (element 2j in
             the low nibble); the value an element stands for is
             E2M1 value * v / S.  Rowwise only.
* the backward takes mu and rsigma as given (the saved fp32 values), forms
  xhat = (x - mu) * rsigma (RMSNorm: x * rsigma), dy = dz * g_eff and
    LayerNorm  dx = rsigma * (dy - mean(dy) - xhat * mean(dy * xhat))
    RMSNorm    dx = rsigma * (dy - xhat * mean(dy * xhat))
  dgamma = sum over rows of dz * xhat, dbeta = sum over rows of dz; dx is
  rounded once to the dtype of x, dgamma / dbeta to fp32.
"""
from __future__ import annotations

import numpy as np

from .formats import (E2M1_MAX, E4M3_MAX, bf16_bits, e2m1_encode, e2m1_pack, e4m3_decode,
                      e4m3_encode, e8m0_from_amax, round_to_bf16)

QUANT_MODES = ("none", "fp8_delayed", "fp8_current", "mxfp8", "nvfp4")
MX_BLOCK = 32
NV_BLOCK = 16


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def _eps32(eps: float) -> float:
    return float(np.float32(eps))


def _g_eff(gamma, zero_centered_gamma: bool) -> np.ndarray:
    g = _f64(gamma)
    return 1.0 + g if zero_centered_gamma else g


# --------------------------------------------------------------- statistics
def layernorm_stats(x, eps):
    """Per-row mean m and r = 1/sqrt(var + eps), two-pass, fp64 -> (m, r)."""
    x = _f64(x)
    H = x.shape[-1]
    m = np.sum(x, axis=-1) / H
    d = x - m[..., None]
    v = np.sum(d * d, axis=-1) / H
    r = 1.0 / np.sqrt(v + _eps32(eps))
    return m, r


def rmsnorm_stats(x, eps):
    """Per-row r = 1/sqrt(mean(x**2) + eps), fp64."""
    x = _f64(x)
    H = x.shape[-1]
    ms = np.sum(x * x, axis=-1) / H
    return 1.0 / np.sqrt(ms + _eps32(eps))


def norm_apply(x, m, r, gamma, beta, zero_centered_gamma):
    """y = (x - m) * r * g_eff + beta; m None -> RMSNorm (no centering)."""
    x = _f64(x)
    g = _g_eff(gamma, zero_centered_gamma)
    c = x if m is None else x - _f64(m)[..., None]
    y = c * _f64(r)[..., None] * g
    if beta is not None:
        y = y + _f64(beta)
    return y


# ------------------------------------------------------------- quantization
def fp8_codes(y32, s) -> np.ndarray:
    """E4M3 codes of fp32(y32 * s) (one fp32 multiply, then E4M3 rounding)."""
    p = np.asarray(y32, dtype=np.float32) * np.float32(s)
    return e4m3_encode(p.astype(np.float64))


def tensor_amax(y32) -> np.float32:
    """max |y32| over the whole tensor (NaN if any element is NaN)."""
    a = np.abs(np.asarray(y32, dtype=np.float32))
    if a.size == 0:
        return np.float32(0.0)
    return np.float32(np.max(a))


def current_scale(amax) -> np.float32:
    """s = fp32(448 / amax) by one IEEE fp32 division; amax = 0 -> 1."""
    a = np.float32(amax)
    if a == 0:
        return np.float32(1.0)
    return np.float32(np.float32(E4M3_MAX) / a)


def scale_inverse(s) -> np.float32:
    return np.float32(np.float32(1.0) / np.float32(s))


def mx_blocks_1d(y32_rows) -> tuple[np.ndarray, np.ndarray]:
    """MX-quantize along the last axis in blocks of 32 -> (codes, e8m0)."""
    y = np.asarray(y32_rows, dtype=np.float32)
    n, h = y.shape
    assert h % MX_BLOCK == 0
    yb = y.reshape(n, h // MX_BLOCK, MX_BLOCK)
    a = np.abs(yb)
    nanblk = np.isnan(a).any(axis=-1)
    amax = np.where(nanblk, np.float32(np.nan), np.nanmax(np.where(np.isnan(a), 0, a), axis=-1))
    code = e8m0_from_amax(amax)
    e = code.astype(np.int64) - 127
    scaled = yb.astype(np.float64) * np.ldexp(1.0, (-e).astype(np.int32))[..., None]
    q = e4m3_encode(scaled)
    q = np.where(nanblk[..., None], np.uint8(0x7F), q).astype(np.uint8)
    return q.reshape(n, h), code


def nvfp4_global_scale(amax) -> np.float32:
    """S = fp32(448 * 6 / amax) by one IEEE fp32 division, capped at the
    largest finite fp32; amax = 0 -> 1."""
    a = np.float32(amax)
    if a == 0:
        return np.float32(1.0)
    with np.errstate(over="ignore", divide="ignore"):
        s = np.float32(np.float32(E4M3_MAX * E2M1_MAX) / a)
    return np.minimum(s, np.float32(np.finfo(np.float32).max))


def nvfp4_blocks_1d(y32_rows, S) -> tuple[np.ndarray, np.ndarray]:
    """NVFP4-quantize along the last axis in blocks of 16 with tensor scale S
    -> (packed E2M1 codes [n, h/2], E4M3 block-scale codes [n, h/16])."""
    y = np.asarray(y32_rows, dtype=np.float32)
    n, h = y.shape
    assert h % NV_BLOCK == 0
    if np.isnan(y).any():
        raise ValueError("NVFP4 has no code for NaN")
    S = np.float32(S)
    k = np.float32(S / np.float32(E2M1_MAX))
    yb = y.reshape(n, h // NV_BLOCK, NV_BLOCK)
    A = np.max(np.abs(yb), axis=-1)                      # fp32, exact
    with np.errstate(over="ignore"):
        sc = e4m3_encode((A * k).astype(np.float64))     # fp32 product, then E4M3
    v = e4m3_decode(sc).astype(np.float32)               # exact
    with np.errstate(divide="ignore"):
        e = np.where(v == 0, np.float32(0.0), S / np.where(v == 0, np.float32(1.0), v))
    e = e.astype(np.float32)
    p = yb * e[..., None]                                # fp32 products
    codes = e2m1_encode(p.astype(np.float64)).reshape(n, h)
    return e2m1_pack(codes), sc


def quantize(y32, mode: str, scale=None, amax=None) -> dict:
    """Quantization stage for a block of fp32 pre-quantization rows.

    ``y32`` [n, H] fp32.  For fp8_current and nvfp4 the tensor-wide ``amax`` may be
    given (when y32 is only a sample of the rows); otherwise it is taken from
    y32.  Returns the fields the entry points return for that mode.
    """
    y32 = np.asarray(y32, dtype=np.float32)
    if mode == "fp8_delayed":
        s = np.float32(scale)
        return {"data": fp8_codes(y32, s), "amax": tensor_amax(y32),
                "scale_inv": scale_inverse(s)}
    if mode == "fp8_current":
        am = tensor_amax(y32) if amax is None else np.float32(amax)
        s = current_scale(am)
        return {"data": fp8_codes(y32, s), "amax": am, "scale": s,
                "scale_inv": scale_inverse(s)}
    if mode == "nvfp4":
        am = tensor_amax(y32) if amax is None else np.float32(amax)
        S = nvfp4_global_scale(am)
        q, sc = nvfp4_blocks_1d(y32, S)
        return {"data": q, "row_scales": sc, "amax": am, "scale": S,
                "scale_inv": scale_inverse(S)}
    if mode == "mxfp8":
        rq, rs = mx_blocks_1d(y32)
        cq, cs = mx_blocks_1d(np.ascontiguousarray(y32.T))
        return {"data": rq, "row_scales": rs, "col_data": cq, "col_scales": cs}
    raise ValueError(mode)


def _out_none(y, out_dtype: str):
    if out_dtype == "bf16":
        return bf16_bits(y)
    if out_dtype == "f32":
        return y.astype(np.float32)
    raise ValueError(out_dtype)


# ------------------------------------------------------------------ forward
def _fwd(x, m, r, gamma, beta, zcg, mode, out_dtype, scale, amax):
    y = norm_apply(x, m, r, gamma, beta, zcg)
    res = {"y": y, "rsigma": np.asarray(r, dtype=np.float64).astype(np.float32)}
    if m is not None:
        res["mu"] = np.asarray(m, dtype=np.float64).astype(np.float32)
    if mode == "none":
        res["data"] = _out_none(y, out_dtype)
    else:
        res.update(quantize(y.astype(np.float32), mode, scale=scale, amax=amax))
    return res


def layernorm_fwd(x, gamma, beta, eps, zero_centered_gamma=False, mode="none",
                  out_dtype="bf16", scale=None, amax=None) -> dict:
    """LayerNorm forward -> dict(data, mu, rsigma, y, [amax, scale_inv, ...])."""
    m, r = layernorm_stats(x, eps)
    return _fwd(x, m, r, gamma, beta, zero_centered_gamma, mode, out_dtype, scale, amax)


def rmsnorm_fwd(x, gamma, eps, zero_centered_gamma=False, mode="none",
                out_dtype="bf16", scale=None, amax=None) -> dict:
    """RMSNorm forward -> dict(data, rsigma, y, ...); no mu."""
    r = rmsnorm_stats(x, eps)
    return _fwd(x, None, r, gamma, None, zero_centered_gamma, mode, out_dtype, scale, amax)


# ----------------------------------------------------------------- backward
def _bwd(dz, x, mu, rsigma, gamma, zcg, dtype):
    dz = _f64(dz)
    x = _f64(x)
    r = _f64(rsigma)[:, None]
    xhat = (x if mu is None else x - _f64(mu)[:, None]) * r
    dy = dz * _g_eff(gamma, zcg)
    c2 = np.mean(dy * xhat, axis=1, keepdims=True)
    if mu is None:
        dx = r * (dy - xhat * c2)
    else:
        c1 = np.mean(dy, axis=1, keepdims=True)
        dx = r * (dy - c1 - xhat * c2)
    res = {"dx64": dx, "dgamma64": np.sum(dz * xhat, axis=0)}
    res["dx"] = bf16_bits(dx) if dtype == "bf16" else dx.astype(np.float32)
    res["dgamma"] = res["dgamma64"].astype(np.float32)
    if mu is not None:
        res["dbeta64"] = np.sum(dz, axis=0)
        res["dbeta"] = res["dbeta64"].astype(np.float32)
    return res


def layernorm_bwd(dz, x, mu, rsigma, gamma, zero_centered_gamma=False, dtype="bf16") -> dict:
    """LayerNorm backward -> dict(dx, dgamma, dbeta, and their fp64 forms)."""
    return _bwd(dz, x, mu, rsigma, gamma, zero_centered_gamma, dtype)


def rmsnorm_bwd(dz, x, rsigma, gamma, zero_centered_gamma=False, dtype="bf16") -> dict:
    """RMSNorm backward -> dict(dx, dgamma, and fp64 forms); no dbeta."""
    return _bwd(dz, x, None, rsigma, gamma, zero_centered_gamma, dtype)


# --------------------------------------------------- residual add + norm
# Source: the page "NVIDIA Megatron-Core ... core.tensor_parallel.
# inference_layers" names a fused reduce-scatter + residual add + RMSNorm +
# all-gather; on one GPU its core is "add the residual, then normalize (and
# quantize)".  The page gives no rounding.  Reading: the sum is the new
# residual stream, kept in the stream's dtype (rounded once, to nearest even),
# and the norm is applied to that stored value, so that the next layer's
# residual input is exactly what was normalized.
def residual_add(x, residual, dtype: str = "bf16") -> np.ndarray:
    """h = x + residual rounded once to `dtype` ("bf16" or "f32"), as fp64.

    The fp64 sum is exact for two bf16 values, and for two fp32 values it
    rounds to fp32 like the exact sum (an addend too small to be exact in
    fp64 is far below half an fp32 ulp of the other).
    """
    s = _f64(x) + _f64(residual)
    if dtype == "bf16":
        return round_to_bf16(s)
    if dtype == "f32":
        return s.astype(np.float32).astype(np.float64)
    raise ValueError(dtype)


def _stream(h, dtype: str):
    return bf16_bits(h) if dtype == "bf16" else h.astype(np.float32)


def rmsnorm_add_fwd(x, residual, gamma, eps, dtype="bf16", zero_centered_gamma=False,
                    mode="none", out_dtype="bf16", scale=None, amax=None) -> dict:
    """RMSNorm of h = residual_add(x, residual) -> rmsnorm_fwd's dict plus
    residual_out (h in the stream dtype)."""
    h = residual_add(x, residual, dtype)
    res = rmsnorm_fwd(h, gamma, eps, zero_centered_gamma, mode, out_dtype, scale, amax)
    res["residual_out"] = _stream(h, dtype)
    res["h"] = h
    return res


def layernorm_add_fwd(x, residual, gamma, beta, eps, dtype="bf16", zero_centered_gamma=False,
                      mode="none", out_dtype="bf16", scale=None, amax=None) -> dict:
    """LayerNorm of h = residual_add(x, residual) -> layernorm_fwd's dict plus
    residual_out."""
    h = residual_add(x, residual, dtype)
    res = layernorm_fwd(h, gamma, beta, eps, zero_centered_gamma, mode, out_dtype, scale, amax)
    res["residual_out"] = _stream(h, dtype)
    res["h"] = h
    return res


# ------------------------------------------- delayed-scaling recipe step
# The page describes delayed scaling (FP8 with a scale chosen from earlier
# steps' amax) without the bookkeeping.  Reading (the common recipe, margin
# 0): the history keeps the most recent amax at index 0; a step shifts it by
# one place and puts the new amax first; the next scale is
# fp32(448 / max(history)) by one IEEE fp32 division, except that a maximum
# that is 0 or not finite keeps the previous scale; scale_inv = fp32(1 / scale).
def amax_history_update(history, amax, scale):
    """-> (new history float32 [L], new scale float32, new scale_inv float32)."""
    h = np.asarray(history, dtype=np.float32)
    new = np.empty_like(h)
    if h.size:
        new[0] = np.float32(amax)
        new[1:] = h[:-1]
    m = np.float32(np.max(new)) if new.size else np.float32(0.0)
    if np.isnan(new).any():
        m = np.float32(np.nan)
    if np.isfinite(m) and m > 0:
        s = np.float32(np.float32(E4M3_MAX) / m)
    else:
        s = np.float32(scale)
    return new, s, np.float32(np.float32(1.0) / s)
