"""Scaled activations, forward and backward (oracle side, fp64, numpy).

Source: the page "Activation + GroupedLinear Fusion for MOE and other MOE
optimizations" (TransformerEngine pull request 3238), sections "Better
Kernels for Scaled Activations" and "Important Files Changed": scaled SReLU,
SwiGLU and clamped SwiGLU become single fused kernels; their backward
returns the input gradient and the gradient of the scales ("grad_scales");
the scales are saved for the backward.  The page prints no formula.
Readings taken (the plainest standard ones):

* "scaled" means one fp32 scale per row (per token, as routing weights in
  a mixture of experts): y[i, j] = s_i * act(x)[i, j]; scales may be absent
  (s_i = 1);
* SReLU(x) = max(x, 0)**2, elementwise, H inputs -> H outputs;
* SwiGLU: a row of 2H inputs splits into a = x[:, :H] (the gated half,
  through SiLU) and b = x[:, H:] (the linear half): act = silu(a) * b,
  silu(a) = a * sigmoid(a), sigmoid(z) = 1 / (1 + exp(-z));
* clamped SwiGLU, with a limit L and a slope alpha given by the caller:
  ac = min(a, L), bc = min(max(b, -L), L), act = ac * sigmoid(alpha * ac) *
  (bc + 1); the clamps pass the gradient where the input is within the
  bounds, bounds included (a <= L; -L <= b <= L);
* backward, with dy [N, H] the gradient of y:
    dx = s_i * dy * act'(x)      (for the GLU forms, the a half and the b
                                  half of the 2H-wide gradient)
    dscales_i = sum_j dy[i, j] * act(x)[i, j]
  dx is rounded once to the dtype of x, dscales to fp32;
* the forward output is y rounded once to the output dtype, or quantized
  from y32 = fp32(y) exactly like the normalization output (FP8 delayed,
  FP8 current, MXFP8 rowwise 1x32 blocks; the columnwise MXFP8 copy is not
  produced for activations).
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_bits, round_to_bf16
from .norm import mx_blocks_1d, quantize

ACTS = ("srelu", "swiglu", "clamped_swiglu")


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def sigmoid(z) -> np.ndarray:
    """1 / (1 + exp(-z)) in fp64, written so that exp never overflows."""
    z = _f64(z)
    e = np.exp(-np.abs(z))
    return np.where(z >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def _split(x, act):
    x = _f64(x)
    if act == "srelu":
        return x, None
    h = x.shape[-1] // 2
    return x[..., :h], x[..., h:]


def act_value(x, act, limit=7.0, alpha=1.702) -> np.ndarray:
    """act(x) per row: [N, H] (SReLU) or [N, 2H] -> [N, H] (GLU forms)."""
    a, b = _split(x, act)
    if act == "srelu":
        return np.maximum(a, 0.0) ** 2
    if act == "swiglu":
        return a * sigmoid(a) * b
    if act == "clamped_swiglu":
        ac = np.minimum(a, limit)
        bc = np.clip(b, -limit, limit)
        return ac * sigmoid(alpha * ac) * (bc + 1.0)
    raise ValueError(act)


def act_grad(x, act, limit=7.0, alpha=1.702):
    """d act / d input, elementwise: (da,) for SReLU, (da, db) for the GLU
    forms (each [N, H])."""
    a, b = _split(x, act)
    if act == "srelu":
        return (2.0 * np.maximum(a, 0.0),)
    if act == "swiglu":
        sg = sigmoid(a)
        return (b * sg * (1.0 + a * (1.0 - sg)), a * sg)
    if act == "clamped_swiglu":
        ac = np.minimum(a, limit)
        bc = np.clip(b, -limit, limit)
        sg = sigmoid(alpha * ac)
        da = np.where(a <= limit, (bc + 1.0) * sg * (1.0 + alpha * ac * (1.0 - sg)), 0.0)
        db = np.where((b >= -limit) & (b <= limit), ac * sg, 0.0)
        return (da, db)
    raise ValueError(act)


def _scales(scales, n):
    return np.ones(n) if scales is None else _f64(scales)


def _out(y, out_dtype):
    if out_dtype == "bf16":
        return bf16_bits(y)
    if out_dtype == "f32":
        return y.astype(np.float32)
    raise ValueError(out_dtype)


def scaled_act_fwd(x, scales, act, mode="none", out_dtype="bf16", limit=7.0, alpha=1.702,
                   scale=None, amax=None) -> dict:
    """y = s_i * act(x)[i, :] -> dict(y (fp64), data, and the quantization
    fields of ``mode``: as the normalization forward; MXFP8 rowwise only)."""
    x = _f64(x)
    y = act_value(x, act, limit, alpha) * _scales(scales, x.shape[0])[:, None]
    res = {"y": y}
    if mode == "none":
        res["data"] = _out(y, out_dtype)
    elif mode == "mxfp8":   # rowwise 1x32 blocks only: N need not be a multiple of 32
        q, sc = mx_blocks_1d(y.astype(np.float32))
        res.update(data=q, row_scales=sc)
    else:
        res.update(quantize(y.astype(np.float32), mode, scale=scale, amax=amax))
    return res


def scaled_act_bwd(dy, x, scales, act, dtype="bf16", limit=7.0, alpha=1.702) -> dict:
    """dx (rounded to ``dtype``; fp64 form dx64) and dscales (fp32; fp64 form
    dscales64)."""
    x = _f64(x)
    dy = _f64(dy)
    s = _scales(scales, x.shape[0])[:, None]
    grads = act_grad(x, act, limit, alpha)
    dx64 = np.concatenate([s * dy * g for g in grads], axis=-1)
    dsc64 = np.sum(dy * act_value(x, act, limit, alpha), axis=-1)
    if dtype == "bf16":
        dx = bf16_bits(dx64)
    elif dtype == "f32":
        dx = dx64.astype(np.float32)
    else:
        raise ValueError(dtype)
    return {"dx": dx, "dx64": dx64, "dscales": dsc64.astype(np.float32), "dscales64": dsc64}


def round_like(v, dtype):
    """Values as the kernel stores them (bf16 rounding or fp32), as fp64."""
    return round_to_bf16(v) if dtype == "bf16" else _f64(v).astype(np.float32).astype(np.float64)
