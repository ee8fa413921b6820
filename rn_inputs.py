"""Seeded synthetic inputs for the normalization and activation workloads.

This module only draws random numbers and stores them in the dtypes the
workloads name.  It holds none of the normalization or quantization
arithmetic: the oracle (CPU, fp64) and the CUDA path both take their inputs
from here and from nowhere else, so that neither depends on the other.

Recipes (one per workload; every draw comes from
``numpy.random.default_rng(seed)`` in the order written below):

* ``rms_small``     RMSNorm fwd+bwd, x bf16 [256 x 1024] ~ N(0,1),
                    gamma fp32 = 1 + 0.1 N(0,1), dz bf16 ~ N(0,1), eps 1e-6,
                    FP8 E4M3 scale fixed at 448/4.
* ``ln_delayed``    LayerNorm fwd+bwd with zero-centered gamma,
                    x bf16 [8192 x 4096] ~ N(mean 0.5, std 2),
                    stored gamma ~ N(0, 0.1), beta ~ N(0, 0.1),
                    dz bf16 ~ N(0,1), eps 1e-5, amax history of 16 values
                    ~ U[3, 6] (the delayed scale is 448 / max(history)).
* ``rms_current``   RMSNorm fwd, x bf16 [16384 x 8192] ~ N(0,1) with
                    ceil(0.001 H) seeded columns multiplied by 50 (so 0.1 %
                    of the entries are outliers, fixed per column),
                    gamma = 1 + 0.05 N(0,1), eps 1e-6.
* ``mxfp8``         LayerNorm / RMSNorm fwd, x bf16 [65536 x 2048] =
                    N(0,1) * c_i with a per-row c_i = 10**U[-2, 2],
                    gamma = 1 + 0.1 N(0,1), beta ~ N(0, 0.1), eps 1e-5.
* ``bwd_f32``       backward, x fp32 [131072 x 1024] ~ N(0,1), dz fp32 ~ N(0,1),
                    gamma = 1 + 0.1 N(0,1), beta ~ N(0, 0.1), eps 1e-5.
* ``bwd_bf16``      backward, x bf16 [3000 x 5120] ~ N(0,1), dz bf16 ~ N(0,1),
                    gamma = 1 + 0.1 N(0,1), beta ~ N(0, 0.1), eps 1e-5.
* ``rms_add``       residual add + RMSNorm (or LayerNorm) fwd, x bf16
                    [8192 x 4096] ~ N(0,1) (a sublayer's output), residual
                    bf16 ~ N(0, 3) (the residual stream), gamma = 1 + 0.1 N(0,1),
                    beta ~ N(0, 0.1), eps 1e-5, FP8 E4M3 scale fixed at 448/8.
* ``moe_act``       scaled activations of a mixture-of-experts MLP (65536
                    tokens, hidden 2048, as in the grouped-MLP measurements
                    the activation page quotes): x bf16 [N x 2H] ~ N(0, 2)
                    (the first fc layer's output: gate half, then linear
                    half), row scales fp32 ~ U[0, 1) (routing weights), dy
                    bf16 [N x H] ~ N(0,1); H = 2048 is the output width.

Every recipe takes optional ``N``/``H`` overrides so that tests can draw the
same distributions at sizes the oracle finishes in seconds.

Storage: a bf16 tensor is returned as its uint16 bit patterns (numpy has no
bf16); ``bf16_bits_to_f32`` decodes them exactly.  Values are drawn in fp64,
cast to fp32 and rounded to bf16 to nearest-even: this is only how the input
values are defined, not part of the method.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload", "make", "WORKLOADS", "bf16_bits_to_f32", "to_bf16_bits",
    "rows_view_f64",
]


def to_bf16_bits(v) -> np.ndarray:
    """fp64/fp32 array -> uint16 bf16 bit patterns (via fp32, ties to even)."""
    f = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    nan = np.isnan(f)
    out = r.astype(np.uint16)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> exact fp32 values."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


@dataclass
class Workload:
    """One seeded workload: arrays in their storage dtypes plus scalars."""
    name: str
    N: int
    H: int
    dtype: str                     # "bf16" or "f32": dtype of x (and dz, dx)
    x: np.ndarray                  # uint16 bits (bf16) or float32, [N, H]
    gamma: np.ndarray              # float32 [H]
    beta: np.ndarray | None        # float32 [H] or None
    dz: np.ndarray | None          # same storage as x, or None
    eps: float
    zero_centered_gamma: bool = False
    scale: float | None = None     # FP8 delayed scale (fp32), when fixed
    amax_history: np.ndarray | None = None  # float32 [16]
    extra: dict = field(default_factory=dict)
    residual: np.ndarray | None = None      # same storage as x (residual add), or None
    scales: np.ndarray | None = None        # float32 [N] row scales (activations), or None

    def x_f64(self, rows=slice(None)) -> np.ndarray:
        return rows_view_f64(self.x, self.dtype, rows)

    def dz_f64(self, rows=slice(None)) -> np.ndarray:
        assert self.dz is not None
        return rows_view_f64(self.dz, self.dtype, rows)

    def residual_f64(self, rows=slice(None)) -> np.ndarray:
        assert self.residual is not None
        return rows_view_f64(self.residual, self.dtype, rows)


def rows_view_f64(a: np.ndarray, dtype: str, rows=slice(None)) -> np.ndarray:
    """Exact fp64 values of (a subset of rows of) a stored array."""
    sub = a[rows]
    if dtype == "bf16":
        return bf16_bits_to_f32(sub).astype(np.float64)
    return np.asarray(sub, dtype=np.float32).astype(np.float64)


def _store(v64: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return to_bf16_bits(v64)
    return np.ascontiguousarray(v64.astype(np.float32))


def _f32(v) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(v, dtype=np.float64).astype(np.float32))


def _rms_small(rng, N, H):
    x = _store(rng.standard_normal((N, H)), "bf16")
    gamma = _f32(1.0 + 0.1 * rng.standard_normal(H))
    dz = _store(rng.standard_normal((N, H)), "bf16")
    return Workload("rms_small", N, H, "bf16", x, gamma, None, dz, 1e-6,
                    scale=float(np.float32(448.0) / np.float32(4.0)))


def _ln_delayed(rng, N, H):
    x = _store(rng.normal(0.5, 2.0, (N, H)), "bf16")
    gamma = _f32(rng.normal(0.0, 0.1, H))
    beta = _f32(rng.normal(0.0, 0.1, H))
    dz = _store(rng.standard_normal((N, H)), "bf16")
    hist = _f32(rng.uniform(3.0, 6.0, 16))
    scale = float(np.float32(448.0) / np.max(hist))
    return Workload("ln_delayed", N, H, "bf16", x, gamma, beta, dz, 1e-5,
                    zero_centered_gamma=True, scale=scale, amax_history=hist)


def _rms_current(rng, N, H):
    n_out = max(1, math.ceil(0.001 * H))
    cols = np.sort(rng.choice(H, size=n_out, replace=False))
    # draw row blocks to bound peak host memory at the full size
    x = np.empty((N, H), dtype=np.uint16)
    step = 2048
    for r0 in range(0, N, step):
        blk = rng.standard_normal((min(step, N - r0), H))
        blk[:, cols] *= 50.0
        x[r0:r0 + blk.shape[0]] = to_bf16_bits(blk)
    gamma = _f32(1.0 + 0.05 * rng.standard_normal(H))
    return Workload("rms_current", N, H, "bf16", x, gamma, None, None, 1e-6,
                    extra={"outlier_cols": cols})


def _mxfp8(rng, N, H):
    c = 10.0 ** rng.uniform(-2.0, 2.0, N)
    x = np.empty((N, H), dtype=np.uint16)
    step = 4096
    for r0 in range(0, N, step):
        n = min(step, N - r0)
        x[r0:r0 + n] = to_bf16_bits(rng.standard_normal((n, H)) * c[r0:r0 + n, None])
    gamma = _f32(1.0 + 0.1 * rng.standard_normal(H))
    beta = _f32(rng.normal(0.0, 0.1, H))
    return Workload("mxfp8", N, H, "bf16", x, gamma, beta, None, 1e-5,
                    extra={"row_scale": c})


def _bwd(rng, N, H, dtype, name):
    x = np.empty((N, H), dtype=np.uint16 if dtype == "bf16" else np.float32)
    dz = np.empty_like(x)
    step = 8192
    for r0 in range(0, N, step):
        n = min(step, N - r0)
        x[r0:r0 + n] = _store(rng.standard_normal((n, H)), dtype)
    for r0 in range(0, N, step):
        n = min(step, N - r0)
        dz[r0:r0 + n] = _store(rng.standard_normal((n, H)), dtype)
    gamma = _f32(1.0 + 0.1 * rng.standard_normal(H))
    beta = _f32(rng.normal(0.0, 0.1, H))
    return Workload(name, N, H, dtype, x, gamma, beta, dz, 1e-5)


def _rms_add(rng, N, H):
    x = _store(rng.standard_normal((N, H)), "bf16")
    residual = _store(rng.normal(0.0, 3.0, (N, H)), "bf16")
    gamma = _f32(1.0 + 0.1 * rng.standard_normal(H))
    beta = _f32(rng.normal(0.0, 0.1, H))
    return Workload("rms_add", N, H, "bf16", x, gamma, beta, None, 1e-5,
                    scale=float(np.float32(448.0) / np.float32(8.0)), residual=residual)


def _moe_act(rng, N, H):
    x = np.empty((N, 2 * H), dtype=np.uint16)
    step = 8192
    for r0 in range(0, N, step):
        n = min(step, N - r0)
        x[r0:r0 + n] = to_bf16_bits(rng.normal(0.0, 2.0, (n, 2 * H)))
    scales = _f32(rng.uniform(0.0, 1.0, N))
    dy = np.empty((N, H), dtype=np.uint16)
    for r0 in range(0, N, step):
        n = min(step, N - r0)
        dy[r0:r0 + n] = to_bf16_bits(rng.standard_normal((n, H)))
    return Workload("moe_act", N, H, "bf16", x, np.ones(0, np.float32), None, dy, 0.0,
                    scales=scales)


WORKLOADS = {
    "rms_small": ((256, 1024), _rms_small),
    "ln_delayed": ((8192, 4096), _ln_delayed),
    "rms_current": ((16384, 8192), _rms_current),
    "mxfp8": ((65536, 2048), _mxfp8),
    "bwd_f32": ((131072, 1024), lambda rng, N, H: _bwd(rng, N, H, "f32", "bwd_f32")),
    "bwd_bf16": ((3000, 5120), lambda rng, N, H: _bwd(rng, N, H, "bf16", "bwd_bf16")),
    "rms_add": ((8192, 4096), _rms_add),
    "moe_act": ((65536, 2048), _moe_act),
}


def make(name: str, N: int | None = None, H: int | None = None, seed: int = 0) -> Workload:
    """Draw workload ``name`` (full size unless N/H given) from ``seed``."""
    (n0, h0), fn = WORKLOADS[name]
    rng = np.random.default_rng(seed)
    return fn(rng, n0 if N is None else N, h0 if H is None else H)
