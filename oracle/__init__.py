"""fp64 CPU oracle for fused LayerNorm / RMSNorm with FP8 and MXFP8 output.

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports this package: only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it.  It shares no code with the CUDA path; both take
their inputs from ``rn_inputs``.

What it computes follows the page "Implementation:NVIDIA TransformerEngine
PyTorch Ext Normalization" (sections Description, Signature, I/O Contract):
LayerNorm and RMSNorm forward returning the normalized, optionally quantized
output together with mu (LayerNorm only) and rsigma; backward returning dx,
dgamma and dbeta (LayerNorm only); zero-centered gamma; four output paths
(unfused, fully fused delayed-scaling FP8 / MXFP8, norm+amax then quantize
for current-scaling FP8).  The residual add + norm follows the fused
reduce-scatter + residual add + RMSNorm + all-gather named on the page "NVIDIA
Megatron-Core ... inference_layers" (its single-GPU core).  The formats come from their public definitions:
FP8 E4M3 from the OCP 8-bit floating point specification, MXFP8 block
scaling (E8M0 shared scale over 32 elements) and the FP4 E2M1 element format
from the OCP Microscaling Formats v1.0 specification; NVFP4 (E2M1 elements,
an E4M3 scale per 16 elements, an fp32 tensor scale) from NVIDIA's published
description of that format, the page naming only the FUSED_NORM_AMAX_NVFP4
path.  The pages give no formula for any of this; the
readings taken where they are silent are listed in each function.

Module map:
  formats  E4M3 and E2M1 decode/encode, E8M0 shared exponents, bf16 rounding.
  norm     row statistics, affine apply, quantization stages, backward,
           residual add + norm, the delayed-scaling history step.
  act      scaled SReLU / SwiGLU / clamped SwiGLU forward and backward (the
           page "Activation + GroupedLinear Fusion for MOE ...").

Parity status: every function here is pinned by CPU tests against closed
forms, exact rational arithmetic, finite differences, brute force or
hand-checked format values.  The pages print no worked example for any norm,
so no pin comes from the pages themselves.
"""
from . import act, formats, norm  # noqa: F401
from .formats import (  # noqa: F401
    E4M3_MAX, e4m3_decode, e4m3_encode, e4m3_magnitudes, e8m0_from_amax,
    round_to_bf16, bf16_bits, E2M1_MAX, e2m1_decode, e2m1_encode, e2m1_magnitudes,
    e2m1_pack, e2m1_unpack,
)
from .norm import (  # noqa: F401
    layernorm_stats, rmsnorm_stats, norm_apply, layernorm_fwd, rmsnorm_fwd,
    layernorm_bwd, rmsnorm_bwd, quantize, QUANT_MODES,
    residual_add, rmsnorm_add_fwd, layernorm_add_fwd, amax_history_update,
)
