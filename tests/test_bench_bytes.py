"""CPU pins of the benchmark's algorithmic byte counts (the numerators of
every GB/s figure): each kind against the bytes its call must move at
least once, counted by hand from the tensors it reads and writes."""
import bench


def test_norm_forward_and_backward_bytes():
    N, H = 8192, 4096
    E = N * H
    # LayerNorm fwd FP8 delayed, bf16: x in (2E), codes out (E), gamma + beta
    # (8H), mu + rsigma (8N)
    assert bench.algorithmic_bytes("fwd_fp8", N, H, 2, True) == 2 * E + E + 8 * H + 8 * N
    # backward: dz, x in and dx out (3 x 2E), mu + rsigma in (8N), gamma in
    # (4H), dgamma + dbeta out (8H)
    assert bench.algorithmic_bytes("bwd", N, H, 2, True) == 6 * E + 8 * N + 12 * H
    # the headline step is their sum
    assert (bench.algorithmic_bytes("fwd_fp8", N, H, 2, True) + bench.algorithmic_bytes("bwd", N, H, 2, True)
            == 302202880)


def test_quantized_forward_bytes():
    N, H = 65536, 2048
    E = N * H
    # MXFP8: x in, rowwise + columnwise codes, one E8M0 byte per 32 each way
    assert bench.algorithmic_bytes("fwd_mxfp8", N, H, 2, True) == 2 * E + 2 * E + 2 * (E // 32) + 8 * H + 8 * N
    assert bench.algorithmic_bytes("fwd_mxfp8_row", N, H, 2, True) == 2 * E + E + E // 32 + 8 * H + 8 * N
    N, H = 16384, 8192
    E = N * H
    # current scaling and NVFP4 read x twice (amax pass, quantize pass) and
    # write / read rsigma once each; RMSNorm has gamma only
    assert bench.algorithmic_bytes("fwd_fp8_current", N, H, 2, False) == 4 * E + E + 4 * H + 8 * N
    assert bench.algorithmic_bytes("fwd_nvfp4", N, H, 2, False) == 4 * E + E // 2 + E // 16 + 4 * H + 8 * N


def test_activation_and_residual_bytes():
    N, H = 65536, 2048
    E = N * H
    # SwiGLU reads 2E inputs per E outputs; row scales 4N
    assert bench.algorithmic_bytes("act_fwd_none", N, H, 2, False) == 4 * E + 2 * E + 4 * N
    assert bench.algorithmic_bytes("act_bwd", N, H, 2, False) == 2 * E + 4 * E + 4 * E + 8 * N
    N, H = 8192, 4096
    E = N * H
    # residual add + FP8: x, residual in, h out, codes out
    assert bench.algorithmic_bytes("fwd_add_fp8", N, H, 2, False) == 6 * E + E + 4 * H + 4 * N
    # the same add with MXFP8 in both directions: two code bytes and two
    # E8M0 bytes per 32 elements instead of one code byte
    assert bench.algorithmic_bytes("fwd_add_mxfp8", N, H, 2, False) == 6 * E + 2 * E + 2 * (E // 32) + 4 * H + 4 * N
