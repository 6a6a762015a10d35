"""bench.py's per-kernel accounting, checked on the CPU: every kernel a step launches has a
name, a byte or flop count and a peak for its operand type, and the counts follow from the
operand sizes (recomputed here from the workload shapes, independently of bench.py)."""
import pytest

import bench
from grouped_gemm_device_gb300 import synth

GEMMS = ("gemm_fc1_fprop", "gemm_fc2_fprop", "gemm_fc2_dgrad", "gemm_fc2_wgrad",
         "gemm_fc1_dgrad", "gemm_fc1_wgrad")


@pytest.mark.parametrize("name", sorted(synth.CONFIGS))
def test_every_timed_kernel_has_bytes_and_flops(name):
    cfg = synth.CONFIGS[name]
    kb = bench.kernel_bytes(cfg)
    gf = bench.gemm_flops(cfg)
    assert set(GEMMS) <= set(kb) and set(GEMMS) == set(gf)
    for k in ("gather_x", "gather_dy", "combine_y", "combine_dx"):
        assert k in kb
    # the launches of repeated kernels are named by their order in a step; each such name
    # has a byte count for the precision that launches it
    for kernel, names in bench.REPEATED.items():
        if kernel.startswith(cfg.precision):
            assert all(n in kb for n in names), (kernel, names)
    assert cfg.precision in bench.TENSOR_RATIO and cfg.precision in bench.DTYPE
    assert sum(gf.values()) == pytest.approx(cfg.flops_fwd_bwd())


def test_nvfp4_bytes_follow_the_operand_sizes():
    cfg = synth.CONFIGS["mixtral_nvfp4"]
    kb = bench.kernel_bytes(cfg)
    R, E, H, F, N1 = cfg.R, cfg.E, cfg.H, cfg.F, cfg.N1
    q = lambda n: n // 2 + n // 16  # noqa: E731  (E2M1 half bytes + one E4M3 scale per 16)
    # FC1: X and W1 copies in, bf16 Z and a_s out
    assert kb["gemm_fc1_fprop"] == q(R * H) + q(E * N1 * H) + 2 * R * N1 + 2 * R * F
    # FC1 weight gradient: the rotated transposed copies of dZ and X in, bf16 dW1 out
    assert kb["gemm_fc1_wgrad"] == q(R * N1) + q(R * H) + 2 * E * N1 * H
    # quantiser: bf16 in, two NVFP4 copies out
    assert kb["nvfp4_quant_w1"] == 2 * E * N1 * H + 2 * q(E * N1 * H)
    assert kb["nvfp4_amax_w2"] == 2 * E * F * H


def test_tensor_peaks_scale_with_the_operand_type():
    assert bench.TENSOR_RATIO["bf16"] == 1.0
    # nominal dense rates: bf16 2.25, fp8 4.5, fp4 13.5 PFLOP/s
    assert bench.TENSOR_RATIO["mxfp8"] == 4.5 / 2.25
    assert bench.TENSOR_RATIO["nvfp4"] == 13.5 / 2.25
