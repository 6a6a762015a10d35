"""GPU parity of the layer with activation recomputation (the forward keeps no FC1 output; the
FC2-dgrad kernel rebuilds it next to dA_s) against the fp64 oracle, and against the same layer
with the saved FC1 output, in BF16 and MXFP8. Same bars as the saved path: relative Frobenius
error <= 5e-3 (BF16) / 3e-2 (MXFP8)."""
import numpy as np
import pytest
import torch

import grouped_gemm_device_gb300 as g
from grouped_gemm_device_gb300 import synth

from .gpu_helpers import BF16_TOL, MX_TOL, LayerRun, Inputs, rel_fro, to_np
from .test_gpu_layer import check_layer

pytestmark = pytest.mark.gpu

CASES = {
    "multi_tile": synth.LayerConfig("rmt", T=1000, E=4, k=2, H=512, F=768, seed=41),
    # F and 2F tails against the 128-column dA tiles, ilv 32
    "tails": synth.LayerConfig("rtl", T=700, E=6, k=2, H=320, F=320, seed=42, ilv=32),
    "skewed": synth.LayerConfig("rsk", T=600, E=64, k=4, H=256, F=256, seed=43, zipf_s=1.1),
    "clamped": synth.LayerConfig("rcl", T=800, E=8, k=4, H=384, F=384, seed=44,
                                 activation="clamped_swiglu", beta=1.702, gate_max=7.0,
                                 lin_lo=-7.0, lin_hi=7.0, lin_offset=1.0),
    "geglu_ilv128": synth.LayerConfig("rge", T=500, E=4, k=2, H=256, F=512, seed=45,
                                      activation="geglu", ilv=128),
    # not gated (N1 = F): the Z tile is the dA tile's own 128 columns; F tail of 64
    "srelu": synth.LayerConfig("rsr", T=600, E=5, k=2, H=384, F=448, seed=46,
                               activation="srelu"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_recompute_layer_matches_oracle(lib, name):
    cfg = CASES[name]
    inp = Inputs(cfg)
    run = LayerRun(inp, recompute=True)
    assert run.layer.layout.z == 2 ** 64 - 1
    check_layer(cfg, inp=inp, run=run)


def test_recompute_agrees_with_saved_z(lib):
    """Same inputs, both ways: forward outputs and dW2 (which reads a_s and dY only) are
    identical; the rest differs by the saved Z's bf16 rounding against the recomputed fp32 Z.
    Each path is within 5e-3 of the oracle, so they are within 2 x 5e-3 of each other."""
    cfg = CASES["multi_tile"]
    inp = Inputs(cfg)
    keep = LayerRun(inp)
    rc = LayerRun(inp, recompute=True)
    assert torch.equal(keep.y, rc.y)
    assert torch.equal(keep.dw2, rc.dw2)
    for a, b in ((rc.dx, keep.dx), (rc.d_probs, keep.d_probs), (rc.dw1p, keep.dw1p)):
        assert rel_fro(to_np(a), to_np(b)) < 2 * BF16_TOL
    ws_keep = g.moe_workspace_size(keep.desc)
    ws_rc = g.moe_workspace_size(rc.desc)
    assert ws_keep - ws_rc >= keep.layer.layout.R_cap * cfg.N1 * 2 - (1 << 20)


MX = dict(precision="mxfp8", align=128)
MX_CASES = {
    "mx_multi_tile": synth.LayerConfig("rmm", T=700, E=4, k=2, H=256, F=384, seed=46, **MX),
    # K tail (H = 2.5 k-blocks of 128), F and N1 tails, ilv 32
    "mx_tails": synth.LayerConfig("rmx", T=500, E=3, k=2, H=320, F=192, seed=47, ilv=32, **MX),
    "mx_skewed": synth.LayerConfig("rms", T=400, E=32, k=4, H=256, F=256, seed=48, zipf_s=1.1,
                                   **MX),
    "mx_clamped": synth.LayerConfig("rmc", T=500, E=8, k=4, H=384, F=320, seed=49,
                                    activation="clamped_swiglu", beta=1.702, gate_max=7.0,
                                    lin_lo=-7.0, lin_hi=7.0, lin_offset=1.0, **MX),
    "mx_geglu": synth.LayerConfig("rmg", T=300, E=4, k=2, H=256, F=256, seed=50,
                                  activation="geglu", **MX),
    # not gated (N1 = F): a 128-column Z tile, one W1 box and scale slab; F tail of 64
    "mx_srelu": synth.LayerConfig("rmr", T=400, E=4, k=2, H=320, F=320, seed=51,
                                  activation="srelu", **MX),
}


@pytest.mark.parametrize("name", list(MX_CASES))
def test_mx_recompute_layer_matches_oracle(lib, name):
    """MXFP8 with recomputation: the FC2-dgrad kernel runs two block-scaled GEMMs (dA_s and the
    tile's Z) and quantises dZ from their fp32 accumulators."""
    cfg = MX_CASES[name]
    inp = Inputs(cfg)
    run = LayerRun(inp, recompute=True)
    assert run.layer.layout.z == 2 ** 64 - 1
    check_layer(cfg, inp=inp, run=run, tol=MX_TOL, recompute=True)


def test_mx_recompute_forward_equals_saved_path(lib):
    """The forward and FC2's weight gradient (a_s and dY only) are the same with or without the
    saved Z; the other gradients each meet the bar against their own oracle reading."""
    cfg = MX_CASES["mx_multi_tile"]
    inp = Inputs(cfg)
    keep = LayerRun(inp)
    rc = LayerRun(inp, recompute=True)
    assert torch.equal(keep.y, rc.y)
    assert torch.equal(keep.dw2, rc.dw2)
