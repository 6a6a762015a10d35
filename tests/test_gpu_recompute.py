"""GPU parity of the layer with activation recomputation (the forward keeps no FC1 output; the
FC2-dgrad kernel rebuilds it next to dA_s) against the fp64 oracle, and against the same layer
with the saved FC1 output, in BF16, MXFP8 and NVFP4. Same bars as the saved path: relative
Frobenius error <= 5e-3 (BF16) / 3e-2 (MXFP8) / 1e-2 (NVFP4)."""
import numpy as np
import pytest
import torch

import grouped_gemm_device_gb300 as g
from grouped_gemm_device_gb300 import synth

from oracle import moe as om

from .gpu_helpers import BF16_TOL, MX_TOL, LayerRun, Inputs, act_params, rel_fro, to_np
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


NV = dict(precision="nvfp4", align=128)
NV_TOL = 1e-2
NV_CASES = {
    "nv_swiglu": synth.LayerConfig("rnv", T=300, E=4, k=2, H=256, F=256, seed=61, **NV),
    # five 64-column dA tiles (F = 320: W2 rows in both halves of a 128-row scale slab), a
    # K tail (H = 576: two k-blocks of 256 and one MMA of 64)
    "nv_tails": synth.LayerConfig("rnt", T=260, E=3, k=2, H=576, F=320, seed=62, **NV),
    # empty experts and long segments
    "nv_clamped_skew": synth.LayerConfig("rnc", T=300, E=64, k=4, H=256, F=256, seed=63,
                                         zipf_s=1.5, activation="clamped_swiglu", beta=1.702,
                                         gate_max=7.0, lin_lo=-7.0, lin_hi=7.0, lin_offset=1.0,
                                         **NV),
    "nv_geglu": synth.LayerConfig("rng", T=300, E=4, k=2, H=256, F=256, seed=64,
                                  activation="geglu", **NV),
    # not gated (N1 = F): the Z tile is the dA tile's own 64 columns
    "nv_srelu": synth.LayerConfig("rns", T=300, E=4, k=2, H=256, F=384, seed=65,
                                  activation="srelu", **NV),
}


def nv_oracle(cfg, inp, recompute):
    return om.layer_nvfp4(inp.logits, om.bf16_to_f64(inp.x), om.bf16_to_f64(inp.w1),
                          om.bf16_to_f64(inp.w2), cfg.k, act_params(cfg),
                          synth.gen_rht_mask(cfg), dy=om.bf16_to_f64(inp.dy), align=cfg.align,
                          recompute=recompute)


@pytest.mark.parametrize("name", list(NV_CASES))
def test_nvfp4_recompute_layer_matches_oracle(lib, name):
    """NVFP4 with recomputation: the FC2-dgrad kernel runs two block-scaled FP4 GEMMs (dA_s from
    dY and W2, the tile's Z from X and W1, all four from the forward's NVFP4 copies) and forms
    dZ, its amaxes and the routing-weight partials from their fp32 accumulators."""
    cfg = NV_CASES[name]
    inp = Inputs(cfg)
    run = LayerRun(inp, recompute=True)
    assert run.layer.layout.z == 2 ** 64 - 1
    r = nv_oracle(cfg, inp, recompute=True)
    counts = np.bincount(r.ids.ravel(), minlength=cfg.E)
    dZ = run.unpack_cols(to_np(run.ws("dz", torch.bfloat16, cfg.N1)))
    off = r.perm.offsets
    for e in range(cfg.E):
        if counts[e]:
            rows = slice(off[e], off[e] + counts[e])
            assert rel_fro(dZ[rows], r.dZ[e]) < BF16_TOL, e
    am = run.layer.ws_view("nv_amax", torch.float32, (16,)).cpu().numpy().astype(np.float64)
    got = dict(zip(g.NV_AMAX, am))
    for k in ("dz", "dzt"):
        assert abs(got[k] - r.amax[k]) <= 2.0 ** -8 * r.amax[k], k
    errs = {"y": rel_fro(to_np(run.y), r.y), "dx": rel_fro(to_np(run.dx), r.dx),
            "d_probs": rel_fro(to_np(run.d_probs), r.d_probs),
            "dW2": rel_fro(to_np(run.dw2), r.dW2), "dW1": rel_fro(run.dw1_logical(), r.dW1)}
    bad = {k: v for k, v in errs.items() if not v <= NV_TOL}
    assert not bad, bad
    if name == "nv_clamped_skew":
        assert (counts == 0).any()


def test_nvfp4_recompute_forward_equals_saved_path(lib):
    """The forward and FC2's weight gradient (from a_s and dY only) are bit-identical with or
    without the saved Z, and dropping Z shrinks the workspace. The other gradients are not
    compared with each other: a one-ulp change of Z moves some dZ values across an FP4 rounding
    boundary, so each is held to its own oracle reading instead."""
    cfg = NV_CASES["nv_swiglu"]
    inp = Inputs(cfg)
    keep = LayerRun(inp)
    rc = LayerRun(inp, recompute=True)
    assert torch.equal(keep.y, rc.y)
    assert torch.equal(keep.dw2, rc.dw2)
    assert g.moe_workspace_size(keep.desc) > g.moe_workspace_size(rc.desc)
