"""GPU parity of the epilogue extras (an FC1 bias added before the activation and a
per-feature scale of the activation output, with their gradients) against the fp64 oracle,
through moe_grouped_mlp_fwd_ex / moe_grouped_mlp_bwd_ex, for BF16, MXFP8 and NVFP4 layers.
Bar: relative Frobenius error <= 5e-3 (BF16) / 3e-2 (MXFP8) / 1e-2 (NVFP4, against the
NVFP4 oracle) per output tensor, as for the plain layers."""
import numpy as np
import pytest
import torch

import grouped_gemm_device_gb300 as g
from grouped_gemm_device_gb300 import synth
from oracle import moe as om

from .gpu_helpers import BF16_TOL, MX_TOL, Inputs, act_params, bf16_dev, rel_fro, to_np

pytestmark = pytest.mark.gpu

CASES = {
    "multi_tile": synth.LayerConfig("xmt", T=1000, E=4, k=2, H=512, F=768, seed=61),
    # F tail against 256-column tiles, ilv 32, ragged experts
    "tails": synth.LayerConfig("xtl", T=700, E=6, k=2, H=320, F=320, seed=62, ilv=32),
    # many small experts, 23 of 64 empty (Zipf skew)
    "skewed": synth.LayerConfig("xsk", T=300, E=64, k=4, H=256, F=256, seed=63, zipf_s=1.1),
    "clamped": synth.LayerConfig("xcl", T=800, E=8, k=4, H=384, F=384, seed=64,
                                 activation="clamped_swiglu", beta=1.702, gate_max=7.0,
                                 lin_lo=-7.0, lin_hi=7.0, lin_offset=1.0),
    "geglu": synth.LayerConfig("xge", T=500, E=4, k=2, H=256, F=512, seed=65,
                               activation="geglu", ilv=128),
    # >= 1024 routed rows per expert: the dGLU epilogue with the extras on CTA pairs
    "large_experts": synth.LayerConfig("xlg", T=2100, E=2, k=1, H=256, F=384, seed=71),
}
MX = dict(precision="mxfp8", align=128)
MX_CASES = {
    "mx_multi_tile": synth.LayerConfig("xmm", T=700, E=4, k=2, H=256, F=384, seed=66, **MX),
    # ilv 32, F and N1 not multiples of 256
    "mx_tails": synth.LayerConfig("xmt", T=500, E=3, k=2, H=320, F=192, seed=67, ilv=32, **MX),
    # many experts, 25 of 64 empty
    "mx_skewed": synth.LayerConfig("xms", T=300, E=64, k=4, H=256, F=256, seed=68, zipf_s=1.1,
                                   **MX),
    "mx_clamped": synth.LayerConfig("xmc", T=500, E=8, k=4, H=384, F=320, seed=69,
                                    activation="clamped_swiglu", beta=1.702, gate_max=7.0,
                                    lin_lo=-7.0, lin_hi=7.0, lin_offset=1.0, **MX),
    "mx_geglu": synth.LayerConfig("xmg", T=300, E=4, k=2, H=256, F=256, seed=70,
                                  activation="geglu", **MX),
}


NV = dict(precision="nvfp4", align=128)
NV_CASES = {
    "nv_swiglu": synth.LayerConfig("xnv", T=300, E=4, k=2, H=256, F=256, seed=81, **NV),
    # ragged: F = 320 (a 256 + 64 split of the dGLU's 128-column tiles), several k-blocks
    "nv_geglu": synth.LayerConfig("xng", T=260, E=4, k=2, H=576, F=320, seed=82,
                                  activation="geglu", **NV),
    # skewed routing with empty experts
    "nv_clamped": synth.LayerConfig("xnc", T=300, E=64, k=4, H=256, F=256, seed=83,
                                    zipf_s=1.5, activation="clamped_swiglu", beta=1.702,
                                    gate_max=7.0, lin_lo=-7.0, lin_hi=7.0, lin_offset=1.0,
                                    **NV),
}
NV_TOL = 1e-2


def run_extras(cfg, extras):
    inp = Inputs(cfg)
    b1 = synth.gen_fc1_bias(cfg) if extras & g.EXTRA_BIAS else None
    sc = synth.gen_feat_scale(cfg) if extras & g.EXTRA_SCALE else None
    mx = cfg.precision == "mxfp8"
    nv = cfg.precision == "nvfp4"
    tol = MX_TOL if mx else NV_TOL if nv else BF16_TOL
    b64 = None if b1 is None else b1.astype(np.float64)
    s64 = None if sc is None else sc.astype(np.float64)
    if nv:
        ref = om.layer_nvfp4(inp.logits, om.bf16_to_f64(inp.x), om.bf16_to_f64(inp.w1),
                             om.bf16_to_f64(inp.w2), cfg.k, act_params(cfg),
                             synth.gen_rht_mask(cfg), dy=om.bf16_to_f64(inp.dy),
                             align=cfg.align, b1=b64, s=s64)
    else:
        ref = om.layer(inp.logits, om.bf16_to_f64(inp.x), om.bf16_to_f64(inp.w1),
                       om.bf16_to_f64(inp.w2), cfg.k, act_params(cfg), mx=mx, align=cfg.align,
                       dy=om.bf16_to_f64(inp.dy), b1=b64, s=s64)
    layer = g.MoELayer(g.desc_from_config(cfg, extras=extras))
    w1p = g.pack_w1(bf16_dev(inp.w1), gated=True, ilv=cfg.ilv)
    w2 = bf16_dev(inp.w2)
    bt = None if b1 is None else torch.from_numpy(b1).cuda()
    st = None if sc is None else torch.from_numpy(sc).cuda()
    layer.route_permute(torch.from_numpy(inp.logits).cuda(), bf16_dev(inp.x), cfg.T)
    y = layer.forward(w1p, w2, cfg.T, fc1_bias=bt, feat_scale=st)
    dx, dw1p, dw2, dp = layer.backward(bf16_dev(inp.dy), w1p, w2, cfg.T, feat_scale=st)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    dw1 = torch.empty(cfg.E, cfg.H, cfg.N1, dtype=torch.bfloat16, device="cuda")
    g.moe_pack_fc1_weight(dw1p, dw1, cfg.E, cfg.H, cfg.F, 1, cfg.ilv, 1)
    torch.cuda.synchronize()
    errs = {"y": rel_fro(to_np(y), ref.y), "dx": rel_fro(to_np(dx), ref.dx),
            "d_probs": rel_fro(to_np(dp), ref.d_probs)}
    dw1, dw2 = to_np(dw1), to_np(dw2)
    if nv:  # the NVFP4 oracle returns stacked weight gradients (zeros for empty experts)
        errs["dW1"] = rel_fro(dw1, ref.dW1)
        errs["dW2"] = rel_fro(dw2, ref.dW2)
    for e in range(cfg.E if not nv else 0):
        if ref.perm.counts[e] == 0:
            continue
        errs[f"dW1[{e}]"] = rel_fro(dw1[e], ref.dW1[e])
        errs[f"dW2[{e}]"] = rel_fro(dw2[e], ref.dW2[e])
    if b1 is not None:
        errs["d_fc1_bias"] = rel_fro(layer.d_fc1_bias.cpu().numpy(), ref.db1)
    if sc is not None:
        errs["d_feat_scale"] = rel_fro(layer.d_feat_scale.cpu().numpy(), ref.ds)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, (bad, max(errs.values()))
    return layer, ref


@pytest.mark.parametrize("name", list(CASES))
def test_bias_and_feature_scale_match_oracle(lib, name):
    run_extras(CASES[name], g.EXTRA_BIAS | g.EXTRA_SCALE)


@pytest.mark.parametrize("extras", [g.EXTRA_BIAS, g.EXTRA_SCALE])
def test_each_extra_alone_matches_oracle(lib, extras):
    run_extras(CASES["tails"], extras)


@pytest.mark.parametrize("name", list(MX_CASES))
def test_mx_bias_and_feature_scale_match_oracle(lib, name):
    run_extras(MX_CASES[name], g.EXTRA_BIAS | g.EXTRA_SCALE)


@pytest.mark.parametrize("extras", [g.EXTRA_BIAS, g.EXTRA_SCALE])
def test_mx_each_extra_alone_matches_oracle(lib, extras):
    run_extras(MX_CASES["mx_tails"], extras)


@pytest.mark.parametrize("name", list(NV_CASES))
def test_nvfp4_bias_and_feature_scale_match_oracle(lib, name):
    run_extras(NV_CASES[name], g.EXTRA_BIAS | g.EXTRA_SCALE)


@pytest.mark.parametrize("extras", [g.EXTRA_BIAS, g.EXTRA_SCALE])
def test_nvfp4_each_extra_alone_matches_oracle(lib, extras):
    run_extras(NV_CASES["nv_geglu"], extras)


@pytest.mark.parametrize("cfg", [CASES["skewed"], MX_CASES["mx_skewed"],
                                 NV_CASES["nv_clamped"]], ids=["bf16", "mxfp8", "nvfp4"])
def test_empty_expert_extras_gradients_are_zero(lib, cfg):
    layer, ref = run_extras(cfg, g.EXTRA_BIAS | g.EXTRA_SCALE)
    empty = np.nonzero(ref.perm.counts == 0)[0]
    assert len(empty) > 0
    assert np.all(layer.d_fc1_bias.cpu().numpy()[empty] == 0)
    assert np.all(layer.d_feat_scale.cpu().numpy()[empty] == 0)


def test_plain_entry_points_reject_a_layer_with_extras(lib):
    layer = g.MoELayer(g.desc_from_config(CASES["tails"], extras=g.EXTRA_BIAS))
    with pytest.raises(g.MoeError) as e:
        g.moe_grouped_mlp_fwd(layer.desc, 0, layer.ws, layer.ws, layer.y, layer.ws,
                              layer.ws_bytes)
    assert e.value.status == 2
