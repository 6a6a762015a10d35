"""Degenerate inputs through the C ABI, every precision: a step with no tokens (every weight
gradient is an exact zero, nothing is written for the absent tokens, no device error) and,
for NVFP4, a single token (all per-tensor amaxes then come from one row)."""
import numpy as np
import pytest
import torch

from grouped_gemm_device_gb300 import synth
from oracle import moe as om

from .gpu_helpers import LayerRun, Inputs, act_params, rel_fro, to_np

pytestmark = pytest.mark.gpu


def _cfg(prec, T):
    return synth.LayerConfig(f"edge_{prec}_{T}", T=T, E=4, k=2, H=128, F=128, precision=prec,
                             align=32 if prec == "bf16" else 128, seed=21)


@pytest.mark.parametrize("prec", ["bf16", "mxfp8", "nvfp4"])
def test_step_with_no_tokens(lib, prec):
    run = LayerRun(Inputs(_cfg(prec, 0)), T_max=64)
    assert run.y.shape[0] == 0 and run.dx.shape[0] == 0 and run.d_probs.shape[0] == 0
    assert not run.dw1p.any() and not run.dw2.any()
    assert torch.isfinite(run.dw1p.float()).all() and torch.isfinite(run.dw2.float()).all()
    assert run.layer.device_error() == 0


def test_nvfp4_single_token(lib):
    cfg = _cfg("nvfp4", 1)
    inp = Inputs(cfg)
    run = LayerRun(inp, T_max=64)
    r = om.layer_nvfp4(inp.logits, om.bf16_to_f64(inp.x), om.bf16_to_f64(inp.w1),
                       om.bf16_to_f64(inp.w2), cfg.k, act_params(cfg), synth.gen_rht_mask(cfg),
                       dy=om.bf16_to_f64(inp.dy), align=cfg.align)
    for got, want in ((to_np(run.y), r.y), (to_np(run.dx), r.dx), (to_np(run.d_probs), r.d_probs),
                      (to_np(run.dw2), r.dW2), (run.dw1_logical(), r.dW1)):
        assert rel_fro(got, want) < 1e-2
    # the experts the token does not use get exact zeros
    unused = np.setdiff1d(np.arange(cfg.E), r.ids[0])
    assert not to_np(run.dw2)[unused].any()
