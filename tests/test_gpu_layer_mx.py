"""GPU parity of the MXFP8 path (block-scaled tcgen05 grouped GEMMs with fused quantise /
transpose epilogues) against the fp64 oracle applying the same operand quantisation,
through the C ABI. Bar: relative Frobenius error <= 3e-2 per output tensor."""
import numpy as np
import pytest
import torch

from grouped_gemm_device_gb300 import synth

from .gpu_helpers import (MX_TOL, LayerRun, Inputs, check_weight_grads_16_byte_aligned, rel_fro,
                          to_np)
from .test_gpu_layer import check_layer

pytestmark = pytest.mark.gpu

MX = dict(precision="mxfp8", align=128)
CASES = {
    "mx_small": synth.LayerConfig("mxs", T=600, E=4, k=2, H=256, F=384, seed=51, **MX),
    # K tail (H = 2.5 k-blocks), F and N1 not multiples of 128, ilv 32
    "mx_tails": synth.LayerConfig("mxt", T=500, E=3, k=2, H=320, F=192, seed=52, ilv=32, **MX),
    # many experts, several empty (Zipf)
    "mx_skewed": synth.LayerConfig("mxk", T=400, E=32, k=4, H=256, F=256, seed=53, zipf_s=1.1,
                                   **MX),
    "mx_clamped": synth.LayerConfig("mxc", T=500, E=8, k=4, H=384, F=320, seed=54, **MX,
                                    activation="clamped_swiglu", beta=1.702, gate_max=7.0,
                                    lin_lo=-7.0, lin_hi=7.0, lin_offset=1.0),
    "mx_geglu": synth.LayerConfig("mxg", T=300, E=4, k=2, H=256, F=256, seed=55,
                                  activation="geglu", **MX),
    "mx_srelu": synth.LayerConfig("mxr", T=300, E=4, k=2, H=256, F=384, seed=56,
                                  activation="srelu", **MX),
}


def test_mx_fc1_output_matches_oracle(lib):
    """The saved FC1 output Z is a pure block-scaled GEMM result (X and W1 quantised along H):
    it isolates the MMA, its scale-factor path and the tile scheduler."""
    cfg = CASES["mx_small"]
    inp = Inputs(cfg)
    ref = inp.oracle(backward=False)
    run = LayerRun(inp, backward=False)
    assert run.layer.device_error() == 0
    off = run.layer.offsets().cpu().numpy()
    assert np.all(off % 128 == 0)
    z = run.unpack_cols(to_np(run.ws("z", torch.bfloat16, cfg.N1)))
    for e in range(cfg.E):
        n = int(ref.perm.counts[e])
        err = rel_fro(z[off[e]:off[e] + n], ref.per_expert[e]["Z"])
        assert err < 4e-3, (e, err)


@pytest.mark.parametrize("name", list(CASES))
def test_mx_layer_fwd_bwd_matches_oracle(lib, name):
    check_layer(CASES[name], tol=MX_TOL)


def test_mx_weight_grads_into_16_byte_aligned_buffers(lib):
    check_weight_grads_16_byte_aligned(CASES["mx_tails"])


def test_mx_cuda_graph_capture_and_replay_with_new_routing(lib):
    """The MXFP8 step (route, the x / dY / weight quantisers, the block-scaled GEMMs with their
    quantising epilogues) has no host sync: capture it once, replay it after overwriting the
    logits in place, and the new routing's layer comes out."""
    cfg = CASES["mx_skewed"]
    run = LayerRun(Inputs(cfg))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            run.run(sync=False)
    lg2 = synth.gen_logits(cfg.with_(seed=97))
    run.logits_d.copy_(torch.from_numpy(lg2))
    graph.replay()
    torch.cuda.synchronize()
    check_layer(cfg, Inputs(cfg, logits=lg2), run, tol=MX_TOL)
    # the replay is the eager step, bit for bit
    got = [t.clone() for t in (run.y, run.dx, run.dw1p, run.dw2, run.d_probs)]
    run.run()
    for a, b in zip(got, (run.y, run.dx, run.dw1p, run.dw2, run.d_probs)):
        assert torch.equal(a, b)


def test_mx_reused_weight_copies(lib):
    """reuse_weights: a second micro-batch that reuses the first forward's MXFP8 weight copies
    gives bit-identical results to one that quantises the weights again."""
    cfg = CASES["mx_clamped"]
    run = LayerRun(Inputs(cfg))
    run.logits_d.copy_(torch.from_numpy(synth.gen_logits(cfg.with_(seed=78))))
    run.run()
    want = [t.clone() for t in (run.y, run.dx, run.dw1p, run.dw2, run.d_probs)]
    run.layer.desc.reuse_weights = 1
    run.run()
    run.layer.desc.reuse_weights = 0
    assert run.layer.device_error() == 0
    for a, b in zip((run.y, run.dx, run.dw1p, run.dw2, run.d_probs), want):
        assert torch.equal(a, b)
