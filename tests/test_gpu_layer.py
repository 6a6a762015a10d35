"""GPU parity of the fused grouped MLP (route -> FC1+GLU -> FC2 -> combine, and the backward)
against the fp64 oracle through the C ABI, at sizes that span several 128x256 tiles with
ragged expert segments, N and K tails, empty experts and every activation."""
import numpy as np
import pytest
import torch

from grouped_gemm_device_gb300 import synth

from .gpu_helpers import (BF16_TOL, LayerRun, Inputs, check_weight_grads_16_byte_aligned, rel_fro,
                          to_np)

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": synth.CONFIGS["tiny"],
    # several M and N tiles per expert, ragged counts
    "multi_tile": synth.LayerConfig("mt", T=1000, E=4, k=2, H=512, F=768, seed=31),
    # N1 = 2F not a multiple of 256, H not a multiple of 256 (N tails), K tail of 64
    "tails": synth.LayerConfig("tl", T=700, E=6, k=2, H=320, F=320, seed=32, ilv=32),
    # many small experts, some empty (Zipf skew)
    "skewed": synth.LayerConfig("sk", T=600, E=64, k=4, H=256, F=256, seed=33, zipf_s=1.1),
    "clamped": synth.LayerConfig("cl", T=800, E=8, k=4, H=384, F=384, seed=34,
                                 activation="clamped_swiglu", beta=1.702, gate_max=7.0,
                                 lin_lo=-7.0, lin_hi=7.0, lin_offset=1.0),
    "geglu": synth.LayerConfig("ge", T=500, E=4, k=2, H=256, F=512, seed=35, activation="geglu",
                               ilv=128),
    "srelu": synth.LayerConfig("sr", T=500, E=4, k=2, H=256, F=384, seed=36, activation="srelu"),
    "single_expert": synth.LayerConfig("one", T=300, E=1, k=1, H=256, F=256, seed=37),
    # >= 1024 routed rows per expert at capacity: the FC2-dgrad + dGLU kernel runs on CTA pairs
    "large_experts": synth.LayerConfig("lg", T=2100, E=2, k=1, H=256, F=512, seed=38),
}


def check_layer(cfg, inp=None, run=None, tol=BF16_TOL, recompute=False):
    inp = inp or Inputs(cfg)
    ref = inp.oracle(recompute=recompute)
    run = run or LayerRun(inp)
    assert run.layer.device_error() == 0
    errs = {"y": rel_fro(to_np(run.y), ref.y), "dx": rel_fro(to_np(run.dx), ref.dx),
            "d_probs": rel_fro(to_np(run.d_probs), ref.d_probs)}
    dw1 = run.dw1_logical()
    dw2 = to_np(run.dw2)
    for e in range(cfg.E):
        if ref.perm.counts[e] == 0:
            assert np.all(dw1[e] == 0) and np.all(dw2[e] == 0), f"expert {e} not zero"
            continue
        errs[f"dW1[{e}]"] = rel_fro(dw1[e], ref.dW1[e])
        errs[f"dW2[{e}]"] = rel_fro(dw2[e], ref.dW2[e])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, (bad, max(errs.values()))
    return run, ref, errs


@pytest.mark.parametrize("name", list(CASES))
def test_layer_fwd_bwd_matches_oracle(lib, name):
    check_layer(CASES[name])


def test_saved_intermediates_match_oracle(lib):
    cfg = CASES["multi_tile"]
    inp = Inputs(cfg)
    ref = inp.oracle()
    run = LayerRun(inp)
    off = run.layer.offsets().cpu().numpy()
    z = run.unpack_cols(to_np(run.ws("z", torch.bfloat16, cfg.N1)))
    a_s = to_np(run.ws("a_s", torch.bfloat16, cfg.F))
    dz = run.unpack_cols(to_np(run.ws("dz", torch.bfloat16, cfg.N1)))
    for e in range(cfg.E):
        n = int(ref.perm.counts[e])
        seg = slice(off[e], off[e] + n)
        pad = slice(off[e] + n, off[e + 1])
        d = ref.per_expert[e]
        assert rel_fro(z[seg], d["Z"]) < 4e-3
        assert rel_fro(a_s[seg], d["a_s"]) < BF16_TOL
        assert rel_fro(dz[seg], d["dZ"]) < BF16_TOL
        assert np.all(a_s[pad] == 0) and np.all(dz[pad] == 0) and np.all(z[pad] == 0)


def test_weight_grads_into_16_byte_aligned_buffers(lib):
    check_weight_grads_16_byte_aligned(CASES["multi_tile"])


def test_sm_margin_and_rerun_are_deterministic(lib):
    cfg = CASES["multi_tile"]
    inp = Inputs(cfg)
    r1 = LayerRun(inp, sm_margin=0)
    r2 = LayerRun(inp, sm_margin=100)
    assert torch.equal(r1.y, r2.y) and torch.equal(r1.dx, r2.dx)
    assert torch.equal(r1.dw1p, r2.dw1p) and torch.equal(r1.dw2, r2.dw2)
    assert torch.equal(r1.d_probs, r2.d_probs)
    y0 = r1.y.clone()
    r1.run()
    assert torch.equal(r1.y, y0)


def test_cuda_graph_capture_and_replay_with_new_routing(lib):
    """The whole layer step (route, fwd, bwd) has no host sync: capture it once, then replay
    it after overwriting the logits in place - the new routing must be used."""
    cfg = CASES["skewed"]
    inp = Inputs(cfg)
    run = LayerRun(inp)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            run.run(sync=False)
    lg2 = synth.gen_logits(cfg.with_(seed=99))
    run.logits_d.copy_(torch.from_numpy(lg2))
    graph.replay()
    torch.cuda.synchronize()
    inp2 = Inputs(cfg, logits=lg2)
    check_layer(cfg, inp2, run)


@pytest.mark.parametrize("prec", ["bf16", "mxfp8", "nvfp4"])
def test_programmatic_dependent_launch_gives_identical_steps(lib, prec):
    """desc.pdl = 1 launches every kernel with programmatic stream serialization; each kernel
    waits for its predecessor before touching memory, so the step is bit-identical to the
    ordinary stream order, eagerly and replayed from a CUDA graph."""
    kw = dict(precision=prec, align=128) if prec != "bf16" else {}
    cfg = synth.LayerConfig("pdl", T=700, E=8, k=2, H=256, F=256, seed=61, zipf_s=1.1, **kw)
    run = LayerRun(Inputs(cfg))
    want = [t.clone() for t in (run.y, run.dx, run.dw1p, run.dw2, run.d_probs)]
    run.layer.desc.pdl = 1
    run.run()
    assert run.layer.device_error() == 0
    for a, b in zip((run.y, run.dx, run.dw1p, run.dw2, run.d_probs), want):
        assert torch.equal(a, b)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            run.run(sync=False)
    for t in (run.y, run.dx, run.dw1p, run.dw2, run.d_probs):
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for a, b in zip((run.y, run.dx, run.dw1p, run.dw2, run.d_probs), want):
        assert torch.equal(a, b)
