"""GPU parity of the NVFP4 path through the C ABI: the quantiser (codes and scale bytes against
the oracle, bit-exact where the value it encodes is the exact bf16 input), the per-tensor amax
kernels, and the NVFP4 layer (outputs, weight gradients, the BF16 intermediates the fused
kernels emit and every per-tensor amax) against oracle.moe.layer_nvfp4.

Tolerances. The kernel and the oracle quantise identical bf16 values with identical fp32
scaling steps, so their codes agree; what differs is (a) the order of the fp32 accumulation in
the tensor cores against fp64 (about 1e-6 relative), (b) bf16 rounding of the outputs and
stored intermediates (2^-9 relative at most) and (c) rare quantisation decisions that flip
because a value computed from (a) sits within an fp32 ulp of a rounding boundary; each flip
moves one value by one E2M1 step (at most a third of it) or one block by one E4M3 scale step
(an eighth), on far fewer than 1e-3 of the values. Outputs therefore agree to NV_TOL = 1e-2
relative (Frobenius), BF16 intermediates to BF16_TOL; NVFP4's own quantisation error, which
a wrong code, scale or layout would show, is about 0.2 on these layers."""
import numpy as np
import pytest
import torch

import grouped_gemm_device_gb300 as g
from grouped_gemm_device_gb300 import synth
from oracle import moe as om
from oracle import mxfp8 as omx
from oracle import nvfp4 as nv

from .gpu_helpers import BF16_TOL, LayerRun, Inputs, act_params, bf16_dev, rel_fro, to_np

pytestmark = pytest.mark.gpu

NV_TOL = 1e-2


def unpack_codes(q: np.ndarray) -> np.ndarray:
    """[rows, n/2] bytes -> [rows, n] E2M1 codes (even index in the low nibble)."""
    out = np.empty((q.shape[0], 2 * q.shape[1]), dtype=np.uint8)
    out[:, 0::2] = q & 0xF
    out[:, 1::2] = q >> 4
    return out


def slab_scales(s: np.ndarray, rows: int, nblk: int, pad: int) -> np.ndarray:
    """Scale bytes [rows, nblk] read from the documented slab layout."""
    r = np.arange(rows)[:, None]
    j = np.arange(nblk)[None, :]
    perm = (r & ~127) | ((r & 31) << 2) | ((r >> 5) & 3)
    return s[((j >> 2) * pad + perm) * 4 + (j & 3)]


def _quantize(x, M, N, amax_row, amax_col, rht, mask):
    q_row = torch.zeros(M, N // 2, dtype=torch.uint8, device="cuda")
    s_row = torch.zeros((N // 64) * M * 4, dtype=torch.uint8, device="cuda")
    Np = -(-N // 128) * 128
    q_col = torch.zeros(N, M // 2, dtype=torch.uint8, device="cuda")
    s_col = torch.zeros((M // 64) * Np * 4, dtype=torch.uint8, device="cuda")
    a_r = torch.tensor([amax_row], dtype=torch.float32, device="cuda")
    a_c = torch.tensor([amax_col], dtype=torch.float32, device="cuda")
    g.nvfp4_quantize(x, M, N, a_r, a_c, rht, mask, q_row, s_row, q_col, s_col)
    torch.cuda.synchronize()
    return (unpack_codes(q_row.cpu().numpy()), slab_scales(s_row.cpu().numpy(), M, N // 16, M),
            unpack_codes(q_col.cpu().numpy()), slab_scales(s_col.cpu().numpy(), N, M // 16, Np))


@pytest.mark.parametrize("M,N,scale,outliers", [
    (128, 64, 1.0, 0), (256, 192, 3.0, 8), (384, 2880, 0.02, 16), (128, 4096, 1e-30, 4),
    (256, 128, 1e25, 8),
])
def test_nvfp4_quantize_bit_exact(lib, M, N, scale, outliers):
    a = synth.gen_bf16_matrix(M * 5 + N, M, N, scale=scale, outlier_rows=outliers)
    v = om.bf16_to_f64(a)
    am = nv.amax(v)
    cr, sr, cc, sc = _quantize(bf16_dev(a), M, N, am, am, 0, 0)
    S = nv.encode_scale(am)
    c_r, sb_r = nv.quantize_blocks(v, 1, S)
    c_c, sb_c = nv.quantize_blocks(v, 0, S)
    assert np.array_equal(sr, omx.e4m3_encode(sb_r))
    assert np.array_equal(cr, c_r)
    assert np.array_equal(sc, omx.e4m3_encode(sb_c).T)
    assert np.array_equal(cc, c_c.T)


def test_nvfp4_quantize_blocks_with_subnormal_maxima(lib):
    """Blocks whose maximum m is below 2^-125, so that fp32(m / 6) is subnormal, with a tensor
    amax that makes S large enough for those blocks to get non-zero E4M3 scales (and small
    enough that fp32(S / s_b) stays finite): the scale bytes then depend on the exact rounding
    of m / 6, which the kernel takes on its IEEE-division branch there."""
    M, N = 256, 128
    rng = np.random.default_rng(91)
    v = rng.uniform(-2.3e-38, 2.3e-38, size=(M, N)) * rng.uniform(0.02, 1.0, size=(M, 1))
    v[5, 7] = 4.1e-33                                   # the tensor amax: S ~ 6.6e35
    a = synth.round_to_bf16_bits(v.astype(np.float32))
    v = om.bf16_to_f64(a)
    am = nv.amax(v)
    S = nv.encode_scale(am)
    c_r, sb_r = nv.quantize_blocks(v, 1, S)
    c_c, sb_c = nv.quantize_blocks(v, 0, S)
    tiny = np.abs(v[:, :16]).max(axis=1) < 2.0 ** -125
    nz = np.count_nonzero(sb_r[tiny, 0])
    assert tiny.sum() > 100 and nz > 50 and tiny.sum() - nz > 20
    cr, sr, cc, sc = _quantize(bf16_dev(a), M, N, am, am, 0, 0)
    assert np.array_equal(sr, omx.e4m3_encode(sb_r))
    assert np.array_equal(cr, c_r)
    assert np.array_equal(sc, omx.e4m3_encode(sb_c).T)
    assert np.array_equal(cc, c_c.T)


def test_nvfp4_quantize_rotated_transpose(lib):
    """The rotated copy: the kernel rotates in fp32 (butterflies), the oracle in fp64 rounded
    to fp32, so a value may differ by an fp32 ulp; codes and scales may then differ only where
    that ulp crosses a rounding boundary, by one step, and rarely."""
    M, N, mask = 512, 320, 0xA5C3
    a = synth.gen_bf16_matrix(77, M, N, outlier_rows=6)
    v = om.bf16_to_f64(a)
    y = nv.to_f32(nv.rht_rows(v, mask))
    am_r = nv.amax(y)
    _, _, cc, sc = _quantize(bf16_dev(a), M, N, nv.amax(v), am_r, 1, mask)
    S = nv.encode_scale(am_r)
    c_c, sb_c = nv.quantize_blocks(y, 0, S)
    want_s = omx.e4m3_encode(sb_c).T
    s_diff = sc != want_s
    assert s_diff.mean() < 1e-2
    assert np.all(np.abs(sc.astype(int) - want_s.astype(int))[s_diff] == 1)
    same_scale = np.repeat(~s_diff, 16, axis=1)
    c_diff = (cc != c_c.T) & same_scale
    assert c_diff.mean() < 1e-3
    mag = lambda c: (c & 7).astype(int)  # noqa: E731  (E2M1 magnitude codes are ordered)
    assert np.all(np.abs(mag(cc) - mag(c_c.T))[c_diff] == 1)
    deq_k = nv.dequantize_blocks(cc, omx.e4m3_decode(sc), 1, S)
    assert rel_fro(deq_k, nv.dequantize_blocks(c_c, sb_c, 0, S).T) < 1e-2


@pytest.mark.parametrize("M,N", [(16, 64), (256, 192), (1040, 2880)])
def test_nvfp4_amax(lib, M, N):
    a = synth.gen_bf16_matrix(M + 3 * N, M, N, outlier_rows=5)
    v = om.bf16_to_f64(a)
    mask = 0x0F0F ^ M
    out = torch.full((2,), -1.0, dtype=torch.float32, device="cuda")
    g.nvfp4_amax(bf16_dev(a), M, N, mask, out.data_ptr(), out.data_ptr() + 4)
    plain = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    g.nvfp4_amax(bf16_dev(a), M, N, mask, plain, None)
    torch.cuda.synchronize()
    o = out.cpu().numpy().astype(np.float64)
    assert o[0] == nv.amax(v) and plain.item() == nv.amax(v)
    want = nv.rht_amax_segments([v], mask)
    assert abs(o[1] - want) <= 1e-6 * want


def _cfg(name, **kw):
    base = synth.LayerConfig(name, T=300, E=4, k=2, H=256, F=256, precision="nvfp4", align=128,
                             seed=11)
    return base.with_(**kw)


_CLAMP = dict(activation="clamped_swiglu", beta=1.702, gate_max=7.0, lin_lo=-7.0, lin_hi=7.0,
              lin_offset=1.0)
CASES = {
    "swiglu": _cfg("nv_swiglu"),
    # ragged tail of 64-column tiles (F = 320: a 256 + 64 split), several k-blocks
    "geglu_ragged": _cfg("nv_geglu", activation="geglu", F=320, H=576, T=260, seed=12),
    # skewed routing: empty experts (all-zero weight-gradient tiles), long segments
    "clamped_skew": _cfg("nv_clamped", T=300, E=64, k=4, zipf_s=1.5, seed=13, **_CLAMP),
    "srelu": _cfg("nv_srelu", activation="srelu", F=384, seed=14),
}


@pytest.mark.parametrize("name", list(CASES))
def test_nvfp4_layer_parity(lib, name):
    cfg = CASES[name]
    inp = Inputs(cfg)
    run = LayerRun(inp)
    r = check_nvfp4(cfg, inp, run)
    if name == "clamped_skew":
        assert (np.bincount(r.ids.ravel(), minlength=cfg.E) == 0).any()


def check_nvfp4(cfg, inp, run):
    mask = synth.gen_rht_mask(cfg)
    r = om.layer_nvfp4(inp.logits, om.bf16_to_f64(inp.x), om.bf16_to_f64(inp.w1),
                       om.bf16_to_f64(inp.w2), cfg.k, act_params(cfg), mask,
                       dy=om.bf16_to_f64(inp.dy), align=cfg.align)
    counts = np.bincount(r.ids.ravel(), minlength=cfg.E)
    # the BF16 tensors the fused kernels emit, row by row of each expert's segment
    Z = run.unpack_cols(to_np(run.ws("z", torch.bfloat16, cfg.N1)))
    A = to_np(run.ws("a_s", torch.bfloat16, cfg.F))
    dZ = run.unpack_cols(to_np(run.ws("dz", torch.bfloat16, cfg.N1)))
    off = r.perm.offsets
    for e in range(cfg.E):
        rows = slice(off[e], off[e] + counts[e])
        if counts[e]:
            assert rel_fro(Z[rows], r.Z[e]) < BF16_TOL, e
            assert rel_fro(A[rows], r.A[e]) < BF16_TOL, e
            assert rel_fro(dZ[rows], r.dZ[e]) < BF16_TOL, e
        assert not A[off[e] + counts[e]:off[e + 1]].any()      # padding rows stay zero
    am = run.layer.ws_view("nv_amax", torch.float32, (16,)).cpu().numpy().astype(np.float64)
    got = dict(zip(g.NV_AMAX, am))
    for k in ("x", "dy", "w1", "w2"):
        assert got[k] == r.amax[k], k
    for k in ("a", "dz", "at", "dzt"):       # from bf16 values that may differ by one ulp
        assert abs(got[k] - r.amax[k]) <= 2.0 ** -8 * r.amax[k], k
    for k in ("xt", "dyt"):                  # exact inputs, fp32 rotation
        assert abs(got[k] - r.amax[k]) <= 1e-6 * r.amax[k], k
    # layer outputs
    assert rel_fro(to_np(run.y), r.y) < NV_TOL
    assert rel_fro(to_np(run.dx), r.dx) < NV_TOL
    assert rel_fro(to_np(run.d_probs), r.d_probs) < NV_TOL
    assert rel_fro(to_np(run.dw2), r.dW2) < NV_TOL
    assert rel_fro(run.dw1_logical(), r.dW1) < NV_TOL
    return r


def test_nvfp4_cuda_graph_capture_and_replay_with_new_routing(lib):
    """The NVFP4 step (route with its amaxes, weight amaxes and copies, the quantisers, all
    GEMMs and the amax resets) has no host sync: capture it once, replay it after
    overwriting the logits in place, and the new routing's layer comes out."""
    cfg = CASES["clamped_skew"]
    run = LayerRun(Inputs(cfg))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            run.run(sync=False)
    lg2 = synth.gen_logits(cfg.with_(seed=98))
    run.logits_d.copy_(torch.from_numpy(lg2))
    graph.replay()
    torch.cuda.synchronize()
    check_nvfp4(cfg, Inputs(cfg, logits=lg2), run)
    # the replay is the eager step, bit for bit
    got = [t.clone() for t in (run.y, run.dx, run.dw1p, run.dw2, run.d_probs)]
    run.run()
    for a, b in zip(got, (run.y, run.dx, run.dw1p, run.dw2, run.d_probs)):
        assert torch.equal(a, b)


def test_nvfp4_reused_weight_copies(lib):
    """reuse_weights: a second micro-batch that reuses the first forward's NVFP4 weight copies
    and amaxes gives bit-identical results to one that quantises the weights again."""
    cfg = CASES["geglu_ragged"]
    run = LayerRun(Inputs(cfg))
    run.logits_d.copy_(torch.from_numpy(synth.gen_logits(cfg.with_(seed=77))))
    run.run()
    want = [t.clone() for t in (run.y, run.dx, run.dw1p, run.dw2, run.d_probs)]
    run.layer.desc.reuse_weights = 1
    run.run()
    run.layer.desc.reuse_weights = 0
    assert run.layer.device_error() == 0
    for a, b in zip((run.y, run.dx, run.dw1p, run.dw2, run.d_probs), want):
        assert torch.equal(a, b)


def test_nvfp4_layer_is_not_the_bf16_layer(lib):
    """The tolerance discriminates: the same layer without quantisation is far outside it."""
    cfg = CASES["swiglu"]
    inp = Inputs(cfg)
    run = LayerRun(inp, backward=False)
    ref = om.layer(inp.logits, om.bf16_to_f64(inp.x), om.bf16_to_f64(inp.w1),
                   om.bf16_to_f64(inp.w2), cfg.k, act_params(cfg), align=cfg.align)
    assert rel_fro(to_np(run.y), ref.y) > 10 * NV_TOL


def test_nvfp4_layer_repeat_is_deterministic(lib):
    run = LayerRun(Inputs(CASES["geglu_ragged"]))
    y, dx, dw1, dw2, dp = (t.clone() for t in (run.y, run.dx, run.dw1p, run.dw2, run.d_probs))
    run.run()
    assert torch.equal(run.y, y) and torch.equal(run.dx, dx) and torch.equal(run.dw2, dw2)
    assert torch.equal(run.dw1p, dw1) and torch.equal(run.d_probs, dp)
