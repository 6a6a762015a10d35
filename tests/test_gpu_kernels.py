"""GPU parity of the standalone kernels through the C ABI: the MXFP8 quantiser and the route +
permute step (both bit-exact against the oracle), and the GLU weight repacking."""
import numpy as np
import pytest
import torch

import grouped_gemm_device_gb300 as g
from grouped_gemm_device_gb300 import synth
from oracle import moe as om
from oracle import mxfp8 as omx

from .gpu_helpers import bf16_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,scale,outliers", [
    (32, 32, 1.0, 0), (64, 64, 1.0, 4), (96, 160, 3.0, 10), (128, 4096, 0.02, 16),
    (2080, 2880, 1.0, 64), (32, 7168, 1e-30, 2), (256, 96, 1e25, 8),
])
def test_mxfp8_quantize_bit_exact(lib, M, N, scale, outliers):
    a = synth.gen_bf16_matrix(M * 7 + N, M, N, scale=scale, outlier_rows=outliers)
    x = bf16_dev(a)
    q_row = torch.empty(M, N, dtype=torch.uint8, device="cuda")
    s_row = torch.empty(M, N // 32, dtype=torch.uint8, device="cuda")
    q_col = torch.empty(M, N, dtype=torch.uint8, device="cuda")
    s_col = torch.empty(N, M // 32, dtype=torch.uint8, device="cuda")
    g.mxfp8_quantize(x, M, N, 1, 1, q_row, s_row, q_col, s_col)
    torch.cuda.synchronize()
    v = om.bf16_to_f64(a)
    c_r, s_r = omx.quantize_blocks(v, axis=1)
    c_c, s_c = omx.quantize_blocks(v, axis=0)
    assert np.array_equal(s_row.cpu().numpy(), s_r)
    assert np.array_equal(q_row.cpu().numpy(), c_r)
    assert np.array_equal(s_col.cpu().numpy(), s_c.T)
    assert np.array_equal(q_col.cpu().numpy(), c_c)


@pytest.mark.parametrize("M,N,groups", [
    (150, 64, [0, 7, 7, 40, 45, 113, 150]),              # ragged, an empty group, short blocks
    (4096 + 77, 2880, None),                               # None: seeded ragged split of 37
    (33, 96, [0, 33]),                                     # one group, one full + one 1-row block
    (256, 4096, [0, 0, 0, 256]),                           # leading empty groups
])
def test_mxfp8_quantize_grouped_colwise_bit_exact(lib, M, N, groups):
    if groups is None:
        r = np.random.default_rng(M)
        cuts = np.sort(r.integers(0, M + 1, size=36))
        groups = [0, *cuts.tolist(), M]
    G = len(groups) - 1
    a = synth.gen_bf16_matrix(M + N, M, N, scale=1.0, outlier_rows=max(1, M // 40))
    x = bf16_dev(a)
    nb = g.mxfp8_grouped_scale_cols(M, G)
    off = torch.tensor(groups, dtype=torch.int32, device="cuda")
    q_row = torch.empty(M, N, dtype=torch.uint8, device="cuda")
    s_row = torch.empty(M, N // 32, dtype=torch.uint8, device="cuda")
    q_col = torch.full((M, N), 0x55, dtype=torch.uint8, device="cuda")
    s_col = torch.full((N, nb), 0x55, dtype=torch.uint8, device="cuda")
    g.mxfp8_quantize(x, M, N, 1, 1, q_row, s_row, q_col, s_col, group_offsets=off,
                     num_groups=G)
    torch.cuda.synchronize()
    v = om.bf16_to_f64(a)
    c_c, s_c = omx.quantize_colwise_groups(v, groups)
    c_r, s_r = omx.quantize_blocks(v, axis=1)
    assert np.array_equal(q_col.cpu().numpy(), c_c)
    assert np.array_equal(s_col.cpu().numpy(), s_c)
    assert np.array_equal(q_row.cpu().numpy(), c_r)
    assert np.array_equal(s_row.cpu().numpy(), s_r)


def test_mxfp8_quantize_one_direction_only(lib):
    M, N = 64, 96
    a = synth.gen_bf16_matrix(5, M, N)
    x = bf16_dev(a)
    q_row = torch.zeros(M, N, dtype=torch.uint8, device="cuda")
    s_row = torch.zeros(M, N // 32, dtype=torch.uint8, device="cuda")
    g.mxfp8_quantize(x, M, N, 1, 0, q_row, s_row, None, None)
    torch.cuda.synchronize()
    c_r, s_r = omx.quantize_blocks(om.bf16_to_f64(a), axis=1)
    assert np.array_equal(q_row.cpu().numpy(), c_r) and np.array_equal(s_row.cpu().numpy(), s_r)


def test_mxfp8_quantize_16_byte_aligned_outputs(lib):
    """Outputs that are 16- but not 32-byte aligned take the 128-bit store path."""
    M, N = 160, 224
    a = synth.gen_bf16_matrix(9, M, N, outlier_rows=3)
    x = bf16_dev(a)
    q_row_buf = torch.zeros(M * N + 16, dtype=torch.uint8, device="cuda")
    q_col_buf = torch.zeros(M * N + 16, dtype=torch.uint8, device="cuda")
    q_row, q_col = q_row_buf[16:].view(M, N), q_col_buf[16:].view(M, N)
    assert q_row.data_ptr() % 32 == 16 and q_col.data_ptr() % 32 == 16
    s_row = torch.empty(M, N // 32, dtype=torch.uint8, device="cuda")
    s_col = torch.empty(N, M // 32, dtype=torch.uint8, device="cuda")
    g.mxfp8_quantize(x, M, N, 1, 1, q_row, s_row, q_col, s_col)
    torch.cuda.synchronize()
    v = om.bf16_to_f64(a)
    c_r, s_r = omx.quantize_blocks(v, axis=1)
    c_c, s_c = omx.quantize_blocks(v, axis=0)
    assert np.array_equal(q_row.cpu().numpy(), c_r) and np.array_equal(s_row.cpu().numpy(), s_r)
    assert np.array_equal(q_col.cpu().numpy(), c_c) and np.array_equal(s_col.cpu().numpy(), s_c.T)
    assert not q_row_buf[:16].any() and not q_col_buf[:16].any()


ROUTE_CASES = {
    "tiny": synth.CONFIGS["tiny"],
    "ragged_T": synth.LayerConfig("r", T=301, E=6, k=2, H=64, F=64, seed=11),
    "single_expert": synth.LayerConfig("s", T=77, E=1, k=1, H=128, F=64, seed=12),
    "k_equals_E": synth.LayerConfig("kE", T=130, E=4, k=4, H=64, F=64, seed=13),
    "zipf_dsv3_shape": synth.LayerConfig("z", T=512, E=256, k=8, H=64, F=64, seed=3, zipf_s=1.1),
    "gptoss_shape": synth.LayerConfig("o", T=1000, E=128, k=4, H=192, F=64, seed=4),
}


def _route_check(cfg, logits):
    x = synth.gen_x(cfg)
    d = g.desc_from_config(cfg)
    L = g.MoELayer(d)
    L.route_permute(torch.from_numpy(logits).cuda(), bf16_dev(x), cfg.T)
    torch.cuda.synchronize()
    ids, probs = om.route(logits, cfg.k)
    pm = om.permutation(ids, cfg.E, cfg.align)
    assert L.device_error() == 0
    assert np.array_equal(L.topk_ids[:cfg.T].cpu().numpy(), ids)
    assert np.allclose(L.topk_probs[:cfg.T].cpu().numpy(), probs, rtol=1e-6, atol=1e-7)
    assert np.array_equal(L.counts.cpu().numpy(), pm.counts)
    assert np.array_equal(L.offsets().cpu().numpy(), pm.offsets)
    used = int(pm.offsets[-1])
    R = L.layout.R_cap
    row_of = L.ws_view("row_of", torch.int32, (d.T_max * cfg.k,))[:cfg.T * cfg.k].cpu().numpy()
    src_of = L.ws_view("src_of", torch.int32, (R,))[:used].cpu().numpy()
    row_prob = L.ws_view("row_prob", torch.float32, (R,))[:used].cpu().numpy()
    assert np.array_equal(row_of, pm.row_of.ravel())
    assert np.array_equal(src_of, pm.src_of)
    want_p = np.zeros(used)
    live = pm.src_of >= 0
    want_p[live] = probs.ravel()[pm.src_of[live]]
    assert np.allclose(row_prob, want_p, rtol=1e-6, atol=1e-7)
    assert np.all(row_prob[~live] == 0)
    # gathered tokens: exact copies; padding and unused capacity rows are zero
    xp = L.ws_view("x_perm", torch.int16, (R, cfg.H)).cpu().numpy().view(np.uint16)
    want = np.zeros((R, cfg.H), dtype=np.uint16)
    want[:used][live] = x[pm.src_of[live] // cfg.k]
    assert np.array_equal(xp, want)
    # the same maps exported into caller tensors (moe_route_export), against the oracle
    i32 = dict(dtype=torch.int32, device="cuda")
    off_o = torch.full((cfg.E + 1,), -7, **i32)
    row_o = torch.full((cfg.T * cfg.k,), -7, **i32)
    src_o = torch.full((R,), -7, **i32)
    prob_o = torch.full((R,), -7.0, dtype=torch.float32, device="cuda")
    g.moe_route_export(d, L.ws, L.ws_bytes, cfg.T, off_o, row_o, src_o, prob_o)
    torch.cuda.synchronize()
    assert np.array_equal(off_o.cpu().numpy(), pm.offsets)
    assert np.array_equal(row_o.cpu().numpy(), pm.row_of.ravel())
    # rows at or beyond offsets[E] are outside the layout's contract: compare the used rows,
    # and the rest with the workspace itself
    src_all = src_o.cpu().numpy()
    assert np.array_equal(src_all[:used], pm.src_of)
    assert np.array_equal(src_all, L.ws_view("src_of", torch.int32, (R,)).cpu().numpy())
    prob_all = prob_o.cpu().numpy()
    assert np.array_equal(prob_all[:used], row_prob)
    # a partial export writes only what it is given
    row2 = torch.full((cfg.T * cfg.k,), -7, **i32)
    src2 = torch.full((R,), -7, **i32)
    g.moe_route_export(d, L.ws, L.ws_bytes, cfg.T, row_of=row2)
    torch.cuda.synchronize()
    assert np.array_equal(row2.cpu().numpy(), pm.row_of.ravel())
    assert np.all(src2.cpu().numpy() == -7)


@pytest.mark.parametrize("name", list(ROUTE_CASES))
def test_route_permute_bit_exact(lib, name):
    cfg = ROUTE_CASES[name]
    _route_check(cfg, synth.gen_logits(cfg))


def test_route_all_tokens_one_expert_and_ties(lib):
    cfg = synth.LayerConfig("hot", T=200, E=8, k=2, H=64, F=64, seed=21)
    lg = synth.gen_logits(cfg)
    lg[:, 5] += 50.0                       # expert 5 takes every token
    lg[::3, 2] = lg[::3, 6] = 1.25         # exact ties for the second slot
    _route_check(cfg, lg)


def test_route_non_finite_logits(lib):
    # NaN logits count as -inf; every chosen id stays in [0, E) and the probabilities are the
    # softmax's limits (uniform when every chosen logit is -inf)
    cfg = synth.LayerConfig("nan", T=300, E=40, k=4, H=64, F=64, seed=23)
    lg = synth.gen_logits(cfg)
    lg[0, :] = np.nan
    lg[1, :] = -np.inf
    lg[2, ::3] = np.nan
    lg[3, [5, 17]] = np.inf
    lg[4, :37] = np.nan
    lg[5, 1::2] = -np.inf
    lg[5, ::2] = np.nan
    lg[6, 39] = np.inf
    lg[7, :] = np.inf
    _route_check(cfg, lg)


def test_route_with_T_below_capacity_and_reuse(lib):
    cfg = synth.LayerConfig("cap", T=96, E=4, k=2, H=64, F=64, seed=22)
    d = g.desc_from_config(cfg, T_max=200)
    L = g.MoELayer(d)
    for T in (96, 37, 0):
        lg = synth.gen_logits(cfg)[:T] if T else np.zeros((0, 4), np.float32)
        x = synth.gen_x(cfg)[:T]
        L.route_permute(torch.from_numpy(np.ascontiguousarray(lg)).cuda() if T else
                        torch.empty(0, 4, device="cuda"),
                        bf16_dev(x) if T else torch.empty(0, 64, dtype=torch.bfloat16,
                                                          device="cuda"), T)
        torch.cuda.synchronize()
        ids, _ = om.route(lg, 2) if T else (np.zeros((0, 2), np.int64), None)
        pm = om.permutation(ids, 4, 32)
        assert np.array_equal(L.counts.cpu().numpy(), pm.counts)
        assert np.array_equal(L.offsets().cpu().numpy(), pm.offsets)


@pytest.mark.parametrize("ilv,gated", [(64, 1), (32, 1), (128, 1), (0, 0)])
def test_pack_fc1_roundtrip(lib, ilv, gated):
    E, H, F = 3, 192, 256
    N1 = 2 * F if gated else F
    a = synth.gen_bf16_matrix(ilv + 1, E * H, N1).reshape(E, H, N1)
    src = bf16_dev(a)
    packed = torch.empty(E, N1, H, dtype=torch.bfloat16, device="cuda")
    g.moe_pack_fc1_weight(src, packed, E, H, F, gated, ilv if gated else 64, 0)
    back = torch.empty_like(src)
    g.moe_pack_fc1_weight(packed, back, E, H, F, gated, ilv if gated else 64, 1)
    torch.cuda.synchronize()
    pk = packed.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(back.view(torch.int16).cpu().numpy().view(np.uint16), a)
    for p in range(N1):
        if gated:
            b = p // ilv
            c = (b % 2) * F + (b // 2) * ilv + p % ilv
        else:
            c = p
        assert np.array_equal(pk[:, p, :], a[:, :, c])
