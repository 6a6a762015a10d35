"""Parity at the full workload sizes (Mixtral-, DeepSeek-V3- and GPT-OSS-shaped layers), in the
launch configuration the benchmark times, on sampled outputs the fp64 oracle computes one by
one:
  * routing, counts and padded offsets: bit-exact for every token;
  * y, dx and d_probs of sampled tokens: the oracle's per-expert definitions evaluated on those
    tokens' rows (every quantity is row-local except the weight gradients);
  * sampled columns of dW1 and dW2 of sampled experts: the definitions restricted to those
    columns, over all of the expert's rows (column-wise MXFP8 blocks included).
Tokens are sampled among those whose k experts all lie in a small set of busy experts, so the
oracle quantises only a few experts' weights. Tolerances as elsewhere: relative Frobenius
5e-3 (BF16) / 3e-2 (MXFP8) over the sample."""
import numpy as np
import pytest
import torch

import grouped_gemm_device_gb300 as g
from grouped_gemm_device_gb300 import synth
from oracle import moe as om
from oracle import mxfp8 as omx

from .gpu_helpers import BF16_TOL, MX_TOL, act_params, bf16_dev, rel_fro, to_np

pytestmark = pytest.mark.gpu

N_TOKENS = 6       # sampled tokens for y / dx / d_probs
N_EXPERTS = 2      # sampled experts for the weight gradients
N_COLS = 6         # sampled columns of each weight gradient


def _fq(v, axis, mx):
    return omx.fake_quant(v, axis) if mx else v


def _fq_rows(v, mx):
    return omx.fake_quant_rows_from(v) if mx else v


def _sample_tokens(ids, counts, k, rng):
    """Tokens whose experts all lie in the smallest set of busiest experts that holds at
    least N_TOKENS such tokens."""
    order = np.argsort(-counts, kind="stable")
    for s in range(k, len(counts) + 1):
        inset = np.zeros(len(counts), bool)
        inset[order[:s]] = True
        cand = np.nonzero(inset[ids].all(axis=1))[0]
        if len(cand) >= N_TOKENS:
            return rng.choice(cand, size=N_TOKENS, replace=False), list(order[:s])
    raise AssertionError("no sample")


@pytest.mark.parametrize("name", ["mixtral_bf16", "mixtral_mxfp8", "gptoss_bf16",
                                  "gptoss_mxfp8", "dsv3_mxfp8"])
def test_fullsize_sampled_parity(lib, name):
    cfg = synth.CONFIGS[name]
    mx = cfg.precision == "mxfp8"
    tol = MX_TOL if mx else BF16_TOL
    act = act_params(cfg)
    F = cfg.F
    rng = np.random.default_rng(1234)

    logits = synth.gen_logits(cfg)
    x = synth.gen_x(cfg)
    dy = synth.gen_dy(cfg)
    # ---------------------------------------------------------------- GPU, bench launch config
    layer = g.MoELayer(g.desc_from_config(cfg))
    w1p = torch.empty(cfg.E, cfg.N1, cfg.H, dtype=torch.bfloat16, device="cuda")
    w2 = torch.empty(cfg.E, cfg.F, cfg.H, dtype=torch.bfloat16, device="cuda")
    for e in range(cfg.E):       # upload (and repack) one expert at a time
        w1e = bf16_dev(synth.gen_w1_expert(cfg, e))[None]
        g.moe_pack_fc1_weight(w1e, w1p[e:e + 1], 1, cfg.H, cfg.F, int(cfg.gated), cfg.ilv, 0)
        w2[e].copy_(bf16_dev(synth.gen_w2_expert(cfg, e)))
    layer.route_permute(torch.from_numpy(logits).cuda(), bf16_dev(x), cfg.T)
    y = to_np(layer.forward(w1p, w2, cfg.T))
    dx, dw1p, dw2, dp = layer.backward(bf16_dev(dy), w1p, w2, cfg.T)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    dx, dp = to_np(dx), to_np(dp)

    # ---------------------------------------------------------------- routing, exact
    ids, probs = om.route(logits, cfg.k)
    pm = om.permutation(ids, cfg.E, cfg.align)
    assert np.array_equal(layer.topk_ids.cpu().numpy(), ids)
    assert np.array_equal(layer.counts.cpu().numpy(), pm.counts)
    assert np.array_equal(layer.offsets().cpu().numpy(), pm.offsets)

    toks, experts = _sample_tokens(ids, pm.counts, cfg.k, rng)
    wexp = experts[:N_EXPERTS]
    xs, dys = om.bf16_to_f64(x[toks]), om.bf16_to_f64(dy[toks])
    y_ref = np.zeros((N_TOKENS, cfg.H))
    dx_ref = np.zeros((N_TOKENS, cfg.H))
    dp_ref = np.zeros((N_TOKENS, cfg.k))
    errs = {}
    for e in experts:
        use_tok = [(i, j) for i in range(N_TOKENS) for j in range(cfg.k) if ids[toks[i], j] == e]
        if not use_tok and e not in wexp:
            continue
        W1 = om.bf16_to_f64(synth.gen_w1_expert(cfg, e))
        W2 = om.bf16_to_f64(synth.gen_w2_expert(cfg, e))
        wq = om.ExpertWeights(W1, W2, mx)
        # ------------------------------------------------------------ sampled tokens' rows
        for i, j in use_tok:
            p = probs[toks[i], j:j + 1]
            Z, a, a_s, Y = om.expert_forward(xs[i:i + 1], W1, W2, p, act, mx, wq)
            _, dX, _, _, d_prob = om.expert_backward(xs[i:i + 1], W1, W2, p, Z, a, a_s,
                                                     dys[i:i + 1], act, mx, wq)
            y_ref[i] += Y[0]
            dx_ref[i] += dX[0]
            dp_ref[i, j] = d_prob[0]
        if e not in wexp:
            continue
        # ------------------------------------------------------------ sampled weight columns
        tok, slot = pm.rows_of_expert[e]
        X = om.bf16_to_f64(x[tok])
        dY = om.bf16_to_f64(dy[tok])
        p = probs[tok, slot][:, None]
        fs = rng.choice(F, size=N_COLS, replace=False)
        hs = rng.choice(cfg.H, size=N_COLS, replace=False)
        Xq = _fq(X, 1, mx)
        Zg = Xq @ wq.w1_h[:, fs]
        if cfg.gated:
            Zl = Xq @ wq.w1_h[:, F + fs]
            a = om.act_forward(act, Zg, Zl)
        else:
            Zl = None
            a = om.act_forward(act, Zg)
        a_s = p * a
        # dW2[f, h] = sum_r a_s[r, f] dY[r, h]   (column-wise MXFP8 along the rows)
        dW2_ref = _fq_rows(a_s, mx).T @ _fq_rows(dY[:, hs], mx)
        fs_t, hs_t = torch.as_tensor(fs, device="cuda"), torch.as_tensor(hs, device="cuda")
        errs[f"dW2[{e}]"] = rel_fro(to_np(dw2[e][fs_t][:, hs_t]), dW2_ref)
        # dW1[h, n] = sum_r X[r, h] dZ[r, n] for n = gate f and linear f
        dA = p * (_fq(dY, 1, mx) @ wq.w2_h[fs].T)
        if cfg.gated:
            dG, dL = om.act_backward(act, Zg, Zl, dA)
            dZ = np.concatenate([dG, dL], axis=1)
            ncols = np.concatenate([fs, F + fs])
            half, w = ncols // F, ncols % F
            prow = (w // cfg.ilv) * 2 * cfg.ilv + half * cfg.ilv + w % cfg.ilv
        else:
            dZ, _ = om.act_backward(act, Zg, None, dA)
            ncols = prow = fs
        dW1_ref = _fq_rows(X[:, hs], mx).T @ _fq_rows(dZ, mx)     # [hs, ncols]
        dW1_gpu = to_np(dw1p[e][torch.as_tensor(prow, device="cuda")][:, hs_t]).T
        errs[f"dW1[{e}]"] = rel_fro(dW1_gpu, dW1_ref)
    errs.update({"y": rel_fro(y[toks], y_ref), "dx": rel_fro(dx[toks], dx_ref),
                 "d_probs": rel_fro(dp[toks], dp_ref)})
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, (name, errs)


def test_fullsize_nvfp4(lib):
    """The Mixtral-shaped NVFP4 layer in the benchmark's launch configuration. The per-tensor
    scales of x, dY, W1 and W2 come from amaxes the oracle computes exactly, so everything
    that depends only on them is checked on samples: the amax slots (plain and rotated), and
    sampled entries of the three BF16 tensors the fused kernels emit (the saved Z, a_s and dZ,
    each row-local given those scales: Z = Q(x) Q_H(W1), a_s = bf16(p act(Z)), dZ =
    bf16(dact(bf16 Z, p Q(dY) Q_H(W2)^T))). The layer outputs pass through the per-tensor
    scales of a_s and dZ, which need the whole tensor; for them the test checks properties:
    finite, and within NVFP4's quantisation-noise band of the unquantised oracle."""
    from oracle import nvfp4 as nv

    cfg = synth.CONFIGS["mixtral_nvfp4"]
    act = act_params(cfg)
    F, H, N1 = cfg.F, cfg.H, cfg.N1
    rng = np.random.default_rng(4321)
    logits, x, dy = synth.gen_logits(cfg), synth.gen_x(cfg), synth.gen_dy(cfg)
    mask = synth.gen_rht_mask(cfg)
    layer = g.MoELayer(g.desc_from_config(cfg))
    w1p = torch.empty(cfg.E, N1, H, dtype=torch.bfloat16, device="cuda")
    w2 = torch.empty(cfg.E, F, H, dtype=torch.bfloat16, device="cuda")
    am_w1 = am_w2 = 0.0
    for e in range(cfg.E):
        w1e, w2e = synth.gen_w1_expert(cfg, e), synth.gen_w2_expert(cfg, e)
        am_w1 = max(am_w1, nv.amax(om.bf16_to_f64(w1e)))
        am_w2 = max(am_w2, nv.amax(om.bf16_to_f64(w2e)))
        g.moe_pack_fc1_weight(bf16_dev(w1e)[None], w1p[e:e + 1], 1, H, F, 1, cfg.ilv, 0)
        w2[e].copy_(bf16_dev(w2e))
    layer.route_permute(torch.from_numpy(logits).cuda(), bf16_dev(x), cfg.T)
    y = to_np(layer.forward(w1p, w2, cfg.T))
    dx, _, _, dp = layer.backward(bf16_dev(dy), w1p, w2, cfg.T)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    dx, dp = to_np(dx), to_np(dp)
    ids, probs = om.route(logits, cfg.k)
    pm = om.permutation(ids, cfg.E, cfg.align)
    assert np.array_equal(layer.offsets().cpu().numpy(), pm.offsets)
    # ------------------------------------------------------------ amax slots
    xf, dyf = om.bf16_to_f64(x), om.bf16_to_f64(dy)
    got = dict(zip(g.NV_AMAX,
                   layer.ws_view("nv_amax", torch.float32, (16,)).cpu().numpy().astype(float)))
    assert got["x"] == nv.amax(xf) and got["dy"] == nv.amax(dyf)
    assert got["w1"] == am_w1 and got["w2"] == am_w2
    segs_x = [xf[tok] for tok, _ in pm.rows_of_expert]
    segs_dy = [dyf[tok] for tok, _ in pm.rows_of_expert]
    for k_, segs in (("xt", segs_x), ("dyt", segs_dy)):
        want = nv.rht_amax_segments(segs, mask)
        assert abs(got[k_] - want) <= 1e-6 * want, k_
    # ------------------------------------------------------------ sampled Z, a_s, dZ entries
    S = {k_: nv.encode_scale(v) for k_, v in (("x", nv.amax(xf)), ("dy", nv.amax(dyf)),
                                              ("w1", am_w1), ("w2", am_w2))}
    toks = rng.choice(cfg.T, size=4, replace=False)
    fs = rng.choice(F, size=8, replace=False)
    ws = layer.layout
    R = ws.R_cap
    Zw = layer.ws_view("z", torch.bfloat16, (R, N1))
    Aw = layer.ws_view("a_s", torch.bfloat16, (R, F))
    dZw = layer.ws_view("dz", torch.bfloat16, (R, N1))
    half_ilv = lambda n: (n % F // cfg.ilv) * 2 * cfg.ilv + (n // F) * cfg.ilv + n % F % cfg.ilv  # noqa: E731
    cols = np.concatenate([fs, F + fs])                 # gate f, linear f (logical)
    pcols = torch.as_tensor([half_ilv(n) for n in cols], device="cuda")
    want_z, want_a, want_dz, got_z, got_a, got_dz = [], [], [], [], [], []
    for t in toks:
        xq = nv.fake_quant(xf[t:t + 1], 1, S["x"])
        dyq = nv.fake_quant(dyf[t:t + 1], 1, S["dy"])
        for j in range(cfg.k):
            e, r = ids[t, j], pm.row_of[t, j]
            W1 = om.bf16_to_f64(synth.gen_w1_expert(cfg, e))[:, cols]      # [H, 16] logical
            W2 = om.bf16_to_f64(synth.gen_w2_expert(cfg, e))[fs]           # [8, H]
            Z = xq @ nv.fake_quant(W1, 0, S["w1"])
            a = om.act_forward(act, Z[:, :8], Z[:, 8:])
            Zb = om.bf16_round(Z)
            dA = probs[t, j] * (dyq @ nv.fake_quant(W2, 1, S["w2"]).T)
            dg, dl = om.act_backward(act, Zb[:, :8], Zb[:, 8:], dA)
            want_z.append(Zb[0])
            want_a.append(om.bf16_round(probs[t, j] * a)[0])
            want_dz.append(om.bf16_round(np.concatenate([dg, dl], axis=1))[0])
            got_z.append(to_np(Zw[r][pcols]))
            got_a.append(to_np(Aw[r][torch.as_tensor(fs, device="cuda")]))
            got_dz.append(to_np(dZw[r][pcols]))
    for name, a_, b_ in (("Z", got_z, want_z), ("a_s", got_a, want_a), ("dZ", got_dz, want_dz)):
        assert rel_fro(np.array(a_), np.array(b_)) < BF16_TOL, name
    # ------------------------------------------------------------ outputs: properties
    assert np.isfinite(y).all() and np.isfinite(dx).all() and np.isfinite(dp).all()
    ref_y, ref_dx = np.zeros((len(toks), H)), np.zeros((len(toks), H))
    for i, t in enumerate(toks):
        for j in range(cfg.k):
            e = ids[t, j]
            W1 = om.bf16_to_f64(synth.gen_w1_expert(cfg, e))
            W2 = om.bf16_to_f64(synth.gen_w2_expert(cfg, e))
            p = probs[t, j:j + 1]
            Z, a, a_s, Y = om.expert_forward(xf[t:t + 1], W1, W2, p, act, False)
            _, dX, _, _, _ = om.expert_backward(xf[t:t + 1], W1, W2, p, Z, a, a_s,
                                                dyf[t:t + 1], act, False)
            ref_y[i] += Y[0]
            ref_dx[i] += dX[0]
    for name, a_, b_ in (("y", y[toks], ref_y), ("dx", dx[toks], ref_dx)):
        rel = rel_fro(a_, b_)
        assert 0.02 < rel < 0.5, (name, rel)
