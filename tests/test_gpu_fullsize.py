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


def _bf(v, mx):
    return om.bf16_round(v) if mx else v


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


def _weight_experts(experts, counts):
    """Experts whose weight-gradient columns are sampled: the busiest of the token sample's
    experts and the least-loaded expert that has rows (on skewed routing a segment of a few
    rows, shorter than one 128-row tile and than one k-block)."""
    live = np.nonzero(counts > 0)[0]
    small = int(live[np.argmin(counts[live])])   # first of the smallest
    return [experts[0]] + ([small] if small != experts[0] else list(experts[1:N_EXPERTS]))


@pytest.mark.parametrize("name", ["mixtral_bf16", "mixtral_mxfp8", "gptoss_bf16",
                                  "gptoss_mxfp8", "dsv3_mxfp8", "gptoss_geglu_bf16",
                                  "gptoss_srelu_bf16", "gptoss_geglu_mxfp8",
                                  "gptoss_srelu_mxfp8"])
def test_fullsize_sampled_parity(lib, name):
    _sampled_parity(name, recompute=False)


@pytest.mark.parametrize("name", ["mixtral_bf16", "mixtral_mxfp8"])
def test_fullsize_recompute_sampled_parity(lib, name):
    """The same sampled checks with activation recomputation (no saved FC1 output; the
    FC2-dgrad kernel rebuilds it in fp32 next to dA_s, so the oracle forms dZ from unrounded
    Z and dA_s), in the launch configuration `bench.py --recompute` times."""
    _sampled_parity(name, recompute=True)


def _sampled_parity(name, recompute):
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
    layer = g.MoELayer(g.desc_from_config(cfg, recompute=recompute))
    if recompute:
        assert layer.layout.z == 2 ** 64 - 1
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
    wexp = _weight_experts(experts, pm.counts)
    xs, dys = om.bf16_to_f64(x[toks]), om.bf16_to_f64(dy[toks])
    y_ref = np.zeros((N_TOKENS, cfg.H))
    dx_ref = np.zeros((N_TOKENS, cfg.H))
    dp_ref = np.zeros((N_TOKENS, cfg.k))
    errs = {}
    for e in list(experts) + [e for e in wexp if e not in experts]:
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
                                                     dys[i:i + 1], act, mx, wq,
                                                     recompute=recompute)
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
        # dW1[h, n] = sum_r X[r, h] dZ[r, n] for n = gate f and linear f; in MXFP8 dZ comes
        # from bf16 Z and bf16 dA_s (oracle reading R15), from fp32 ones when recomputed
        rb = mx and not recompute
        dA = p * _bf(_fq(dY, 1, mx) @ wq.w2_h[fs].T, rb)
        Zg, Zl = _bf(Zg, rb), (_bf(Zl, rb) if Zl is not None else None)
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


def nvfp4_fullsize_reference(cfg, logits, x, dy, w1, w2, toks, wexp, fs, hs):
    """fp64 oracle quantities of the NVFP4 layer (oracle.moe.layer_nvfp4's definitions) needed
    to check a full-size run on samples, computed by streaming the experts (w1, w2: lists of
    each expert's logical bf16 weights):
      * every per-tensor amax, including those of a_s and dZ (plain and rotated), which need
        the whole tensor: Z, a_s and dZ of every routed row are formed expert by expert;
      * y, dx and d_probs of the sampled tokens `toks`;
      * dW2[e][fs][:, hs] and dW1[e] at the gate/linear columns fs and the H columns hs, for
        the experts `wexp` (the rotation and the column-wise quantisation act on each column
        alone, so restricting to columns is exact).
    Experts are worked on in parallel threads. Returns (amax dict, y [n, H], dx [n, H],
    d_probs [n, k], {e: (dW2 cols [fs, hs], dW1 cols [hs, gate fs | linear fs])})."""
    import concurrent.futures as cf
    import os
    from oracle import nvfp4 as nv

    act = act_params(cfg)
    F, H = cfg.F, cfg.H
    mask = synth.gen_rht_mask(cfg)
    ids, probs = om.route(logits, cfg.k)
    pm = om.permutation(ids, cfg.E, cfg.align)
    xf, dyf = om.bf16_to_f64(x), om.bf16_to_f64(dy)
    am = {"x": nv.amax(xf), "dy": nv.amax(dyf),
          "w1": max(nv.amax(om.bf16_to_f64(w)) for w in w1),
          "w2": max(nv.amax(om.bf16_to_f64(w)) for w in w2),
          "xt": nv.rht_amax_segments([xf[tok] for tok, _ in pm.rows_of_expert], mask),
          "dyt": nv.rht_amax_segments([dyf[tok] for tok, _ in pm.rows_of_expert], mask)}
    S = {n: nv.encode_scale(v) for n, v in am.items()}
    xq = nv.fake_quant(xf, 1, S["x"])
    dyq = nv.fake_quant(dyf, 1, S["dy"])

    def expert(e):
        """amax contributions of expert e, its sampled rows, its kept columns."""
        tok, slot = pm.rows_of_expert[e]
        out = {"a": 0.0, "at": 0.0, "dz": 0.0, "dzt": 0.0, "rows": {}, "keep": None}
        if not len(tok):
            return out
        W1, W2 = om.bf16_to_f64(w1[e]), om.bf16_to_f64(w2[e])
        p = probs[tok, slot][:, None]
        Z = xq[tok] @ nv.fake_quant(W1, 0, S["w1"])
        a = om.act_forward(act, Z[:, :F], Z[:, F:]) if cfg.gated else om.act_forward(act, Z)
        A = om.bf16_round(p * a)
        dA_s = dyq[tok] @ nv.fake_quant(W2, 1, S["w2"]).T
        Zb = om.bf16_round(Z)
        del Z
        if cfg.gated:
            dg, dl = om.act_backward(act, Zb[:, :F], Zb[:, F:], p * om.bf16_round(dA_s))
            dZ = om.bf16_round(np.concatenate([dg, dl], axis=1))
            del dg, dl
        else:
            dZ = om.bf16_round(om.act_backward(act, Zb, None, p * om.bf16_round(dA_s))[0])
        del Zb
        out.update(a=nv.amax(A), dz=nv.amax(dZ), at=nv.rht_amax_segments([A], mask),
                   dzt=nv.rht_amax_segments([dZ], mask))
        pos = {int(t): i for i, t in enumerate(tok)}
        for i, t in enumerate(toks):
            for j in range(cfg.k):
                if ids[t, j] == e:
                    r = pos[int(t)]
                    out["rows"][(i, j)] = (A[r], dZ[r], float((dA_s[r] * a[r]).sum()))
        if e in wexp:
            ncols = np.concatenate([fs, F + fs]) if cfg.gated else fs
            out["keep"] = (A[:, fs].copy(), dyf[tok][:, hs], dZ[:, ncols].copy(), xf[tok][:, hs])
        return out

    with cf.ThreadPoolExecutor(max_workers=max(1, min(cfg.E, (os.cpu_count() or 2) // 2))) as ex:
        per = list(ex.map(expert, range(cfg.E)))
    for k_ in ("a", "at", "dz", "dzt"):
        am[k_] = max(o[k_] for o in per)
    S.update({k_: nv.encode_scale(am[k_]) for k_ in ("a", "at", "dz", "dzt")})
    y = np.zeros((len(toks), H))
    dx = np.zeros((len(toks), H))
    dp = np.zeros((len(toks), cfg.k))
    for e, o in enumerate(per):
        if not o["rows"]:
            continue
        w2_f = nv.fake_quant(om.bf16_to_f64(w2[e]), 0, S["w2"])    # FC2: W2 along F
        w1_n = nv.fake_quant(om.bf16_to_f64(w1[e]), 1, S["w1"])    # FC1 dgrad: W1 along N1
        for (i, j), (ra, rdz, d_prob) in o["rows"].items():
            y[i] += nv.fake_quant(ra[None], 1, S["a"])[0] @ w2_f
            dx[i] += nv.fake_quant(rdz[None], 1, S["dz"])[0] @ w1_n.T
            dp[i, j] = d_prob
    wg = {}
    for e, o in enumerate(per):
        if o["keep"] is None:
            continue
        A_f, dY_h, dZ_n, X_h = o["keep"]
        at_q = nv.colwise_rht_segments([A_f], mask, S["at"])[0]
        dyt_q = nv.colwise_rht_segments([dY_h], mask, S["dyt"])[0]
        dzt_q = nv.colwise_rht_segments([dZ_n], mask, S["dzt"])[0]
        xt_q = nv.colwise_rht_segments([X_h], mask, S["xt"])[0]
        wg[e] = (at_q.T @ dyt_q, xt_q.T @ dzt_q)
    return am, y, dx, dp, wg


def test_fullsize_nvfp4(lib):
    """The Mixtral-shaped NVFP4 layer in the benchmark's launch configuration against the
    oracle's definitions (oracle.moe.layer_nvfp4), evaluated by streaming the experts: every
    per-tensor amax (the ten slots, those of a_s and dZ formed from all routed rows), then y,
    dx and d_probs of sampled tokens and sampled columns of dW1 and dW2 of the busiest experts,
    at the NVFP4 tolerance of the small-shape layer tests (1e-2 relative Frobenius)."""
    from .test_gpu_nvfp4 import NV_TOL

    cfg = synth.CONFIGS["mixtral_nvfp4"]
    F, H, N1 = cfg.F, cfg.H, cfg.N1
    rng = np.random.default_rng(4321)
    logits, x, dy = synth.gen_logits(cfg), synth.gen_x(cfg), synth.gen_dy(cfg)
    w1h = [synth.gen_w1_expert(cfg, e) for e in range(cfg.E)]
    w2h = [synth.gen_w2_expert(cfg, e) for e in range(cfg.E)]
    layer = g.MoELayer(g.desc_from_config(cfg))
    w1p = torch.empty(cfg.E, N1, H, dtype=torch.bfloat16, device="cuda")
    w2 = torch.empty(cfg.E, F, H, dtype=torch.bfloat16, device="cuda")
    for e in range(cfg.E):
        g.moe_pack_fc1_weight(bf16_dev(w1h[e])[None], w1p[e:e + 1], 1, H, F, 1, cfg.ilv, 0)
        w2[e].copy_(bf16_dev(w2h[e]))
    layer.route_permute(torch.from_numpy(logits).cuda(), bf16_dev(x), cfg.T)
    y = to_np(layer.forward(w1p, w2, cfg.T))
    dx, dw1p, dw2, dp = layer.backward(bf16_dev(dy), w1p, w2, cfg.T)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    dx, dp = to_np(dx), to_np(dp)
    got = dict(zip(g.NV_AMAX,
                   layer.ws_view("nv_amax", torch.float32, (16,)).cpu().numpy().astype(float)))
    ids, probs = om.route(logits, cfg.k)
    pm = om.permutation(ids, cfg.E, cfg.align)
    assert np.array_equal(layer.offsets().cpu().numpy(), pm.offsets)

    toks, experts = _sample_tokens(ids, pm.counts, cfg.k, rng)
    wexp = experts[:N_EXPERTS]
    fs = rng.choice(F, size=N_COLS, replace=False)
    hs = rng.choice(H, size=N_COLS, replace=False)
    am, y_ref, dx_ref, dp_ref, wg = nvfp4_fullsize_reference(cfg, logits, x, dy, w1h, w2h, toks,
                                                             wexp, fs, hs)
    # the plain amaxes are maxima of bf16 (or input) values: exact; the rotated ones are maxima
    # of fp32 rotations (the oracle rotates in fp64)
    for k_ in ("x", "dy", "w1", "w2", "a", "dz"):
        assert got[k_] == am[k_], (k_, got[k_], am[k_])
    for k_ in ("xt", "dyt", "at", "dzt"):
        assert abs(got[k_] - am[k_]) <= 1e-6 * am[k_], (k_, got[k_], am[k_])
    errs = {"y": rel_fro(y[toks], y_ref), "dx": rel_fro(dx[toks], dx_ref),
            "d_probs": rel_fro(dp[toks], dp_ref)}
    fs_t, hs_t = torch.as_tensor(fs, device="cuda"), torch.as_tensor(hs, device="cuda")
    ncols = np.concatenate([fs, F + fs])
    half, w = ncols // F, ncols % F
    prow = torch.as_tensor((w // cfg.ilv) * 2 * cfg.ilv + half * cfg.ilv + w % cfg.ilv,
                           device="cuda")
    for e, (dW2_ref, dW1_ref) in wg.items():
        errs[f"dW2[{e}]"] = rel_fro(to_np(dw2[e][fs_t][:, hs_t]), dW2_ref)
        errs[f"dW1[{e}]"] = rel_fro(to_np(dw1p[e][prow][:, hs_t]).T, dW1_ref)
    bad = {k_: v for k_, v in errs.items() if not v <= NV_TOL}
    assert not bad, errs
