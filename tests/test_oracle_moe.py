"""Pins for oracle.moe against independent statements of the same mathematics:
brute-force routing, invariants of the permutation, closed forms of the activations,
central finite differences and torch autograd (fp64, CPU) for every derivative, the
per-token expert loop with index_add of the Transformer Engine MoE article (Challenge 1),
a dense MLP special case, and a scalar brute-force MXFP8 expert on tiny shapes."""
import itertools
import math

import numpy as np
import pytest
import torch

from grouped_gemm_device_gb300 import synth
from oracle import moe

ACTS = {
    "swiglu": moe.ActParams("swiglu", beta=1.0),
    "clamped_swiglu": moe.ActParams("clamped_swiglu", beta=1.702, gate_max=7.0, lin_lo=-7.0,
                                    lin_hi=7.0, lin_offset=1.0),
    "geglu": moe.ActParams("geglu"),
    "srelu": moe.ActParams("srelu"),
}

# --------------------------------------------------------------------------- routing


def brute_topk(row, k):
    E = len(row)
    order = sorted(range(E), key=lambda e: (-float(row[e]), e))[:k]
    m = max(float(row[e]) for e in order)
    w = [math.exp(float(row[e]) - m) for e in order]
    s = sum(w)
    return order, [x / s for x in w]


def test_route_brute_force_with_ties():
    rng = np.random.default_rng(0)
    lg = rng.standard_normal((200, 9)).astype(np.float32)
    lg[::7, 2] = lg[::7, 5]                 # exact ties between experts 2 and 5
    lg[::11] = 0.25                         # whole rows tied
    for k in (1, 2, 3, 9):
        ids, probs = moe.route(lg, k)
        for t in range(lg.shape[0]):
            o, p = brute_topk(lg[t], k)
            assert list(ids[t]) == o
            assert np.allclose(probs[t], p, rtol=1e-14, atol=0)


def test_route_non_finite_logits_are_limits_of_finite_ones():
    # NaN behaves as -inf; +-inf behave as the limit of very large finite logits: brute force
    # on the row with +-inf (and NaN) replaced by +-1e300 in fp64 gives the same choice and
    # the same probabilities (exp of a difference of two such values is exactly 1 or 0)
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((64, 8)).astype(np.float32)
    lg[0, [1, 4]] = np.nan
    lg[1, :] = np.nan
    lg[2, [0, 5]] = np.inf
    lg[3, :] = -np.inf
    lg[4, [2, 3, 6]] = -np.inf
    lg[5, :] = np.nan
    lg[5, 7] = -np.inf
    lg[6, 3] = np.inf
    lg[6, 5] = np.nan
    lg[7, ::2] = np.nan
    lg[7, 1::2] = np.inf
    big = np.where(np.isnan(lg), -1e300, np.where(np.isinf(lg), np.sign(lg).astype(np.float64) * 1e300,
                                                  lg.astype(np.float64)))
    for k in (1, 2, 3, 8):
        ids, probs = moe.route(lg, k)
        assert np.all((ids >= 0) & (ids < 8))
        for t in range(lg.shape[0]):
            o, p = brute_topk(big[t], k)
            assert list(ids[t]) == o, (t, k)
            assert np.allclose(probs[t], p, rtol=1e-14, atol=0), (t, k)


def test_route_softmax_equals_renormalised_full_softmax():
    rng = np.random.default_rng(1)
    lg = rng.standard_normal((50, 16)).astype(np.float32) * 3
    ids, probs = moe.route(lg, 4)
    full = np.exp(lg.astype(np.float64))
    full /= full.sum(1, keepdims=True)
    sel = np.take_along_axis(full, ids, 1)
    assert np.allclose(probs, sel / sel.sum(1, keepdims=True), rtol=1e-13)
    assert np.allclose(probs.sum(1), 1.0)


@pytest.mark.parametrize("E,k,T", [(1, 1, 37), (4, 4, 50), (8, 2, 300), (64, 6, 129)])
def test_permutation_invariants(E, k, T):
    rng = np.random.default_rng(E * 100 + k)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    if E >= 8:
        lg[:, 0] += 3.0                      # one hot expert, some empty ones
    ids, _ = moe.route(lg, k)
    pm = moe.permutation(ids, E, 32)
    assert pm.counts.sum() == T * k
    assert np.all(pm.offsets % 32 == 0) and pm.offsets[0] == 0
    assert np.all(np.diff(pm.offsets) >= pm.counts)
    assert np.all(np.diff(pm.offsets) - pm.counts < 32)
    # row_of is a bijection onto the non-padding rows, and src_of inverts it
    rows = pm.row_of.ravel()
    assert len(set(rows.tolist())) == T * k
    assert np.all(pm.src_of[rows] == np.arange(T * k))
    assert np.sum(pm.src_of >= 0) == T * k
    # rows are ordered by (expert, token)
    src = pm.src_of[pm.src_of >= 0]
    tok, slot = src // k, src % k
    ex = ids[tok, slot]
    key = ex * (T + 1) + tok
    assert np.all(np.diff(key) > 0)
    for e in range(E):
        seg = pm.src_of[pm.offsets[e]:pm.offsets[e + 1]]
        assert np.sum(seg >= 0) == pm.counts[e]
        assert np.all(seg[pm.counts[e]:] == -1)


# --------------------------------------------------------------------------- activations


def test_activation_closed_forms():
    p = ACTS["swiglu"]
    l = np.linspace(-3, 3, 13)
    assert np.all(moe.act_forward(p, np.zeros_like(l), l) == 0)
    g = np.full_like(l, 40.0)
    assert np.allclose(moe.act_forward(p, g, l), l * 40.0, rtol=1e-15)
    assert np.allclose(moe.act_forward(p, np.full_like(l, -40.0), l), 0, atol=1e-15)
    assert moe.act_forward(p, np.array([1.0]), np.array([1.0]))[0] == pytest.approx(
        1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    c = ACTS["clamped_swiglu"]
    s = lambda x: 1 / (1 + math.exp(-1.702 * x))
    assert c and moe.act_forward(c, np.array([9.0]), np.array([2.0]))[0] == pytest.approx(
        3.0 * 7.0 * s(7.0), rel=1e-14)
    assert moe.act_forward(c, np.array([2.0]), np.array([-9.0]))[0] == pytest.approx(
        -6.0 * 2.0 * s(2.0), rel=1e-14)
    assert moe.act_forward(c, np.array([2.0]), np.array([8.0]))[0] == pytest.approx(
        8.0 * 2.0 * s(2.0), rel=1e-14)
    ge = ACTS["geglu"]
    assert moe.act_forward(ge, np.array([0.0]), np.array([5.0]))[0] == 0.0
    assert moe.act_forward(ge, np.array([1.0]), np.array([1.0]))[0] == pytest.approx(
        0.8413447460685429, rel=1e-14)                       # Phi(1)
    sr = ACTS["srelu"]
    assert list(moe.act_forward(sr, np.array([-2.0, 0.0, 3.0]))) == [0.0, 0.0, 9.0]


@pytest.mark.parametrize("name", list(ACTS))
def test_activation_derivative_finite_differences(name):
    p = ACTS[name]
    rng = np.random.default_rng(5)
    g = rng.standard_normal(400) * 4
    l = rng.standard_normal(400) * 4
    # keep away from the clamp kinks where the derivative is one-sided
    if name == "clamped_swiglu":
        g = g[np.abs(g - 7) > 1e-3]
        l = l[: len(g)]
        g = g[np.abs(np.abs(l) - 7) > 1e-3]
        l = l[np.abs(np.abs(l) - 7) > 1e-3]
    if name == "srelu":
        g = g[np.abs(g) > 1e-3]
        l = None
    dA = rng.standard_normal(len(g))
    dg, dl = moe.act_backward(p, g, l, dA)
    h = 1e-6
    f = lambda gg, ll: moe.act_forward(p, gg, ll)
    num_g = (f(g + h, l) - f(g - h, l)) / (2 * h) * dA
    assert np.allclose(dg, num_g, rtol=1e-7, atol=1e-7)
    if l is not None:
        num_l = (f(g, l + h) - f(g, l - h)) / (2 * h) * dA
        assert np.allclose(dl, num_l, rtol=1e-7, atol=1e-7)


def torch_act(name, g, l):
    """The activations restated in torch (fp64), for autograd."""
    if name == "swiglu":
        return l * g * torch.sigmoid(g)
    if name == "clamped_swiglu":
        gc = torch.clamp(g, max=7.0)
        lc = torch.clamp(l, -7.0, 7.0)
        return (lc + 1.0) * gc * torch.sigmoid(1.702 * gc)
    if name == "geglu":
        return l * torch.nn.functional.gelu(g, approximate="none")
    if name == "srelu":
        return torch.relu(g) ** 2
    raise ValueError(name)


@pytest.mark.parametrize("name", list(ACTS))
def test_activation_derivative_vs_torch_autograd(name):
    p = ACTS[name]
    rng = np.random.default_rng(6)
    g = rng.standard_normal(1000) * 5
    l = rng.standard_normal(1000) * 5
    g[:5] = [7.0, -7.0, 0.0, 8.0, 6.0]        # clamp boundaries and beyond
    l[:5] = [7.0, -7.0, 8.0, -8.0, 0.0]
    dA = rng.standard_normal(1000)
    tg = torch.tensor(g, requires_grad=True)
    tl = torch.tensor(l, requires_grad=True)
    out = torch_act(name, tg, tl if p.gated else None) if p.gated else torch_act(name, tg, None)
    out.backward(torch.tensor(dA))
    dg, dl = moe.act_backward(p, g, l if p.gated else None, dA)
    assert np.allclose(moe.act_forward(p, g, l if p.gated else None), out.detach().numpy(),
                       rtol=1e-13, atol=1e-14)
    if name == "clamped_swiglu":
        # torch.clamp passes the gradient at equality too; compare everywhere
        pass
    assert np.allclose(dg, tg.grad.numpy(), rtol=1e-12, atol=1e-13)
    if p.gated:
        assert np.allclose(dl, tl.grad.numpy(), rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------- the layer


def small_inputs(T=64, E=4, k=2, H=64, F=32, act="swiglu", seed=0):
    cfg = synth.LayerConfig("t", T=T, E=E, k=k, H=H, F=F, seed=seed, activation=act)
    lg = synth.gen_logits(cfg)
    x = moe.bf16_to_f64(synth.gen_x(cfg))
    W1 = moe.bf16_to_f64(synth.gen_w1(cfg)) * 10
    W2 = moe.bf16_to_f64(synth.gen_w2(cfg)) * 10
    dy = moe.bf16_to_f64(synth.gen_dy(cfg))
    return cfg, lg, x, W1, W2, dy


def hf_loop_forward(lg, x, W1, W2, k, p: moe.ActParams):
    """The per-expert loop of the Transformer Engine MoE article (Challenge 1): for each
    expert, find its (token, slot) pairs, run the expert FFN on those tokens, multiply by
    the routing weight and index_add into the output. Routing is done by brute force."""
    T, E = lg.shape
    sel = np.zeros((T, k), dtype=np.int64)
    rw = np.zeros((T, k))
    for t in range(T):
        o, w = brute_topk(lg[t], k)
        sel[t], rw[t] = o, w
    out = np.zeros_like(x)
    F = W2.shape[1]
    for e in range(E):
        top_x, idx = np.where(sel == e)
        cur = x[top_x]
        z = cur @ W1[e]
        a = moe.act_forward(p, z[:, :F], z[:, F:]) if p.gated else moe.act_forward(p, z)
        h = (a @ W2[e]) * rw[top_x, idx][:, None]
        np.add.at(out, top_x, h)
    return out


@pytest.mark.parametrize("name", list(ACTS))
def test_layer_forward_equals_per_expert_loop(name):
    cfg, lg, x, W1, W2, _ = small_inputs(act=name)
    p = ACTS[name]
    r = moe.layer(lg, x, W1, W2, cfg.k, p)
    ref = hf_loop_forward(lg, x, W1, W2, cfg.k, p)
    assert np.allclose(r.y, ref, rtol=1e-12, atol=1e-12)


def torch_layer(lg, x, W1, W2, k, name):
    """Dense per-(token, slot) restatement in torch fp64 for autograd."""
    ids, _ = moe.route(lg, k)
    lt = torch.tensor(lg.astype(np.float64))
    chosen = torch.gather(lt, 1, torch.tensor(ids))
    probs = torch.softmax(chosen, dim=1).detach().requires_grad_(True)
    xt = torch.tensor(x, requires_grad=True)
    w1 = torch.tensor(W1, requires_grad=True)
    w2 = torch.tensor(W2, requires_grad=True)
    F = W2.shape[1]
    y = torch.zeros_like(xt)
    for j in range(k):
        z = torch.einsum("th,thn->tn", xt, w1[ids[:, j]])
        if name == "srelu":
            a = torch_act(name, z, None)
        else:
            a = torch_act(name, z[:, :F], z[:, F:])
        y = y + probs[:, j:j + 1] * torch.einsum("tf,tfh->th", a, w2[ids[:, j]])
    return y, probs, xt, w1, w2


@pytest.mark.parametrize("name", list(ACTS))
def test_layer_backward_vs_torch_autograd(name):
    cfg, lg, x, W1, W2, dy = small_inputs(act=name, E=5, k=3, T=48)
    p = ACTS[name]
    r = moe.layer(lg, x, W1, W2, cfg.k, p, dy=dy)
    y, probs, xt, w1, w2 = torch_layer(lg, x, W1, W2, cfg.k, name)
    assert np.allclose(r.y, y.detach().numpy(), rtol=1e-11, atol=1e-12)
    y.backward(torch.tensor(dy))
    dW1, dW2 = moe.stack_weight_grads(r, cfg.E)
    assert np.allclose(r.dx, xt.grad.numpy(), rtol=1e-10, atol=1e-11)
    assert np.allclose(dW1, w1.grad.numpy(), rtol=1e-10, atol=1e-11)
    assert np.allclose(dW2, w2.grad.numpy(), rtol=1e-10, atol=1e-11)
    assert np.allclose(r.d_probs, probs.grad.numpy(), rtol=1e-10, atol=1e-11)


def test_empty_expert_gets_zero_weight_gradient():
    cfg, lg, x, W1, W2, dy = small_inputs(E=6, k=1, T=40)
    lg[:, 3] = -100.0
    r = moe.layer(lg, x, W1, W2, 1, ACTS["swiglu"], dy=dy)
    assert r.perm.counts[3] == 0
    assert np.all(r.dW1[3] == 0) and np.all(r.dW2[3] == 0)


def test_single_expert_is_a_dense_mlp():
    cfg, lg, x, W1, W2, dy = small_inputs(E=1, k=1, T=33)
    p = ACTS["swiglu"]
    r = moe.layer(lg, x, W1, W2, 1, p, dy=dy)
    z = x @ W1[0]
    F = W2.shape[1]
    a = z[:, F:] * z[:, :F] / (1 + np.exp(-z[:, :F]))
    assert np.allclose(r.probs, 1.0)
    assert np.allclose(r.y, a @ W2[0], rtol=1e-12, atol=1e-13)


def test_prob_scaling_commutes_with_fc2():
    cfg, lg, x, W1, W2, _ = small_inputs()
    r = moe.layer(lg, x, W1, W2, cfg.k, ACTS["swiglu"], keep_intermediates=True)
    for e in range(cfg.E):
        tok, slot = r.perm.rows_of_expert[e]
        d = r.per_expert[e]
        p = r.probs[tok, slot][:, None]
        assert np.allclose(d["Y"], p * (d["a"] @ W2[e]), rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------- MXFP8 expert


def scalar_mx_rows(mat, along_rows):
    """Scalar MXFP8 fake-quantisation of a small matrix, written with plain Python loops:
    blocks of 32 along columns (along_rows=False) or rows (True), exponent by math.frexp,
    elements by exhaustive nearest search over the E4M3 magnitudes."""
    from tests.test_oracle_mxfp8 import brute_round
    m = [list(map(float, r)) for r in mat]
    R, C = len(m), len(m[0]) if m else 0
    out = [[0.0] * C for _ in range(R)]
    if along_rows:
        groups = [[(r, c) for r in range(r0, min(R, r0 + 32))] for c in range(C)
                  for r0 in range(0, R, 32)]
    else:
        groups = [[(r, c) for c in range(c0, c0 + 32)] for r in range(R) for c0 in range(0, C, 32)]
    for grp in groups:
        amax = max(abs(m[r][c]) for r, c in grp)
        if amax == 0:
            e = -127
        else:
            e = max(-127, min(127, math.frexp(amax)[1] - 1 - 8))
        for r, c in grp:
            out[r][c] = brute_round(m[r][c] / 2.0 ** e) * 2.0 ** e
    return np.array(out)


def test_mx_expert_matches_scalar_brute_force():
    rng = np.random.default_rng(9)
    m, H, F = 40, 64, 32
    X = rng.standard_normal((m, H))
    W1 = rng.standard_normal((H, 2 * F)) * 0.1
    W2 = rng.standard_normal((F, H)) * 0.1
    p = rng.uniform(0.1, 1, m)
    dY = rng.standard_normal((m, H))
    act = ACTS["swiglu"]
    Z, a, a_s, Y = moe.expert_forward(X, W1, W2, p, act, mx=True)
    dZ, dX, dW1, dW2, d_prob = moe.expert_backward(X, W1, W2, p, Z, a, a_s, dY, act, mx=True)
    q = scalar_mx_rows
    Zb = q(X, False) @ q(W1, True)
    ab = Zb[:, F:] * Zb[:, :F] / (1 + np.exp(-Zb[:, :F]))
    asb = p[:, None] * ab
    Yb = q(asb, False) @ q(W2, True)
    assert np.allclose(Z, Zb, rtol=1e-13, atol=1e-13)
    assert np.allclose(Y, Yb, rtol=1e-12, atol=1e-12)
    dAs = q(dY, False) @ q(W2, False).T
    # dZ from the dGLU's inputs as the epilogue holds them: bf16 Z and bf16 dA_s, each
    # rounded here through fp32 by truncation plus the round-to-nearest-even carry
    def bf16(v):
        u = np.asarray(v, np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
        return ((((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).astype(np.uint32)
                .view(np.float32).astype(np.float64))
    Zr = bf16(Zb)
    s = 1 / (1 + np.exp(-Zr[:, :F]))
    dA = p[:, None] * bf16(dAs)
    dZb = np.concatenate([dA * Zr[:, F:] * s * (1 + Zr[:, :F] * (1 - s)), dA * Zr[:, :F] * s], 1)
    assert np.allclose(d_prob, (dAs * ab).sum(1), rtol=1e-12, atol=1e-12)
    assert np.allclose(dZ, dZb, rtol=1e-12, atol=1e-12)
    assert np.allclose(dW2, q(asb, True).T @ q(dY, True), rtol=1e-12, atol=1e-12)
    assert np.allclose(dW1, q(X, True).T @ q(dZb, True), rtol=1e-12, atol=1e-12)
    assert np.allclose(dX, q(dZb, False) @ q(W1, False).T, rtol=1e-12, atol=1e-12)


def torch_layer_extras(lg, x, W1, W2, b1, sc, k, name):
    """torch_layer with the FC1 bias added to z and the feature scale on the activation."""
    ids, _ = moe.route(lg, k)
    lt = torch.tensor(lg.astype(np.float64))
    chosen = torch.gather(lt, 1, torch.tensor(ids))
    probs = torch.softmax(chosen, dim=1).detach().requires_grad_(True)
    xt = torch.tensor(x, requires_grad=True)
    w1 = torch.tensor(W1, requires_grad=True)
    w2 = torch.tensor(W2, requires_grad=True)
    bt = torch.tensor(b1, requires_grad=True)
    st = torch.tensor(sc, requires_grad=True)
    F = W2.shape[1]
    y = torch.zeros_like(xt)
    for j in range(k):
        e = ids[:, j]
        z = torch.einsum("th,thn->tn", xt, w1[e]) + bt[e]
        a = torch_act(name, z[:, :F], z[:, F:]) * st[e]
        y = y + probs[:, j:j + 1] * torch.einsum("tf,tfh->th", a, w2[e])
    return y, probs, xt, w1, w2, bt, st


@pytest.mark.parametrize("name", ["swiglu", "clamped_swiglu", "geglu"])
def test_bias_and_feature_scale_vs_torch_autograd(name):
    cfg, lg, x, W1, W2, dy = small_inputs(act=name, E=5, k=3, T=48)
    p = ACTS[name]
    rng = np.random.default_rng(7)
    b1 = 0.3 * rng.standard_normal((cfg.E, W1.shape[2]))
    sc = 1.0 + 0.5 * rng.standard_normal((cfg.E, W2.shape[1]))
    r = moe.layer(lg, x, W1, W2, cfg.k, p, dy=dy, b1=b1, s=sc)
    y, probs, xt, w1, w2, bt, st = torch_layer_extras(lg, x, W1, W2, b1, sc, cfg.k, name)
    assert np.allclose(r.y, y.detach().numpy(), rtol=1e-11, atol=1e-12)
    y.backward(torch.tensor(dy))
    dW1, dW2 = moe.stack_weight_grads(r, cfg.E)
    assert np.allclose(r.dx, xt.grad.numpy(), rtol=1e-10, atol=1e-11)
    assert np.allclose(dW1, w1.grad.numpy(), rtol=1e-10, atol=1e-11)
    assert np.allclose(dW2, w2.grad.numpy(), rtol=1e-10, atol=1e-11)
    assert np.allclose(r.d_probs, probs.grad.numpy(), rtol=1e-10, atol=1e-11)
    assert np.allclose(r.db1, bt.grad.numpy(), rtol=1e-10, atol=1e-11)
    assert np.allclose(r.ds, st.grad.numpy(), rtol=1e-10, atol=1e-11)


def test_zero_bias_unit_scale_change_nothing():
    cfg, lg, x, W1, W2, dy = small_inputs(act="swiglu", E=4, k=2, T=40)
    p = ACTS["swiglu"]
    plain = moe.layer(lg, x, W1, W2, cfg.k, p, dy=dy)
    ext = moe.layer(lg, x, W1, W2, cfg.k, p, dy=dy, b1=np.zeros((cfg.E, W1.shape[2])),
                    s=np.ones((cfg.E, W2.shape[1])))
    for a, b in ((plain.y, ext.y), (plain.dx, ext.dx), (plain.d_probs, ext.d_probs)):
        assert np.array_equal(a, b)
