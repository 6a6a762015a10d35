"""fp64 oracle of the MoE expert layer: routing, permutation, grouped FC1 -> GLU -> prob scale
-> FC2, and its backward, in BF16-operand or MXFP8-operand form.

TEST INFRASTRUCTURE ONLY (see the package docstring). Plain definitions, computed per
expert with numpy matmul as the only library step; no blocking, fusion or reordering.

Readings of the pages (where they are silent or ambiguous), used consistently below:
  R1 top-k: larger logit first, ties to the lower expert index; slot j = rank j.
     Probabilities are the softmax over the k chosen logits (= full softmax renormalised
     over the top-k).                                           [TE-MoE] Figure 1 (top-2 router)
  R2 row order: expert ascending, then token ascending - the order in which the per-expert
     loop's torch.where visits tokens.                          [TE-MoE] Challenge 1 loop
  R3 expert segments start at offsets padded to `align` rows (32); padding rows are zero
     and carry probability 0.                  [NV-blog] device-resident per-group token counts
  R4 W1 logical columns [0,F) are the gate (the Swish side, "W" in the SwiGLU equation),
     [F,2F) the linear side ("V").                      [NV-blog] SwiGLU equation, b = c = 0
  R5 the routing probability scales the activation before FC2 (ScaledSwiGLU); FC2 has no
     bias, so this equals scaling the expert output.             [TE-MoE] Challenge 3
  R6 GeGLU uses the exact erf GELU; sReLU is the non-gated squared ReLU (FC1 width F).
  R7 clamped SwiGLU: g' = min(g, gate_max), l' = clip(l, lin_lo, lin_hi),
     a = (l' + lin_offset) * g' * sigmoid(beta * g'); a clamp passes the gradient at
     equality (the clamp is active only strictly beyond the limit).
  R8 MXFP8 operands (all six GEMMs): every GEMM consumes MXFP8 operands blocked along its
     own reduction dimension, fp32-or-better accumulation; column-wise blocks of the
     weight-gradient GEMMs start at each expert's first row.
  R9 d_prob[t, j] = sum_f dA_s * a (a unscaled); d_logits is not part of the layer.
  R15 MXFP8 backward: dZ, whose E4M3 codes are integer decisions the pages give no precision
     for, is formed from the fused dGLU epilogue's inputs in the precision the epilogue reads
     them: the saved FC1 output in bf16 and dA_s rounded to bf16 (with activation
     recomputation: both in fp32, so unrounded).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
from scipy.special import erf as _erf

from . import mxfp8

# ----------------------------------------------------------------------------- inputs


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp64 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


@dataclass
class ActParams:
    kind: str = "swiglu"            # swiglu | clamped_swiglu | geglu | srelu
    beta: float = 1.0
    gate_max: float = math.inf
    lin_lo: float = -math.inf
    lin_hi: float = math.inf
    lin_offset: float = 0.0

    @property
    def gated(self) -> bool:
        return self.kind != "srelu"


# ----------------------------------------------------------------------------- routing


def route(logits: np.ndarray, k: int):
    """Top-k expert choice and renormalised softmax over the chosen logits (R1).

    logits: fp32 [T, E]. Returns ids int64 [T, k], probs fp64 [T, k].
    [TE-MoE] Figure 1: a top-2 router sends each token to two of eight experts and the
    outputs are combined as a weighted sum.

    Non-finite logits (R1): a NaN logit counts as -inf; a chosen logit equal to the chosen
    maximum has weight 1, the others exp(l - max) - the limit of the softmax when the maximum
    is +inf (weight shared by the +inf logits) or -inf (uniform over the k chosen).
    """
    lg = np.asarray(logits, dtype=np.float32)
    lg = np.where(np.isnan(lg), np.float32(-np.inf), lg)
    T, E = lg.shape
    # stable sort of the negated logits keeps equal logits in index order
    ids = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    chosen = np.take_along_axis(lg, ids, axis=1).astype(np.float64)
    m = chosen.max(axis=1, keepdims=True)
    with np.errstate(invalid="ignore"):
        ex = np.where(chosen == m, 1.0, np.exp(chosen - m))
    probs = ex / ex.sum(axis=1, keepdims=True)
    return ids.astype(np.int64), probs


@dataclass
class Permutation:
    counts: np.ndarray          # [E]
    offsets: np.ndarray         # [E+1], padded segment starts
    row_of: np.ndarray          # [T, k] row of (token, slot)
    src_of: np.ndarray          # [R_used] flattened t*k+j, -1 for padding rows
    rows_of_expert: list = field(default_factory=list)   # per expert: (tokens, slots)


def permutation(ids: np.ndarray, E: int, align: int) -> Permutation:
    """Rows sorted by (expert, token) (R2), expert segments padded to `align` (R3).

    [NV-blog] section on removing host-device synchronisation: the grouped GEMM keeps each
    group's token count in device memory; here counts and padded offsets are the plain
    histogram and its exclusive scan.
    """
    T, k = ids.shape
    counts = np.bincount(ids.ravel(), minlength=E).astype(np.int64)
    padded = -(-counts // align) * align
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    row_of = np.full((T, k), -1, dtype=np.int64)
    src_of = np.full(int(offsets[-1]), -1, dtype=np.int64)
    rows = []
    for e in range(E):
        tok, slot = np.nonzero(ids == e)        # row-major: token ascending
        r = offsets[e] + np.arange(len(tok))
        row_of[tok, slot] = r
        src_of[r] = tok * k + slot
        rows.append((tok, slot))
    return Permutation(counts, offsets, row_of, src_of, rows)


# ----------------------------------------------------------------------------- activations


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _Phi(x):
    """Standard normal CDF via the library erf."""
    return 0.5 * (1.0 + _erf(np.asarray(x, dtype=np.float64) / math.sqrt(2.0)))


def _phi(x):
    return np.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)


def act_forward(p: ActParams, g: np.ndarray, l: np.ndarray | None = None) -> np.ndarray:
    """GLU activations of [NV-blog] (SwiGLU equation with b = c = 0; GeGLU; sReLU) with
    optional clamp and scale (R6, R7). For sReLU `g` is the whole FC1 output."""
    g = np.asarray(g, dtype=np.float64)
    if p.kind == "swiglu":
        return l * g * _sigmoid(p.beta * g)
    if p.kind == "clamped_swiglu":
        gc = np.minimum(g, p.gate_max)
        lc = np.clip(l, p.lin_lo, p.lin_hi)
        return (lc + p.lin_offset) * gc * _sigmoid(p.beta * gc)
    if p.kind == "geglu":
        return l * g * _Phi(g)
    if p.kind == "srelu":
        r = np.maximum(g, 0.0)
        return r * r
    raise ValueError(p.kind)


def act_backward(p: ActParams, g, l, dA):
    """Derivative of act_forward; returns (d_gate, d_linear) (d_linear None for sReLU).

    [NV-blog] GLU-epilogue section: the backward epilogue reads the saved FC1 output and
    computes dSwiGLU (here also dGeGLU / dsReLU and the clamped variant).
    """
    g = np.asarray(g, dtype=np.float64)
    if p.kind == "swiglu":
        s = _sigmoid(p.beta * g)
        return dA * l * s * (1.0 + p.beta * g * (1.0 - s)), dA * g * s
    if p.kind == "clamped_swiglu":
        gc = np.minimum(g, p.gate_max)
        lc = np.clip(l, p.lin_lo, p.lin_hi)
        s = _sigmoid(p.beta * gc)
        g_pass = (g <= p.gate_max).astype(np.float64)
        l_pass = ((l >= p.lin_lo) & (l <= p.lin_hi)).astype(np.float64)
        dg = dA * (lc + p.lin_offset) * s * (1.0 + p.beta * gc * (1.0 - s)) * g_pass
        dl = dA * gc * s * l_pass
        return dg, dl
    if p.kind == "geglu":
        return dA * l * (_Phi(g) + g * _phi(g)), dA * g * _Phi(g)
    if p.kind == "srelu":
        return dA * 2.0 * np.maximum(g, 0.0), None
    raise ValueError(p.kind)


# ----------------------------------------------------------------------------- one expert


def _q(v, axis, mx):
    return mxfp8.fake_quant(v, axis) if mx else v


def _qrows(v, mx):
    return mxfp8.fake_quant_rows_from(v) if mx else v


class ExpertWeights:
    """One expert's weights and, in MXFP8, their quantised copies along each reduction
    direction (computed once, so sampled checks can reuse them across many rows)."""

    def __init__(self, W1, W2, mx: bool):
        self.W1, self.W2 = W1, W2
        self.w1_h = _q(W1, 0, mx)   # FC1 fprop: along H
        self.w1_n = _q(W1, 1, mx)   # FC1 dgrad: along N1
        self.w2_f = _q(W2, 0, mx)   # FC2 fprop: along F
        self.w2_h = _q(W2, 1, mx)   # FC2 dgrad: along H


def expert_forward(X, W1, W2, p, act: ActParams, mx: bool, wq: ExpertWeights | None = None,
                   b1=None, s=None):
    """One expert's share of the fused forward.

    X [m, H] (its routed rows), W1 [H, N1] logical, W2 [F, H], p [m] routing probs.
    Z = X W1 (+ b1);  a = act(gate, lin);  a_s = p * (s * a) (ScaledSwiGLU, R5);  Y = a_s W2.
    Optional epilogue extras ([NV-blog] GLU-epilogue section: bias-vector addition and
    feature scaling; the SwiGLU equation's b and c; reading R13): b1 [N1] logical
    [gate | linear] bias added to Z (which is what the backward sees as the saved Z), s [F] a
    per-feature scale of the activation output. The returned `a` is the unscaled activation.
    [TE-MoE] Challenge 3 (GroupedLinear -> ScaledSwiGLU -> GroupedLinear) and [NV-blog]
    Figure 1 (FC1 + activation + quantise fused, then FC2). In MXFP8 (R8) each GEMM uses
    MXFP8 operands blocked along its reduction dimension: X and W1 along H, a_s and W2 along F.
    `wq` optionally supplies the weights' quantised copies (ExpertWeights of W1, W2).
    """
    wq = wq or ExpertWeights(W1, W2, mx)
    F = W2.shape[0]
    Z = _q(X, 1, mx) @ wq.w1_h
    if b1 is not None:
        Z = Z + b1[None, :]
    if act.gated:
        a = act_forward(act, Z[:, :F], Z[:, F:])
    else:
        a = act_forward(act, Z)
    a_s = p[:, None] * (a * s[None, :] if s is not None else a)
    Y = _q(a_s, 1, mx) @ wq.w2_f
    return Z, a, a_s, Y


def expert_backward(X, W1, W2, p, Z, a, a_s, dY, act: ActParams, mx: bool,
                    wq: ExpertWeights | None = None, s=None, extras: dict | None = None,
                    recompute: bool = False):
    """One expert's share of the backward ([NV-blog] Figure 1: FC2 dgrad + dActivation +
    quantise fused; the weight-gradient GEMMs unfused).

      dA_s = dY W2^T;  d_prob = sum_f dA_s * s * a  (R9);  dA = p * s * dA_s;
      (dG, dL) = dact(Z, dA);  dZ = [dG | dL];
      dW2 = a_s^T dY;  dW1 = X^T dZ;  dX = dZ W1^T.
    With the epilogue extras (s the feature scale, 1 when absent) `extras` receives
    db1 = sum over rows of dZ and ds = sum over rows of p * dA_s * a.
    MXFP8 (R8): dY and W2 along H for dgrad; a_s and dY column-wise (along rows) for dW2;
    dZ along N1 and W1 along N1 for dX; X and dZ column-wise for dW1.
    MXFP8, R15: the E4M3 codes of dZ are integer decisions taken on the values the fused dGLU
    epilogue reads, so the oracle forms dZ from the same inputs: the saved FC1 output in bf16
    (the saved activation is bf16) and the FC2-dgrad result dA_s rounded to bf16 (the
    precision in which the epilogue holds it); d_prob keeps the plain definition. With
    `recompute` (activation recomputation: the epilogue reads Z and dA_s in fp32 from the
    tensor-core accumulators) dZ is formed from the unrounded values.
    """
    wq = wq or ExpertWeights(W1, W2, mx)
    F = W2.shape[0]
    dA_s = _q(dY, 1, mx) @ wq.w2_h.T
    sa = a * s[None, :] if s is not None else a
    d_prob = (dA_s * sa).sum(axis=1)
    dA_in, Z_in = (bf16_round(dA_s), bf16_round(Z)) if mx and not recompute else (dA_s, Z)
    dA = p[:, None] * (dA_in * s[None, :] if s is not None else dA_in)
    if act.gated:
        dg, dl = act_backward(act, Z_in[:, :F], Z_in[:, F:], dA)
        dZ = np.concatenate([dg, dl], axis=1)
    else:
        dZ, _ = act_backward(act, Z_in, None, dA)
    dW2 = _qrows(a_s, mx).T @ _qrows(dY, mx)
    dW1 = _qrows(X, mx).T @ _qrows(dZ, mx)
    dX = _q(dZ, 1, mx) @ wq.w1_n.T
    if extras is not None:
        extras["db1"] = dZ.sum(axis=0)
        extras["ds"] = (p[:, None] * dA_s * a).sum(axis=0)
    return dZ, dX, dW1, dW2, d_prob


# ----------------------------------------------------------------------------- the layer


@dataclass
class LayerResult:
    ids: np.ndarray
    probs: np.ndarray
    perm: Permutation
    y: np.ndarray
    dx: np.ndarray | None = None
    dW1: np.ndarray | None = None
    dW2: np.ndarray | None = None
    d_probs: np.ndarray | None = None
    db1: np.ndarray | None = None      # [E, N1] FC1 bias gradient (when a bias is given)
    ds: np.ndarray | None = None       # [E, F] feature-scale gradient (when a scale is given)
    per_expert: list = field(default_factory=list)   # dicts of intermediates by expert


def layer(logits, x, W1, W2, k: int, act: ActParams, mx: bool = False, align: int = 32,
          dy=None, keep_intermediates: bool = False, experts=None, b1=None,
          s=None, recompute: bool = False) -> LayerResult:
    """Forward (and, when dy is given, backward) of the MoE expert layer.

    logits fp32 [T,E]; x fp64 [T,H]; W1 fp64 [E,H,N1] (or a callable e -> [H,N1]);
    W2 fp64 [E,F,H] (or callable); dy fp64 [T,H].
    y[t] = sum_j Y[row_of[t,j]]: the index_add of [TE-MoE] Challenge 1's per-expert loop.
    `experts` restricts the computation to a subset (y / dx then hold only their share).
    b1 [E, N1] and s [E, F] are the optional epilogue extras (expert_forward).
    """
    T, E = np.asarray(logits).shape
    ids, probs = route(logits, k)
    perm = permutation(ids, E, align)
    H = x.shape[1]
    w1 = W1 if callable(W1) else (lambda e: W1[e])
    w2 = W2 if callable(W2) else (lambda e: W2[e])
    y = np.zeros((T, H))
    res = LayerResult(ids, probs, perm, y)
    if dy is not None:
        res.dx = np.zeros((T, H))
        res.d_probs = np.zeros((T, k))
        res.dW1, res.dW2 = {}, {}
        if b1 is not None:
            res.db1 = np.zeros_like(np.asarray(b1, dtype=np.float64))
        if s is not None:
            res.ds = np.zeros_like(np.asarray(s, dtype=np.float64))
    for e in (range(E) if experts is None else experts):
        tok, slot = perm.rows_of_expert[e]
        W1e, W2e = w1(e), w2(e)
        wq = ExpertWeights(W1e, W2e, mx)
        X = x[tok]
        p = probs[tok, slot]
        b1e = None if b1 is None else b1[e]
        se = None if s is None else s[e]
        Z, a, a_s, Y = expert_forward(X, W1e, W2e, p, act, mx, wq, b1=b1e, s=se)
        np.add.at(y, tok, Y)
        inter = dict(Z=Z, a=a, a_s=a_s, Y=Y) if keep_intermediates else {}
        if dy is not None:
            dY = dy[tok]
            ex = {}
            dZ, dX, dW1, dW2, d_prob = expert_backward(X, W1e, W2e, p, Z, a, a_s, dY, act, mx,
                                                       wq, s=se, extras=ex,
                                                       recompute=recompute)
            if b1 is not None:
                res.db1[e] = ex["db1"]
            if s is not None:
                res.ds[e] = ex["ds"]
            np.add.at(res.dx, tok, dX)
            res.d_probs[tok, slot] = d_prob
            res.dW1[e], res.dW2[e] = dW1, dW2
            if keep_intermediates:
                inter.update(dZ=dZ, dX=dX, d_prob=d_prob)
        res.per_expert.append(inter)
    return res


def stack_weight_grads(res: LayerResult, E: int):
    return np.stack([res.dW1[e] for e in range(E)]), np.stack([res.dW2[e] for e in range(E)])


# ----------------------------------------------------------------------------- NVFP4 layer


def bf16_round(v: np.ndarray) -> np.ndarray:
    """Round to fp32 and then to the nearest bf16 (ties to even), the kernels' order of
    conversions for a value held in fp32; returned as fp64."""
    u = np.asarray(v, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return bf16_to_f64(u.astype(np.uint16))


@dataclass
class Nvfp4Result:
    ids: np.ndarray
    probs: np.ndarray
    perm: Permutation
    y: np.ndarray
    amax: dict                                   # per-tensor amax of every NVFP4 copy
    dx: np.ndarray | None = None
    dW1: np.ndarray | None = None                # [E, H, N1] logical
    dW2: np.ndarray | None = None                # [E, F, H]
    d_probs: np.ndarray | None = None
    Z: list = field(default_factory=list)        # per expert: FC1 output, bf16-rounded
    A: list = field(default_factory=list)        # per expert: a_s, bf16-rounded
    dZ: list = field(default_factory=list)       # per expert: dZ, bf16-rounded
    db1: np.ndarray | None = None                # [E, N1] FC1 bias gradient (with a bias)
    ds: np.ndarray | None = None                 # [E, F] feature-scale gradient (with a scale)


def layer_nvfp4(logits, x, W1, W2, k: int, act: ActParams, mask: int, dy=None,
                align: int = 128, b1=None, s=None, recompute: bool = False) -> Nvfp4Result:
    """Forward (and, with dy, backward) of the expert layer with NVFP4 GEMM operands.

    The same layer as `layer` (R1-R9), with every GEMM consuming NVFP4 copies of its operands
    (oracle.nvfp4, readings N1-N6) blocked along its reduction dimension, and with the BF16
    tensors that the fused kernels emit ([NV-blog] section "fused MXFP8 and NVFP4
    quantisation") rounded to bf16 where the pipeline stores them:
      forward:  Z = Q(X) Q_H(W1)            saved in bf16 (the backward reads the saved Z)
                a_s = bf16(p * act(Z))      the FC1 kernel's BF16 output, with amax(a_s)
                Y = Q(a_s) Q_F(W2)
      backward: dA_s = Q(dY) Q_H(W2)^T, d_prob = sum_f dA_s * a,
                dZ = bf16(dact(bf16 Z, p * bf16 dA_s))   the FC2-dgrad kernel's BF16 output,
                                            with the amax of its Hadamard-rotated transpose
                dX = Q(dZ) Q_N1(W1)^T
                dW2 = Q_rows(RHT(a_s))^T Q_rows(RHT(dY)),  dW1 = Q_rows(RHT(dZ))^T Q_rows(RHT(X))
    Q(.) quantises along the row (the reduction dimension of the row-grouped GEMMs) with its
    tensor's encode scale; Q_rows(RHT(.)) rotates each expert's rows in blocks of 16 from the
    expert's first row (zero rows pad the last block) and quantises down the columns. Every
    per-tensor amax is taken over the whole tensor (all experts). Weights: W1 [E, H, N1]
    logical, W2 [E, F, H]; W1's amax is shared by its two copies, W2's likewise.
    Optional epilogue extras, as in `expert_forward` / `expert_backward` (reading R13): b1
    [E, N1] logical [gate | linear] FC1 bias added to Z before it is saved, s [E, F] a
    per-feature scale of the activation (a_s = p * (a * s); d_prob = sum_f dA_s * s * a;
    dA = p * s * dA_s), with db1 = sum over an expert's rows of dZ (the unrounded dact
    output) and ds = sum over its rows of p * dA_s * a.
    dZ is an input of integer decisions (its NVFP4 codes) whose precision the pages do not fix,
    so it is formed from the dGLU epilogue's inputs as the kernel holds them (reading R14, as
    R15 for MXFP8): the saved Z in bf16 and dA_s rounded to bf16 (the epilogue keeps the FC2
    dgrad accumulator packed to bf16 in TMEM); d_prob, db1's rows and ds keep the plain
    definitions.
    `recompute` (activation recomputation): the backward forms dZ from the FC1 output and
    dA_s as the tensor cores compute them (unrounded, the same quantised operands) instead of
    the saved bf16 copy and the packed dA_s; nothing else changes.
    """
    from . import nvfp4 as nv

    lg = np.asarray(logits, dtype=np.float32)
    T, E = lg.shape
    ids, probs = route(lg, k)
    perm = permutation(ids, E, align)
    H = x.shape[1]
    F = W2.shape[1]
    segs = perm.rows_of_expert
    Xs = [x[tok] for tok, _ in segs]
    Ps = [probs[tok, slot] for tok, slot in segs]
    am = {"x": nv.amax(x), "w1": nv.amax(W1), "w2": nv.amax(W2)}
    S = lambda name: nv.encode_scale(am[name])  # noqa: E731
    xq = nv.fake_quant(x, 1, S("x")) if T else x
    y = np.zeros((T, H))
    res = Nvfp4Result(ids, probs, perm, y, am)
    acts, z_full = [], []
    for e in range(E):
        tok, _ = segs[e]
        Ze = xq[tok] @ nv.fake_quant(W1[e], 0, S("w1"))
        if b1 is not None:
            Ze = Ze + np.asarray(b1[e], dtype=np.float64)[None, :]
        z_full.append(Ze)
        ae = act_forward(act, Ze[:, :F], Ze[:, F:]) if act.gated else act_forward(act, Ze)
        acts.append(ae)
        res.Z.append(bf16_round(Ze))
        sa = ae * np.asarray(s[e], dtype=np.float64)[None, :] if s is not None else ae
        res.A.append(bf16_round(Ps[e][:, None] * sa))
    am["a"] = max([nv.amax(a) for a in res.A] + [0.0])
    am["at"] = nv.rht_amax_segments(res.A, mask)
    for e in range(E):
        tok, _ = segs[e]
        if len(tok):
            Ye = nv.fake_quant(res.A[e], 1, S("a")) @ nv.fake_quant(W2[e], 0, S("w2"))
            np.add.at(y, tok, Ye)
    if dy is None:
        return res
    dy = np.asarray(dy, dtype=np.float64)
    DYs = [dy[tok] for tok, _ in segs]
    am["dy"] = nv.amax(dy)
    am["dyt"] = nv.rht_amax_segments(DYs, mask)
    am["xt"] = nv.rht_amax_segments(Xs, mask)
    dyq = nv.fake_quant(dy, 1, S("dy")) if T else dy
    res.dx = np.zeros((T, H))
    res.d_probs = np.zeros((T, k))
    res.dW1 = np.zeros((E,) + W1.shape[1:])
    res.dW2 = np.zeros((E,) + W2.shape[1:])
    if b1 is not None:
        res.db1 = np.zeros((E, W1.shape[2]))
    if s is not None:
        res.ds = np.zeros((E, F))
    for e in range(E):
        tok, slot = segs[e]
        dA_s = dyq[tok] @ nv.fake_quant(W2[e], 1, S("w2")).T
        se = np.asarray(s[e], dtype=np.float64)[None, :] if s is not None else 1.0
        res.d_probs[tok, slot] = (dA_s * se * acts[e]).sum(axis=1)
        dA = Ps[e][:, None] * ((dA_s if recompute else bf16_round(dA_s)) * se)
        Zb = z_full[e] if recompute else res.Z[e]
        if act.gated:
            dg, dl = act_backward(act, Zb[:, :F], Zb[:, F:], dA)
            dZe = np.concatenate([dg, dl], axis=1)
        else:
            dZe, _ = act_backward(act, Zb, None, dA)
        res.dZ.append(bf16_round(dZe))
        if b1 is not None:
            res.db1[e] = dZe.sum(axis=0)
        if s is not None:
            res.ds[e] = (Ps[e][:, None] * dA_s * acts[e]).sum(axis=0)
    am["dz"] = max([nv.amax(d) for d in res.dZ] + [0.0])
    am["dzt"] = nv.rht_amax_segments(res.dZ, mask)
    at_q = nv.colwise_rht_segments(res.A, mask, S("at"))
    dyt_q = nv.colwise_rht_segments(DYs, mask, S("dyt"))
    dzt_q = nv.colwise_rht_segments(res.dZ, mask, S("dzt"))
    xt_q = nv.colwise_rht_segments(Xs, mask, S("xt"))
    for e in range(E):
        tok, _ = segs[e]
        if len(tok):
            dXe = nv.fake_quant(res.dZ[e], 1, S("dz")) @ nv.fake_quant(W1[e], 1, S("w1")).T
            np.add.at(res.dx, tok, dXe)
        res.dW2[e] = at_q[e].T @ dyt_q[e]
        res.dW1[e] = xt_q[e].T @ dzt_q[e]
    return res
