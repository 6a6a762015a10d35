"""Pins for oracle.nvfp4 and oracle.moe.layer_nvfp4, each against something other than the
code under test: the E2M1 value set worked out from its bit layout, brute-force nearest
rounding, a hand-derived worked example of the two-level scaling, lossless round trips,
scipy's Hadamard matrix, the rotation's orthogonality, torch's bf16 conversion, and the BF16
oracle (the NVFP4 layer with its quantisers taken out must equal it)."""
import numpy as np
import pytest
import scipy.linalg
import torch

from oracle import moe as om
from oracle import nvfp4 as nv

F32_MAX = float(np.finfo(np.float32).max)


# ----------------------------------------------------------------------------- E2M1


def test_e2m1_value_set_from_its_bit_layout():
    # 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent field 0 is subnormal (no implicit 1)
    want = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    t = nv.e2m1_decode_table()
    assert list(t[:8]) == want
    assert list(t[8:]) == [-v for v in want]
    assert np.signbit(t[8])


def _brute_round(v):
    """Nearest E2M1 magnitude by exhaustive search; a tie goes to the even code (the value
    whose code has mantissa bit 0); beyond 6 saturates."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    out = []
    for x in v:
        a = min(abs(x), 6.0)
        d = [abs(a - m) for m in mags]
        best = min(d)
        cands = [i for i, di in enumerate(d) if di == best]
        i = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
        out.append(np.copysign(mags[i], x))
    return np.array(out)


def test_e2m1_rounding_matches_brute_force_including_every_tie():
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    rng = np.random.default_rng(1)
    v = np.concatenate([grid, mids, 6.5 + np.arange(4.0), rng.uniform(-8, 8, 4000),
                        np.nextafter(np.array(mids), 0), np.nextafter(np.array(mids), 10)])
    v = np.concatenate([v, -v])
    assert np.array_equal(nv.e2m1_round(v), _brute_round(v))
    # the ties by name: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    assert list(nv.e2m1_round(np.array(mids))) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_e2m1_codes_round_trip_and_keep_the_sign_of_zero():
    t = nv.e2m1_decode_table()
    assert np.array_equal(nv.e2m1_encode(t), np.arange(16, dtype=np.uint8))
    assert nv.e2m1_encode(np.array([-0.1]))[0] == 0x8
    assert nv.e2m1_encode(np.array([0.1]))[0] == 0x0


# ----------------------------------------------------------------------------- scales


def test_encode_scale_special_values():
    assert nv.encode_scale(2688.0) == np.float32(1.0)
    assert nv.encode_scale(1.0) == np.float32(2688.0)
    assert nv.encode_scale(0.0) == np.float32(F32_MAX)
    assert nv.encode_scale(1e-38) == np.float32(F32_MAX)   # 2688 / 1e-38 overflows fp32


def test_worked_example_of_the_two_level_scaling():
    """Hand derivation (S = 1, from a tensor amax of 2688 = 6 * 448):
    block 0 amax 2688: t = 2688/6 * 1 = 448 -> s_b = 448 (E4M3 max); 2688 * (1/448) = 6 -> 6,
       -1344 / 448 = -3 -> -3, 100 / 448 = 0.2232 -> 0 (nearer 0 than 0.5).
    block 1 amax 7: t = 7/6 = 1.1667 -> E4M3 spacing 1/8 in [1, 2): 1.125 (|d| 0.042 < 0.083);
       factor S / s_b = 1/1.125 = 0.8889; 7 -> 6.22 -> 6 (saturates), 5 -> 4.44 -> 4,
       1 -> 0.889 -> 1, 0.75 -> 0.667 -> 0.5, -0.25 -> -0.222 -> -0 (code 8).
    block 2 all zero: s_b = 0, codes 0."""
    v = np.zeros(48)
    v[0], v[1], v[2] = 2688.0, -1344.0, 100.0
    v[16:21] = [7.0, 5.0, 1.0, 0.75, -0.25]
    codes, sb = nv.quantize_blocks(v[None, :], 1, nv.encode_scale(nv.amax(v)))
    assert list(sb[0]) == [448.0, 1.125, 0.0]
    assert list(codes[0, :3]) == [0x7, 0xD, 0x0]         # 6, -3, 0
    assert list(codes[0, 16:21]) == [0x7, 0x6, 0x2, 0x1, 0x8]
    assert not codes[0, 32:].any()
    deq = nv.dequantize_blocks(codes, sb, 1, 1.0)[0]
    assert list(deq[:3]) == [2688.0, -1344.0, 0.0]
    assert list(deq[16:21]) == [6.75, 4.5, 1.125, 0.5625, 0.0]


def test_lossless_when_every_block_is_on_its_grid():
    """Blocks whose values are E2M1 values times 2^j with the block maximum 6 * 2^j, in a
    tensor whose amax is 6 * 448 (S = 1): every scale is exact and nothing is lost."""
    rng = np.random.default_rng(2)
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    rows = []
    for j in [-6, -2, 0, 3, 8]:
        b = rng.choice(mags, 16) * rng.choice([-1.0, 1.0], 16)
        b[rng.integers(16)] = 6.0
        rows.append(b * 2.0 ** j)
    blk = np.concatenate(rows)
    blk[-16:] *= 448.0 / 256.0          # the last block's scale is 448 = 1.75 * 2^8
    v = np.stack([blk, -blk])
    S = nv.encode_scale(nv.amax(v))
    assert S == np.float32(1.0)
    assert np.array_equal(nv.fake_quant(v, 1, S), v)
    assert np.array_equal(nv.fake_quant(v.T, 0, S), v.T)   # blocks down the columns


def test_dequantised_value_is_the_nearest_point_of_its_blocks_grid():
    rng = np.random.default_rng(3)
    v = om.bf16_round(rng.standard_normal((8, 64)) * np.exp(rng.uniform(-3, 3, (8, 1))))
    S = nv.encode_scale(nv.amax(v))
    codes, sb = nv.quantize_blocks(v, 1, S)
    deq = nv.dequantize_blocks(codes, sb, 1, S)
    grid = nv.e2m1_decode_table()
    for r in range(v.shape[0]):
        for b in range(v.shape[1] // 16):
            pts = grid * sb[r, b] / float(S)
            for i in range(16 * b, 16 * b + 16):
                x = v[r, i]
                best = np.min(np.abs(pts - x))
                # the encoding factor S/s_b is an fp32 rounding of the exact ratio; allow that
                # relative slack, and saturation at the block's largest point
                sat = abs(x) > 6.0 * sb[r, b] / float(S)
                assert sat or abs(deq[r, i] - x) <= best * (1 + 1e-6) + 1e-300


def test_quantize_rejects_values_that_are_not_fp32():
    with pytest.raises(ValueError):
        nv.quantize_blocks(np.full((1, 16), 1.0 + 2.0 ** -40), 1, 1.0)


# ----------------------------------------------------------------------------- RHT


def test_rotation_is_scipys_hadamard_with_the_sign_vector():
    rng = np.random.default_rng(4)
    mask = 0b1010011100010110
    v = rng.standard_normal((48, 5))
    d = np.array([(-1.0 if (mask >> j) & 1 else 1.0) for j in range(16)])
    Q = scipy.linalg.hadamard(16) * d[None, :] / 4.0
    want = np.concatenate([Q @ v[16 * b:16 * b + 16] for b in range(3)])
    assert np.allclose(nv.rht_rows(v, mask), want, rtol=0, atol=1e-14)


def test_rotation_entries_by_popcount():
    """H[i][j] = (-1)^popcount(i & j), checked on unit vectors."""
    for j in range(16):
        e = np.zeros((16, 1))
        e[j] = 1.0
        col = nv.rht_rows(e, 0)[:, 0]
        want = np.array([0.25 * (-1) ** bin(i & j).count("1") for i in range(16)])
        assert np.array_equal(col, want)


def test_rotation_preserves_the_weight_gradient_product():
    rng = np.random.default_rng(5)
    a, b = rng.standard_normal((64, 7)), rng.standard_normal((64, 9))
    for mask in (0, 0xFFFF, 0x5A3C):
        ra, rb = nv.rht_rows(a, mask), nv.rht_rows(b, mask)
        assert np.allclose(ra.T @ rb, a.T @ b, rtol=1e-12, atol=1e-12)
    assert np.allclose(nv.rht_rows(nv.rht_rows(a, 0), 0), a, atol=1e-14)   # H/4 is symmetric


def test_rht_amax_segments_pads_each_segment_from_its_first_row():
    rng = np.random.default_rng(6)
    segs = [rng.standard_normal((m, 3)) for m in (0, 5, 16, 21)]
    want = 0.0
    for s in segs:
        for c in range(3):
            col = np.concatenate([s[:, c], np.zeros(-len(s) % 16)])
            for b in range(len(col) // 16):
                x = col[16 * b:16 * b + 16] * nv.sign_vector(0x00F0)
                for i in range(16):
                    y = 0.25 * sum((-1) ** bin(i & j).count("1") * x[j] for j in range(16))
                    want = max(want, abs(y))
    assert np.isclose(nv.rht_amax_segments(segs, 0x00F0), want, rtol=1e-14)


# ----------------------------------------------------------------------------- the layer


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(7)
    v = rng.standard_normal(5000) * np.exp(rng.uniform(-20, 20, 5000))
    want = torch.from_numpy(v).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(om.bf16_round(v), want)


def _small_layer(seed=8, T=48, E=4, H=64, F=64, k=2):
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    x = om.bf16_round(rng.standard_normal((T, H)))
    W1 = om.bf16_round(0.1 * rng.standard_normal((E, H, 2 * F)))
    W2 = om.bf16_round(0.1 * rng.standard_normal((E, F, H)))
    dy = om.bf16_round(rng.standard_normal((T, H)))
    return lg, x, W1, W2, dy, k


_ACTS = {
    "swiglu": om.ActParams(),
    "clamped_swiglu": om.ActParams("clamped_swiglu", 1.702, 2.0, -2.0, 2.0, 1.0),
    "geglu": om.ActParams("geglu"),
    "srelu": om.ActParams("srelu"),
}


@pytest.mark.parametrize("kind,skew", [("swiglu", False), ("clamped_swiglu", True),
                                       ("geglu", False), ("srelu", True)])
def test_layer_without_quantisers_is_the_bf16_oracle(monkeypatch, kind, skew):
    """Taking out the quantisers and the bf16 roundings leaves the plain layer: this pins the
    stage-by-stage plumbing (segments, the d_prob and weight-gradient products, the rotation
    of both weight-gradient operands, which cancels), for every activation, and with routing
    skewed so that some experts get no tokens."""
    lg, x, W1, W2, dy, k = _small_layer(E=8 if skew else 4)
    if skew:
        lg = lg.copy()
        lg[:, :3] += 4.0        # experts 0-2 take (nearly) every token
    act = _ACTS[kind]
    if not act.gated:
        W1 = W1[:, :, :W2.shape[1]]
    monkeypatch.setattr(nv, "fake_quant", lambda v, axis, S: np.asarray(v, dtype=np.float64))
    monkeypatch.setattr(nv, "to_f32", lambda v: np.asarray(v, dtype=np.float64))
    monkeypatch.setattr(om, "bf16_round", lambda v: np.asarray(v, dtype=np.float64))
    got = om.layer_nvfp4(lg, x, W1, W2, k, act, 0x3C5A, dy=dy)
    ref = om.layer(lg, x, W1, W2, k, act, dy=dy)
    if skew:
        assert (np.bincount(got.ids.ravel(), minlength=W1.shape[0]) == 0).any()
    dW1, dW2 = om.stack_weight_grads(ref, W1.shape[0])
    for a, b in [(got.y, ref.y), (got.dx, ref.dx), (got.dW1, dW1), (got.dW2, dW2),
                 (got.d_probs, ref.d_probs)]:
        assert np.allclose(a, b, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("kind", ["swiglu", "clamped_swiglu", "geglu"])
def test_layer_extras_without_quantisers_are_the_bf16_oracles(monkeypatch, kind):
    """The epilogue extras (FC1 bias, feature scale) with the quantisers and roundings taken
    out: the layer and both extras gradients equal the plain oracle's, whose extras are
    pinned against autograd (test_oracle_moe)."""
    lg, x, W1, W2, dy, k = _small_layer(seed=12)
    E, F = W1.shape[0], W2.shape[1]
    rng = np.random.default_rng(13)
    b1 = 0.3 * rng.standard_normal((E, 2 * F))
    s = rng.uniform(0.5, 1.5, size=(E, F))
    act = _ACTS[kind]
    monkeypatch.setattr(nv, "fake_quant", lambda v, axis, S: np.asarray(v, dtype=np.float64))
    monkeypatch.setattr(nv, "to_f32", lambda v: np.asarray(v, dtype=np.float64))
    monkeypatch.setattr(om, "bf16_round", lambda v: np.asarray(v, dtype=np.float64))
    got = om.layer_nvfp4(lg, x, W1, W2, k, act, 0x3C5A, dy=dy, b1=b1, s=s)
    ref = om.layer(lg, x, W1, W2, k, act, dy=dy, b1=b1, s=s)
    dW1, dW2 = om.stack_weight_grads(ref, E)
    for a, b in [(got.y, ref.y), (got.dx, ref.dx), (got.dW1, dW1), (got.dW2, dW2),
                 (got.d_probs, ref.d_probs), (got.db1, ref.db1), (got.ds, ref.ds)]:
        assert np.allclose(a, b, rtol=1e-10, atol=1e-10)


def test_layer_extras_neutral_values_and_power_of_two_scale():
    """With the quantisers in place: a zero bias and a unit scale change nothing, bit for bit;
    a feature scale of 2 doubles a_s, y, dZ, dx, both weight gradients and d_prob exactly
    (each NVFP4 encode scale halves with its amax, so every code stays the same) and leaves
    Z and ds unchanged."""
    lg, x, W1, W2, dy, k = _small_layer(seed=14)
    E, F = W1.shape[0], W2.shape[1]
    act = om.ActParams()
    base = om.layer_nvfp4(lg, x, W1, W2, k, act, 0x0F0F, dy=dy)
    zero = om.layer_nvfp4(lg, x, W1, W2, k, act, 0x0F0F, dy=dy, b1=np.zeros((E, 2 * F)),
                          s=np.ones((E, F)))
    for a, b in [(zero.y, base.y), (zero.dx, base.dx), (zero.dW1, base.dW1),
                 (zero.dW2, base.dW2), (zero.d_probs, base.d_probs)]:
        assert np.array_equal(a, b)
    two = om.layer_nvfp4(lg, x, W1, W2, k, act, 0x0F0F, dy=dy, s=np.full((E, F), 2.0))
    for a, b in [(two.y, base.y), (two.dx, base.dx), (two.dW1, base.dW1),
                 (two.dW2, base.dW2), (two.d_probs, base.d_probs)]:
        assert np.array_equal(a, 2.0 * b)
    for e in range(E):
        assert np.array_equal(two.Z[e], base.Z[e])
        assert np.array_equal(two.A[e], 2.0 * base.A[e])
        assert np.array_equal(two.dZ[e], 2.0 * base.dZ[e])
    assert np.array_equal(two.ds, zero.ds)


def test_layer_bias_enters_the_saved_fc1_output():
    """With W1 = 0 the FC1 output is the bias alone: every row of an expert's saved Z is its
    bias (rounded to bf16), in logical [gate | linear] order."""
    lg, x, W1, W2, dy, k = _small_layer(seed=15)
    E, F = W1.shape[0], W2.shape[1]
    b1 = om.bf16_round(np.random.default_rng(16).standard_normal((E, 2 * F)))
    r = om.layer_nvfp4(lg, x, np.zeros_like(W1), W2, k, om.ActParams(), 0x1111, dy=dy, b1=b1)
    for e in range(E):
        if len(r.Z[e]):
            assert np.array_equal(r.Z[e], np.broadcast_to(b1[e], r.Z[e].shape))
    assert r.db1 is not None and r.ds is None


def test_layer_recompute_changes_only_the_fc1_output_the_backward_reads():
    """Recomputation: the forward and everything that does not read Z (y, a_s, its amaxes,
    dW2) are identical; dZ is formed from the unrounded Z and dA_s, so it differs from the
    saved-path dZ by about their bf16 roundings only; with the bf16 roundings taken out the
    two coincide."""
    lg, x, W1, W2, dy, k = _small_layer(seed=17)
    act = om.ActParams()
    sv = om.layer_nvfp4(lg, x, W1, W2, k, act, 0x2222, dy=dy)
    rc = om.layer_nvfp4(lg, x, W1, W2, k, act, 0x2222, dy=dy, recompute=True)
    assert np.array_equal(sv.y, rc.y) and np.array_equal(sv.dW2, rc.dW2)
    assert sv.amax["a"] == rc.amax["a"] and sv.amax["at"] == rc.amax["at"]
    for e in range(len(sv.Z)):
        assert np.array_equal(sv.Z[e], rc.Z[e]) and np.array_equal(sv.A[e], rc.A[e])
        if len(sv.dZ[e]):
            d = np.abs(sv.dZ[e] - rc.dZ[e]).max()
            assert d <= 2.0 ** -6 * np.abs(sv.dZ[e]).max()
    assert any(not np.array_equal(a, b) for a, b in zip(sv.dZ, rc.dZ) if len(a))


def test_layer_recompute_without_roundings_is_the_saved_path(monkeypatch):
    """With the quantisers and roundings taken out the saved and the recomputed Z are the same
    value, so the two backward paths coincide exactly."""
    lg, x, W1, W2, dy, k = _small_layer(seed=18)
    monkeypatch.setattr(nv, "fake_quant", lambda v, axis, S: np.asarray(v, dtype=np.float64))
    monkeypatch.setattr(nv, "to_f32", lambda v: np.asarray(v, dtype=np.float64))
    monkeypatch.setattr(om, "bf16_round", lambda v: np.asarray(v, dtype=np.float64))
    act = _ACTS["geglu"]
    sv = om.layer_nvfp4(lg, x, W1, W2, k, act, 0x0F00, dy=dy)
    rc = om.layer_nvfp4(lg, x, W1, W2, k, act, 0x0F00, dy=dy, recompute=True)
    for a, b in [(sv.y, rc.y), (sv.dx, rc.dx), (sv.dW1, rc.dW1), (sv.dW2, rc.dW2),
                 (sv.d_probs, rc.d_probs)]:
        assert np.array_equal(a, b)


def test_layer_error_is_the_size_of_nvfp4_quantisation_noise():
    lg, x, W1, W2, dy, k = _small_layer(seed=9)
    act = om.ActParams()
    got = om.layer_nvfp4(lg, x, W1, W2, k, act, 0x1234, dy=dy)
    ref = om.layer(lg, x, W1, W2, k, act, dy=dy)
    rel = np.linalg.norm(got.y - ref.y) / np.linalg.norm(ref.y)
    # two chained 4-bit GEMMs: far from exact, far from garbage
    assert 0.05 < rel < 0.5


def test_layer_amaxes_are_those_of_the_stored_tensors():
    lg, x, W1, W2, dy, k = _small_layer(seed=10)
    r = om.layer_nvfp4(lg, x, W1, W2, k, om.ActParams(), 0x00FF, dy=dy)
    assert r.amax["x"] == np.abs(x).max() and r.amax["dy"] == np.abs(dy).max()
    assert r.amax["w1"] == np.abs(W1).max() and r.amax["w2"] == np.abs(W2).max()
    assert r.amax["a"] == max(np.abs(a).max() for a in r.A if a.size)
    assert r.amax["dz"] == max(np.abs(d).max() for d in r.dZ if d.size)
    for a in r.A + r.dZ:
        assert np.array_equal(om.bf16_round(a), a)


def test_fake_quant_is_the_dequantised_encoding():
    rng = np.random.default_rng(11)
    v = om.bf16_round(rng.standard_normal((48, 128)) * np.exp(rng.uniform(-6, 6, (48, 1))))
    S = nv.encode_scale(nv.amax(v))
    for axis in (0, 1):
        c, sb = nv.quantize_blocks(v, axis, S)
        assert np.array_equal(nv.fake_quant(v, axis, S), nv.dequantize_blocks(c, sb, axis, S))
