"""Pins for oracle.mxfp8 against things other than itself: the E4M3 bit layout enumerated
code by code, brute-force nearest-value search, torch's float8_e4m3fn cast (a library
routine, in-range values), math.log2 / math.frexp for the scale rule, and exhaustive bf16."""
import math

import numpy as np
import pytest
import torch

from oracle import mxfp8

# Brute-force table built here from the format's definition, independently of the oracle:
# E4M3FN: bias 7, subnormals m/8*2^-6, max 448, S.1111.111 is NaN.


def _table():
    out = {}
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        out[c] = -mag if s else mag
    return out


TABLE = _table()
POS = sorted((v, c) for c, v in TABLE.items() if c < 0x80)


def brute_round(x: float) -> float:
    """Nearest E4M3 magnitude by exhaustive search; ties to the even code; saturating."""
    a = abs(x)
    if a >= 448.0:
        r = 448.0
    else:
        best = min(POS, key=lambda vc: (abs(vc[0] - a), vc[1] & 1))
        r = best[0]
    return math.copysign(r, x)


def test_decode_table_matches_format():
    dec = mxfp8.e4m3_decode_table()
    for c in range(256):
        if c in TABLE:
            assert dec[c] == TABLE[c], c
        else:
            assert np.isnan(dec[c])
    assert dec[0x7E] == 448.0 and dec[0x01] == 2.0 ** -9 and dec[0x08] == 2.0 ** -6


def test_every_code_roundtrips():
    codes = np.array(sorted(TABLE), dtype=np.uint8)
    vals = mxfp8.e4m3_decode(codes)
    back = mxfp8.e4m3_encode(vals)
    # +0 and -0 keep their sign bits
    assert np.array_equal(back, codes)


def test_midpoints_round_half_to_even_and_neighbours():
    mags = [v for v, _ in POS]
    for i in range(len(mags) - 1):
        lo, hi = mags[i], mags[i + 1]
        mid = 0.5 * (lo + hi)
        want = brute_round(mid)
        got = float(mxfp8.e4m3_round(np.array([mid]))[0])
        assert got == want, (lo, hi, got, want)
        # the even one of the two codes wins the tie
        assert mxfp8.e4m3_encode(np.array([mid]))[0] % 2 == 0
        eps = (hi - lo) * 1e-6
        assert mxfp8.e4m3_round(np.array([mid - eps]))[0] == lo
        assert mxfp8.e4m3_round(np.array([mid + eps]))[0] == hi
        assert mxfp8.e4m3_round(np.array([-mid]))[0] == -want


def test_saturation_and_tiny():
    v = np.array([448.0, 449.0, 464.0, 479.9, 480.0, 511.9, 1e30, -1e30, 2.0 ** -11, -2.0 ** -11,
                  2.0 ** -10, 3 * 2.0 ** -11])
    r = mxfp8.e4m3_round(v)
    assert list(r[:8]) == [448.0] * 6 + [448.0, -448.0]
    assert r[8] == 0.0 and np.signbit(r[9])               # below half the smallest subnormal
    assert r[10] == 0.0                                     # exactly half: tie to even (0)
    assert r[11] == 2.0 ** -9                               # 0.75 of a 2^-9 quantum rounds up
    codes = mxfp8.e4m3_encode(np.array([-0.0, 0.0, -2.0 ** -12]))
    assert list(codes) == [0x80, 0x00, 0x80]


def test_random_values_match_brute_force():
    rng = np.random.default_rng(123)
    v = rng.standard_normal(4000) * np.exp2(rng.integers(-12, 10, 4000))
    got = mxfp8.e4m3_round(v)
    want = np.array([brute_round(float(x)) for x in v])
    assert np.array_equal(got, want)


def test_matches_torch_float8_cast_in_range():
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(200000) * np.exp2(rng.integers(-14, 8, 200000))).astype(np.float32)
    v = v[np.abs(v) <= 448.0]
    t = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = mxfp8.e4m3_encode(v.astype(np.float64))
    # torch rounds a value below the smallest subnormal to a signed zero as well
    assert np.array_equal(ours, t)


def test_block_exponent_rule():
    rng = np.random.default_rng(3)
    amax = np.abs(rng.standard_normal(5000)) * np.exp2(rng.integers(-130, 130, 5000))
    amax = np.concatenate([amax, np.exp2(np.arange(-140, 135, dtype=np.float64)), [0.0]])
    e = mxfp8.block_exponent(amax)
    for a, ee in zip(amax, e):
        if a == 0:
            assert ee == -127
        else:
            want = max(-127, min(127, math.floor(math.log2(a)) - 8))
            # log2 of an exact power of two is exact; elsewhere confirm with frexp
            m, x = math.frexp(a)
            assert want == max(-127, min(127, x - 1 - 8))
            assert ee == want


def _bf16_all_finite():
    bits = np.arange(65536, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    return f[np.isfinite(f)].astype(np.float64)


@pytest.mark.parametrize("e", [-127, -100, -20, -9, -1, 0, 1, 7, 40, 119])
def test_all_bf16_values_under_a_forced_scale(e):
    """Every finite bf16 value v, placed in a block whose amax fixes the exponent e, is
    encoded as the nearest E4M3 value of v/2^e (ties even, saturating), i.e. within half an
    E4M3 ulp of v/2^e when unsaturated."""
    vals = _bf16_all_finite()
    big = 2.0 ** (e + 8)                         # amax giving exactly exponent e
    vals = vals[np.abs(vals) <= big]
    if vals.size == 0:
        pytest.skip("no bf16 value fits")
    nb = -(-vals.size // 31)
    pad = np.zeros(nb * 31)
    pad[: vals.size] = vals
    blocks = np.concatenate([pad.reshape(nb, 31), np.full((nb, 1), big)], axis=1)
    codes, scales = mxfp8.quantize_blocks(blocks, axis=1)
    assert np.all(scales == e + 127)
    q = mxfp8.e4m3_decode(codes[:, :31]).ravel()[: vals.size]
    x = vals / 2.0 ** e
    ax = np.abs(x)
    # half-ulp bound for unsaturated values: 2^(max(floor(log2|x|), -6) - 4)
    with np.errstate(divide="ignore"):
        fl = np.where(ax > 0, np.floor(np.log2(np.where(ax > 0, ax, 1.0))), -6)
    bound = np.exp2(np.maximum(fl, -6) - 4)
    unsat = ax <= 448.0
    assert np.all(np.abs(q - x)[unsat] <= bound[unsat])
    assert np.all(np.abs(q[~unsat]) == 448.0)
    # and it is exactly the brute-force nearest value on a sample
    idx = np.random.default_rng(e + 200).choice(vals.size, size=min(1500, vals.size),
                                                replace=False)
    for i in idx:
        assert q[i] == brute_round(float(x[i]))


def test_quantize_axis_and_permutation_commute():
    rng = np.random.default_rng(11)
    v = rng.standard_normal((64, 96)) * np.exp2(rng.integers(-5, 5, (64, 1)))
    c1, s1 = mxfp8.quantize_blocks(v, axis=1)
    perm = rng.permutation(64)
    c2, s2 = mxfp8.quantize_blocks(v[perm], axis=1)
    assert np.array_equal(c1[perm], c2) and np.array_equal(s1[perm], s2)
    # column-wise = row-wise of the transpose
    c3, s3 = mxfp8.quantize_blocks(v, axis=0)
    c4, s4 = mxfp8.quantize_blocks(v.T.copy(), axis=1)
    assert np.array_equal(c3, c4.T) and np.array_equal(s3, s4.T)
    # an outlier moves only its own block's scale
    w = v.copy()
    w[5, 40] = 1e6
    _, sw = mxfp8.quantize_blocks(w, axis=1)
    diff = np.argwhere(sw != s1)
    assert diff.tolist() == [[5, 1]]


def test_zero_block_and_padding_rows():
    v = np.zeros((32, 32))
    c, s = mxfp8.quantize_blocks(v, axis=0)
    assert np.all(s == 0) and np.all(c == 0)
    rng = np.random.default_rng(1)
    x = rng.standard_normal((40, 32))
    fq = mxfp8.fake_quant_rows_from(x)
    full = np.zeros((64, 32))
    full[:40] = x
    assert np.array_equal(fq, mxfp8.fake_quant(full, 0)[:40])


def test_grouped_colwise_reduces_to_plain_blocks_on_32_aligned_groups():
    # groups that start on multiples of 32 rows and hold multiples of 32 rows: the codes are
    # the plain column-wise codes, and group g's scales are the plain ones shifted by g entries
    rng = np.random.default_rng(5)
    v = rng.standard_normal((192, 64)) * 2.0 ** rng.integers(-20, 20, size=(192, 1))
    off = [0, 64, 64, 160, 192]
    c, s = mxfp8.quantize_colwise_groups(v, off)
    c0, s0 = mxfp8.quantize_blocks(v, axis=0)
    assert np.array_equal(c, c0)
    assert s.shape == (64, 4 * ((6 + 4 + 3) // 4))
    for g in range(4):
        for blk in range(off[g] // 32, off[g + 1] // 32):
            assert np.array_equal(s[:, blk + g], s0[blk])
    owned = {blk + g for g in range(4) for blk in range(off[g] // 32, off[g + 1] // 32)}
    assert not s[:, [j for j in range(s.shape[1]) if j not in owned]].any()


def test_grouped_colwise_brute_force_on_ragged_groups():
    # every element against its own block, found by scanning: amax over the block's rows,
    # exponent by the definition, E4M3 of v / 2^e; empty groups own no entry
    rng = np.random.default_rng(6)
    M, N = 150, 32
    v = rng.standard_normal((M, N)) * 2.0 ** rng.integers(-8, 8, size=(M, 1))
    v[40:45] = 0.0
    off = [0, 7, 7, 40, 45, 113, 150]
    c, s = mxfp8.quantize_colwise_groups(v, off)
    owned = np.zeros(s.shape[1], bool)
    for g in range(len(off) - 1):
        for r in range(off[g], off[g + 1]):
            i = (r - off[g]) // 32
            lo, hi = off[g] + 32 * i, min(off[g] + 32 * i + 32, off[g + 1])
            j = off[g] // 32 + g + i
            owned[j] = True
            for col in range(N):
                amax = max(abs(v[q, col]) for q in range(lo, hi))
                e = -127 if amax == 0 else max(-127, min(127, math.floor(math.log2(amax)) - 8))
                assert s[col, j] == e + 127
                assert c[r, col] == mxfp8.e4m3_encode(np.array([v[r, col] / 2.0 ** e]))[0]
    assert not s[:, ~owned].any()
