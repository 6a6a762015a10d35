"""Pins the oracle's number formats to the facts the pages print (tests/golden/
number_formats.txt): the BF16 bit layout, the E4M3 element layout, the E8M0 scale and the
32-element block. Each check rebuilds the decoding from the printed bit counts alone (plus the
usual sign / biased exponent / implicit-one reading of such a layout), independently of the
oracle's own code."""
import os

import numpy as np

from oracle import moe as om
from oracle import mxfp8

HERE = os.path.dirname(os.path.abspath(__file__))


def _facts():
    out = {}
    for line in open(os.path.join(HERE, "golden", "number_formats.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = (s.strip() for s in line.split("=", 1))
        out[k] = int(v) if v.isdigit() else v
    return out


F = _facts()


def test_fixture_is_self_consistent():
    assert F["bf16.sign_bits"] + F["bf16.exponent_bits"] + F["bf16.mantissa_bits"] == F["bf16.bits"]
    assert 1 + F["mxfp8.element_exponent_bits"] + F["mxfp8.element_mantissa_bits"] == \
        F["mxfp8.element_bits"]
    assert F["mxfp8.element"] == f"E{F['mxfp8.element_exponent_bits']}M{F['mxfp8.element_mantissa_bits']}"
    assert F["mxfp8.scale"] == f"E{F['mxfp8.scale_exponent_bits']}M{F['mxfp8.scale_mantissa_bits']}"


def test_bf16_decoding_follows_the_printed_layout():
    eb, mb = F["bf16.exponent_bits"], F["bf16.mantissa_bits"]
    bias = 2 ** (eb - 1) - 1
    codes = np.arange(2 ** F["bf16.bits"], dtype=np.uint32)
    s = codes >> (eb + mb)
    e = (codes >> mb) & (2 ** eb - 1)
    m = codes & (2 ** mb - 1)
    finite = e != 2 ** eb - 1
    mag = np.where(e == 0, m / 2.0 ** mb * 2.0 ** (1 - bias),
                   (1 + m / 2.0 ** mb) * 2.0 ** (e.astype(np.int64) - bias))
    want = np.where(s == 1, -mag, mag)
    got = om.bf16_to_f64(codes.astype(np.uint16))
    assert np.array_equal(got[finite], want[finite])
    assert np.all(~np.isfinite(got[~finite]))


def test_e4m3_elements_follow_the_printed_layout():
    eb, mb = F["mxfp8.element_exponent_bits"], F["mxfp8.element_mantissa_bits"]
    bias = 2 ** (eb - 1) - 1
    table = mxfp8.e4m3_decode_table()
    assert table.shape == (2 ** F["mxfp8.element_bits"],)
    for c in range(2 ** F["mxfp8.element_bits"]):
        s, e, m = c >> (eb + mb), (c >> mb) & (2 ** eb - 1), c & (2 ** mb - 1)
        if e == 2 ** eb - 1 and m == 2 ** mb - 1:  # the single NaN code of E4M3 (no infinities)
            assert np.isnan(table[c])
            continue
        mag = m / 2.0 ** mb * 2.0 ** (1 - bias) if e == 0 else (1 + m / 2.0 ** mb) * 2.0 ** (e - bias)
        assert table[c] == (-mag if s else mag), c


def test_one_e8m0_scale_per_printed_block():
    n = F["mxfp8.block"]
    rng = np.random.default_rng(0)
    v = rng.standard_normal((3, 4 * n))
    codes, scales = mxfp8.quantize_blocks(v, axis=1)
    assert codes.shape == v.shape and codes.dtype == np.uint8
    assert scales.shape == (3, 4) and scales.dtype == np.uint8  # E8M0: one byte per block
    # a scale byte is a pure power of two 2^(byte - 127): decoding multiplies by it exactly
    deq = mxfp8.dequantize_blocks(codes, scales, axis=1)
    for b in range(4):
        blk = slice(b * n, (b + 1) * n)
        np.testing.assert_array_equal(
            deq[:, blk], mxfp8.e4m3_decode_table()[codes[:, blk]] * 2.0 ** (scales[:, b:b + 1] - 127.0))
    # changing one element can only change its own block's scale and codes
    w = v.copy()
    w[1, n + 5] *= 1000.0
    c2, s2 = mxfp8.quantize_blocks(w, axis=1)
    changed = np.argwhere(s2 != scales)
    assert all(tuple(x) == (1, 1) for x in changed)
    diff_cols = np.unique(np.argwhere(c2 != codes)[:, 1])
    assert np.all((diff_cols >= n) & (diff_cols < 2 * n))
