"""NVFP4 (E2M1 elements, one E4M3 scale per 16 values, one fp32 scale per tensor) and the
16-point random Hadamard rotation, in fp64 with the quantiser's decisions taken in fp32.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages name NVFP4 as the second low-precision recipe whose quantisation the fused kernels
prepare ([NV-blog] section "fused MXFP8 and NVFP4 quantisation": the forward kernel emits its
BF16 output plus a per-tensor amax, the backward kernel the amax of the Hadamard-rotated
transposed output), and as Blackwell's 4-bit float format ([MoE-summary], the NVIDIA
hardware list, Blackwell item). They do not define the format; this module takes the
published NVFP4 definition:

  element  E2M1: s ee m, exponent bias 1; e == 0: (-1)^s * m/2, else (-1)^s * (1 + m/2) *
           2^(e-1). Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 (no Inf/NaN).
  block    16 consecutive values along the GEMM's reduction dimension share one unsigned
           E4M3 scale s_b;
  tensor   one fp32 encode scale S per tensor, from the tensor's amax.

Readings (the pages leave these open; every step below is in fp32 with round-to-nearest-even,
the precision the kernels take them in):
  N1  S = min(6 * 448 / amax, FLT_MAX)  (amax == 0 gives +inf, hence FLT_MAX): the block with
      the tensor's largest value gets the largest E4M3 scale, 448.
  N2  s_b = E4M3_RNE_sat( fp32(amax_b / 6) * S ): the scale maps the block maximum onto
      E2M1's largest magnitude, 6.
  N3  q = E2M1_RNE_sat( x * fp32(S / s_b) ), with the factor 0 when s_b == 0 (the block is all
      (signed) zeros); the sign of zero is kept, as for E4M3.
  N4  value = E2M1(q) * s_b / S; a GEMM on two NVFP4 operands accumulates
      sum (q_a s_a)(q_b s_b) and multiplies by 1 / (S_a S_b).
  N5  Random Hadamard transform (RHT): y = (1/4) H16 diag(d) x on each block of 16 along the
      token dimension, H16 the Sylvester Hadamard matrix (H[i][j] = (-1)^popcount(i & j)) and
      d a +-1 sign vector drawn once and passed in (bit j of a 16-bit mask set = -1). It is
      applied to the weight-gradient operands (the column-wise copies) only; since (1/4)H16 D
      is orthogonal, the weight gradients are unchanged in exact arithmetic.
  N6  no stochastic rounding and no 2-D (16 x 16) weight blocks: the pages mention neither.
"""
from __future__ import annotations

import numpy as np

BLOCK = 16
E2M1_MAX = 6.0
E4M3_MAX = 448.0
FLT_MAX = float(np.finfo(np.float32).max)

from .mxfp8 import e4m3_round  # noqa: E402  (the same E4M3 rounding serves the block scales)


# ----------------------------------------------------------------------------- E2M1


def e2m1_decode_table() -> np.ndarray:
    """Value of each of the 16 codes."""
    vals = np.empty(16, dtype=np.float64)
    for c in range(16):
        s = -1.0 if c & 0x8 else 1.0
        e = (c >> 1) & 0x3
        m = c & 0x1
        vals[c] = s * (m / 2.0) if e == 0 else s * (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return vals


_DECODE = e2m1_decode_table()
_POS = _DECODE[:8].copy()   # 0, 0.5, 1, 1.5, 2, 3, 4, 6 (strictly increasing)


def e2m1_round(v: np.ndarray) -> np.ndarray:
    """Round to the nearest E2M1 value, ties to even, saturating at +-6; sign of zero kept.

    Within the binade [2^E, 2^(E+1)) (E >= 0) the spacing is 2^(E-1); below 1 the subnormal
    spacing is 0.5 = 2^(0-1). So the quantum for |v| is 2^(max(floor(log2|v|), 0) - 1) and
    |v| / quantum is rounded half-to-even (an even multiple is an even mantissa).
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    E = np.maximum(((a.view(np.int64) >> 52) & 0x7FF) - 1023, 0)
    quantum = ((E - 1 + 1023) << 52).view(np.float64)
    inv_quantum = ((1 - E + 1023) << 52).view(np.float64)
    r = np.minimum(np.rint(a * inv_quantum) * quantum, E2M1_MAX)
    return np.copysign(r, v)


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """fp64 -> E2M1 codes (uint8 0..15), RNE, saturating; sign of zero kept."""
    r = e2m1_round(v)
    mag = np.abs(r)
    idx = np.searchsorted(_POS, mag)
    if not np.all(_POS[np.minimum(idx, 7)] == mag):
        raise AssertionError("e2m1_round produced a non-representable value")
    return (idx.astype(np.uint8) | (np.signbit(r).astype(np.uint8) << 3)).astype(np.uint8)


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    return _DECODE[np.asarray(codes, dtype=np.uint8)]


# ----------------------------------------------------------------------------- scales (fp32)


def encode_scale(amax) -> np.float32:
    """N1: the per-tensor encode scale S (fp32)."""
    a = np.float32(amax)
    with np.errstate(divide="ignore", over="ignore"):
        s = np.float32(6.0 * 448.0) / a
    return np.float32(min(float(s), FLT_MAX))


def _blocks(v: np.ndarray, axis: int):
    v = np.asarray(v, dtype=np.float64)
    axis = axis % v.ndim
    n = v.shape[axis]
    if n % BLOCK:
        raise ValueError("blocked axis must be a multiple of 16")
    vm = np.moveaxis(v, axis, -1)
    return vm.reshape(vm.shape[:-1] + (n // BLOCK, BLOCK)), vm.shape, axis


def _round_blocks(v: np.ndarray, axis: int, S):
    """N2, N3 up to the E2M1 rounding: returns (the rounded E2M1 values per block [..., n/16,
    16] fp64, the E4M3 scale values [..., n/16] fp64, v's moved shape, axis)."""
    S = np.float32(S)
    b, shape, axis = _blocks(v, axis)
    b32 = b.astype(np.float32)
    if not np.array_equal(b32.astype(np.float64), b):
        raise ValueError("NVFP4 quantisation takes fp32-representable values")
    amax_b = np.abs(b32).max(axis=-1)
    t = (amax_b / np.float32(6.0)).astype(np.float32) * S          # fp32 products
    sb = e4m3_round(t.astype(np.float32).astype(np.float64))       # RNE + saturation
    sb32 = sb.astype(np.float32)
    with np.errstate(divide="ignore"):
        enc = np.where(sb32 > 0, S / np.where(sb32 > 0, sb32, np.float32(1)), np.float32(0))
    w = (b32 * enc.astype(np.float32)[..., None]).astype(np.float32)
    return e2m1_round(w.astype(np.float64)), sb, shape, axis


def quantize_blocks(v: np.ndarray, axis: int, S):
    """N2, N3: NVFP4-quantise along `axis` (a multiple of 16 long) with encode scale S.

    v must hold fp32-representable values (the kernels quantise fp32 values). Returns
    (E2M1 codes uint8 with v's shape, E4M3 scale values fp64 with v's shape except axis/16).
    """
    r, sb, shape, axis = _round_blocks(v, axis, S)
    codes = e2m1_encode(r).reshape(shape)
    return np.moveaxis(codes, -1, axis), np.moveaxis(sb, -1, axis)


def dequantize_blocks(codes: np.ndarray, sb: np.ndarray, axis: int, S) -> np.ndarray:
    """N4: E2M1(q) * s_b / S."""
    codes = np.asarray(codes)
    axis = axis % codes.ndim
    cm = np.moveaxis(codes, axis, -1)
    sm = np.moveaxis(np.asarray(sb, dtype=np.float64), axis, -1)
    vals = e2m1_decode(cm).reshape(cm.shape[:-1] + (cm.shape[-1] // BLOCK, BLOCK))
    out = vals * sm[..., None] / float(np.float32(S))
    return np.moveaxis(out.reshape(cm.shape), -1, axis)


def fake_quant(v: np.ndarray, axis: int, S) -> np.ndarray:
    """Quantise along `axis` and return the dequantised fp64 values, E2M1(q) * s_b / S: the
    values quantize_blocks encodes, taken straight from the rounding (no code-table round
    trip, so that it is fast on full-size weights)."""
    r, sb, shape, axis = _round_blocks(v, axis, S)
    out = r * sb[..., None] / float(np.float32(S))
    return np.moveaxis(out.reshape(shape), -1, axis)


def amax(v: np.ndarray) -> float:
    v = np.asarray(v, dtype=np.float64)
    return float(np.abs(v).max()) if v.size else 0.0


# ----------------------------------------------------------------------------- RHT


def sylvester_hadamard(n: int = BLOCK) -> np.ndarray:
    """H_1 = [1], H_2m = [[H_m, H_m], [H_m, -H_m]]."""
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def sign_vector(mask: int) -> np.ndarray:
    """N5: d_j = -1 where bit j of the 16-bit mask is set, else +1."""
    return np.array([-1.0 if (mask >> j) & 1 else 1.0 for j in range(BLOCK)])


def rht_rows(v: np.ndarray, mask: int) -> np.ndarray:
    """N5 along axis 0 (the token rows), blocks of 16 from the first row; the row count must
    be a multiple of 16. Returns fp64."""
    v = np.asarray(v, dtype=np.float64)
    m = v.shape[0]
    if m % BLOCK:
        raise ValueError("row count must be a multiple of 16")
    Q = 0.25 * sylvester_hadamard() * sign_vector(mask)[None, :]   # (1/4) H16 diag(d)
    blocks = v.reshape((m // BLOCK, BLOCK) + v.shape[1:])
    return np.einsum("ij,bj...->bi...", Q, blocks).reshape(v.shape)


def pad_rows16(v: np.ndarray) -> np.ndarray:
    """Zero rows appended up to the next multiple of 16 (a segment's zero padding rows)."""
    v = np.asarray(v, dtype=np.float64)
    m = v.shape[0]
    mp = -(-m // BLOCK) * BLOCK
    out = np.zeros((mp,) + v.shape[1:])
    out[:m] = v
    return out


def to_f32(v: np.ndarray) -> np.ndarray:
    """Round fp64 values to fp32 (the kernels' working precision), returned as fp64."""
    return np.asarray(v, dtype=np.float64).astype(np.float32).astype(np.float64)


def colwise_rht_segments(segments: list, mask: int, S) -> list:
    """The weight-gradient (column-wise) copy of a token-row tensor given per expert segment:
    each segment [m_e, N] is zero-padded to a multiple of 16 rows, rotated (N5) in fp64,
    rounded to fp32 and quantised in 16-row blocks along the rows with encode scale S.
    Returns the dequantised padded segments."""
    out = []
    for seg in segments:
        r = to_f32(rht_rows(pad_rows16(seg), mask))
        out.append(fake_quant(r, 0, S) if r.shape[0] else r)
    return out


def rht_amax_segments(segments: list, mask: int) -> float:
    """amax over all segments of the rotated (N5) rows, fp64."""
    m = 0.0
    for seg in segments:
        if np.asarray(seg).shape[0]:
            m = max(m, amax(rht_rows(pad_rows16(seg), mask)))
    return m
