"""MXFP8 (E4M3 elements + one E8M0 scale per 32 contiguous values) in fp64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Format: [TE-MoE] Challenge 2 and its Figure 3 - 8-bit E4M3 elements sharing one E8M0 scale
per block of 32 consecutive values. The scale rule is the one the layer specification fixes:
    scale = 2^e,  e = clamp(floor(log2(amax)) - 8, -127, 127),  E8M0 byte = e + 127,
    q     = E4M3FN(v / 2^e) with round-to-nearest-even and saturation to +-448.
Readings (the pages leave these open):
  * amax == 0: e = -127 (byte 0), every element encodes as a zero of its own sign.
  * |v / 2^e| in (448, 512) saturates to 448: floor(log2 amax) - 8 leaves the block maximum
    in [256, 512), above E4M3's 448, so saturation (not NaN) is part of the definition.
  * The sign of zero is kept (a conversion of a negative value that rounds to zero gives
    the code 0x80).
  * Inputs are finite; NaN / Inf behaviour is not defined here.

E4M3FN (no infinities): code = s eeee mmm, exponent bias 7,
  e == 0 : (-1)^s * m/8 * 2^-6         (subnormals, smallest 2^-9)
  e >= 1 : (-1)^s * (1 + m/8) * 2^(e-7) (largest finite 1.75 * 2^8 = 448; e=15,m=7 is NaN)
"""
from __future__ import annotations

import numpy as np

BLOCK = 32
E4M3_MAX = 448.0


def e4m3_decode_table() -> np.ndarray:
    """Value of each of the 256 codes (NaN for the two NaN codes)."""
    vals = np.empty(256, dtype=np.float64)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            vals[c] = np.nan
        elif e == 0:
            vals[c] = s * (m / 8.0) * 2.0 ** -6
        else:
            vals[c] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_DECODE = e4m3_decode_table()
# Non-negative finite magnitudes in code order 0x00..0x7E (strictly increasing).
_POS = _DECODE[:0x7F].copy()


def e4m3_round(v: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest E4M3 value, ties to even, saturating at +-448.

    Worked from the format: within the binade [2^E, 2^(E+1)) (E >= -6) the E4M3 spacing is
    2^(E-3); below 2^-6 the subnormal spacing is 2^-9 = 2^(-6-3). So the quantum for |v| is
    2^(max(floor(log2|v|), -6) - 3), and |v| / quantum is rounded half-to-even.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    # floor(log2 a) from the fp64 exponent field (zero and fp64 subnormals give -1023, whose
    # quantum is the subnormal one and which round to 0), floored at the subnormal binade
    E = np.maximum(((a.view(np.int64) >> 52) & 0x7FF) - 1023, -6)
    quantum = ((E - 3 + 1023) << 52).view(np.float64)      # 2^(E-3), exact
    inv_quantum = ((3 - E + 1023) << 52).view(np.float64)  # 2^(3-E), exact
    r = np.rint(a * inv_quantum) * quantum    # rint: half to even
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, v)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """fp64 -> E4M3FN codes (uint8), RNE, saturating; sign of zero kept."""
    r = e4m3_round(v)
    mag = np.abs(r)
    idx = np.searchsorted(_POS, mag)
    if not np.all(_POS[np.minimum(idx, 0x7E)] == mag):
        raise AssertionError("e4m3_round produced a non-representable value")
    sign = np.signbit(r).astype(np.uint8) << 7
    return (idx.astype(np.uint8) | sign).astype(np.uint8)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return _DECODE[np.asarray(codes, dtype=np.uint8)]


def block_exponent(amax: np.ndarray) -> np.ndarray:
    """e = clamp(floor(log2 amax) - 8, -127, 127); amax == 0 -> -127. Exact via frexp."""
    amax = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(amax)
    e = (ex - 1) - 8
    e = np.clip(e, -127, 127)
    return np.where(amax == 0, -127, e).astype(np.int64)


def quantize_blocks(v: np.ndarray, axis: int):
    """MXFP8-quantise along `axis` in blocks of 32 (the axis length must be a multiple of 32).

    Returns (codes uint8 with v's shape, scale bytes uint8 with v's shape except axis/32).
    """
    v = np.asarray(v, dtype=np.float64)
    axis = axis % v.ndim
    n = v.shape[axis]
    if n % BLOCK:
        raise ValueError("blocked axis must be a multiple of 32")
    vm = np.moveaxis(v, axis, -1)
    blocks = vm.reshape(vm.shape[:-1] + (n // BLOCK, BLOCK))
    amax = np.abs(blocks).max(axis=-1)
    e = block_exponent(amax)
    scaled = blocks / np.ldexp(1.0, e)[..., None]
    codes = e4m3_encode(scaled).reshape(vm.shape)
    return (np.moveaxis(codes, -1, axis),
            np.moveaxis((e + 127).astype(np.uint8), -1, axis))


def dequantize_blocks(codes: np.ndarray, scale_bytes: np.ndarray, axis: int) -> np.ndarray:
    codes = np.asarray(codes)
    axis = axis % codes.ndim
    cm = np.moveaxis(codes, axis, -1)
    sm = np.moveaxis(np.asarray(scale_bytes), axis, -1)
    vals = e4m3_decode(cm).reshape(cm.shape[:-1] + (cm.shape[-1] // BLOCK, BLOCK))
    out = vals * np.ldexp(1.0, sm.astype(np.int64) - 127)[..., None]
    return np.moveaxis(out.reshape(cm.shape), -1, axis)


def fake_quant(v: np.ndarray, axis: int) -> np.ndarray:
    """Quantise to MXFP8 along `axis` and return the dequantised fp64 values:
    2^e * E4M3_RNE(v / 2^e) per block of 32, the same values quantize_blocks encodes (taken
    straight from the rounding, without the code-table round trip, so that it is fast on
    full-size weights)."""
    v = np.asarray(v, dtype=np.float64)
    axis = axis % v.ndim
    n = v.shape[axis]
    if n % BLOCK:
        raise ValueError("blocked axis must be a multiple of 32")
    vm = np.moveaxis(v, axis, -1)
    blocks = vm.reshape(vm.shape[:-1] + (n // BLOCK, BLOCK))
    scale = np.ldexp(1.0, block_exponent(np.abs(blocks).max(axis=-1)))[..., None]
    out = e4m3_round(blocks / scale) * scale
    return np.moveaxis(out.reshape(vm.shape), -1, axis)


def fake_quant_rows_from(v: np.ndarray) -> np.ndarray:
    """Column-wise (along axis 0) MXFP8 of a block of rows whose count need not be a multiple
    of 32: the rows are padded with zeros to the next multiple of 32 (zeros do not change a
    block's amax), quantised in 32-row blocks starting at the first row, and cut back."""
    v = np.asarray(v, dtype=np.float64)
    m = v.shape[0]
    mp = -(-m // BLOCK) * BLOCK
    if mp == 0:
        return v.copy()
    pad = np.zeros((mp,) + v.shape[1:], dtype=np.float64)
    pad[:m] = v
    return fake_quant(pad, 0)[:m]


def quantize_colwise_groups(v: np.ndarray, offsets) -> tuple:
    """Column-wise (along axis 0) MXFP8 of row groups of any size: group g is rows
    [offsets[g], offsets[g+1]); its blocks of 32 rows start at the group's first row (the last
    one padded with zeros, which do not change a block's amax), as for the per-expert token
    groups of a GroupedLinear ([TE-MoE] Challenge 1) quantised for the weight gradients.

    Returns (codes uint8 [M, N], scale bytes uint8 [N, nb]) with the scale of column c and
    block i of group g at [c, offsets[g] // 32 + g + i], nb = 4 * ceil((ceil(M/32) + G) / 4),
    and 0 in the entries no block owns (the layout of the library's grouped quantiser)."""
    v = np.asarray(v, dtype=np.float64)
    M, N = v.shape
    G = len(offsets) - 1
    nb = 4 * ((-(-M // BLOCK) + G + 3) // 4)
    codes = np.zeros((M, N), dtype=np.uint8)
    scales = np.zeros((N, nb), dtype=np.uint8)
    for g in range(G):
        a, b = int(offsets[g]), int(offsets[g + 1])
        m = b - a
        if m <= 0:
            continue
        mp = -(-m // BLOCK) * BLOCK
        pad = np.zeros((mp, N))
        pad[:m] = v[a:b]
        c, sb = quantize_blocks(pad, axis=0)          # sb [mp / 32, N]
        codes[a:b] = c[:m]
        base = a // BLOCK + g
        scales[:, base:base + mp // BLOCK] = sb.T
    return codes, scales
