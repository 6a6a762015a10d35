// NVFP4 device helpers shared by the quantiser / amax kernels (nvfp4.cu) and the FP4 grouped
// GEMM (gemm_fp4.cu).
//
// [NV-blog] section "fused MXFP8 and NVFP4 quantisation": for NVFP4 the fused kernels emit a
// BF16 output plus a per-tensor amax (forward) and the amax of the Hadamard-rotated transposed
// output (backward), so that the quantiser needs no extra pass for them. The format is the
// published NVFP4 one: E2M1 elements, one unsigned E4M3 scale per 16 values along the
// reduction dimension, one fp32 encode scale per tensor. Every scaling step is one IEEE fp32
// operation, round to nearest even, in this order:
//   S   = min(2688 / amax, FLT_MAX)           (2688 = 6 * 448; amax == 0 -> FLT_MAX)
//   s_b = E4M3_sat(fp32(amax_b / 6) * S)
//   q   = E2M1_sat(x * fp32(S / s_b))          (factor 0 when s_b == 0)
// and a GEMM of two NVFP4 operands multiplies its fp32 accumulator by 1 / (S_a * S_b).
// Scales sit in the MMA slab layout of sf_mma_offset with the k index counting 16-element
// blocks: one 512-byte slab per 128 rows x 64 elements, exactly what one
// tcgen05.mma.kind::mxf4nvf4 (scale_vec::4X, K = 64) consumes per 128 rows.
//
// Random Hadamard transform (RHT) of the weight-gradient operands: y = (1/4) H16 diag(d) x over
// 16 consecutive token rows, H16 the Sylvester Hadamard matrix and d a +-1 vector given as a
// 16-bit mask (bit j set: d_j = -1). Computed as four butterfly stages (pair distance 1, 2, 4,
// 8; the lower index takes a + b, the upper a - b) and a final exact * 0.25; the register and
// the warp-shuffle forms below perform the same fp32 operations on the same operands, so they
// give identical results.
#pragma once

#include <cfloat>

#include "common.cuh"

namespace moe {

constexpr float kNvfp4ScaleNum = 2688.0f;  // 6 (largest E2M1) * 448 (largest E4M3)

MOE_DEVICE float nvfp4_encode_scale(float amax) {
  return fminf(__fdiv_rn(kNvfp4ScaleNum, amax), FLT_MAX);
}

// Value of an E4M3 byte of a non-negative scale (the sign bit is 0), exact.
MOE_DEVICE float e4m3_pos_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  return e == 0 ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Eight fp32 -> eight E2M1 codes, round to nearest even, saturating to +-6; v[0] lands in the
// lowest nibble (element order of a packed FP4 operand).
MOE_DEVICE uint32_t cvt_e2m1x8(const float* v) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// ----------------------------------------------------------------- packed fp32 pairs
// Two fp32 values in one 64-bit register; add / sub / mul of pairs are two independent IEEE
// fp32 operations (round to nearest even), so they give exactly the scalar results.
MOE_DEVICE uint64_t pack_f32x2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
MOE_DEVICE float f32x2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
MOE_DEVICE float f32x2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
MOE_DEVICE uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
MOE_DEVICE uint64_t sub_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
MOE_DEVICE uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// fp32(m / 6) for m >= 0, IEEE round to nearest even, without the division routine for the
// usual range: the product with c = RN(1/6) corrected by one exact FMA residual,
// q = RN(q0 + RN(m - 6 q0) c) (Markstein's correction step for division by a constant). It
// equals the IEEE quotient for m = 0 and every m in [2^-125, FLT_MAX] (checked exhaustively
// against IEEE division over all such fp32 values); below 2^-125 (subnormal quotients), and for
// inf and NaN, the IEEE division itself is taken.
MOE_DEVICE float nvfp4_div6(float m) {
  constexpr float kSixth = 0x1.555556p-3f;  // RN(1/6)
  if ((m < 0x1p-125f && m != 0.0f) || !(m <= FLT_MAX)) return __fdiv_rn(m, 6.0f);
  const float q0 = __fmul_rn(m, kSixth);
  return __fmaf_rn(__fmaf_rn(-q0, 6.0f, m), kSixth, q0);
}

// The encoding factors fp32(S / s_b) of one tensor for every E4M3 scale byte b < 127 (0 for
// b = 0: the block is all zeros), so that a block's factor is a table read instead of a
// division, with the same IEEE result. Filled by `nthreads` threads; the caller synchronises.
MOE_DEVICE void nvfp4_fill_enc_table(float* tab, float S, int tid, int nthreads) {
  for (int b = tid; b < 128; b += nthreads) {
    const float v = b < 127 ? e4m3_pos_value((uint32_t)b) : 0.f;
    tab[b] = v > 0.f ? __fdiv_rn(S, v) : 0.f;
  }
}

// One 16-value block of a row, given as 8 bf16 pairs: its codes in q[0..1], its scale byte
// returned (enc_tab: the tensor's factor table).
MOE_DEVICE uint32_t nvfp4_quant16_bf16(const uint32_t (&bw)[8], float S, const float* enc_tab,
                                       uint32_t (&q)[2]) {
  float m = 0.f;
  uint64_t x[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float lo = bf16_lo(bw[i]), hi = bf16_hi(bw[i]);
    m = fmaxf(m, fmaxf(fabsf(lo), fabsf(hi)));
    x[i] = pack_f32x2(lo, hi);
  }
  const uint32_t sb = cvt_e4m3x2(__fmul_rn(nvfp4_div6(m), S), 0.f) & 0xFFu;
  const float e = enc_tab[sb];
  const uint64_t e2 = pack_f32x2(e, e);
  float w[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint64_t p = mul_f32x2(x[i], e2);
    w[2 * i] = f32x2_lo(p);
    w[2 * i + 1] = f32x2_hi(p);
  }
  q[0] = cvt_e2m1x8(w);
  q[1] = cvt_e2m1x8(w + 8);
  return sb;
}

// RHT of two columns at once: x[i] = (column a, column b) of row i of the block; the same
// fp32 operations as rht16_regs on each column.
MOE_DEVICE void rht16_pair(uint64_t (&x)[16], uint32_t mask) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if ((mask >> i) & 1u) x[i] ^= 0x8000000080000000ull;
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & m) continue;
      const uint64_t a = x[i], b = x[i | m];
      x[i] = add_f32x2(a, b);
      x[i | m] = sub_f32x2(a, b);
    }
  }
  const uint64_t quarter = pack_f32x2(0.25f, 0.25f);
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = mul_f32x2(x[i], quarter);
}

// Two 16-value column blocks held as pairs (x[i] = (a_i, b_i)): codes of column a in qa, of
// column b in qb; returns the scale bytes (a in bits 0-7, b in bits 8-15).
MOE_DEVICE uint32_t nvfp4_quant16_pair(const uint64_t (&x)[16], float S, const float* enc_tab,
                                       uint32_t (&qa)[2], uint32_t (&qb)[2]) {
  float ma = 0.f, mb = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    ma = fmaxf(ma, fabsf(f32x2_lo(x[i])));
    mb = fmaxf(mb, fabsf(f32x2_hi(x[i])));
  }
  const uint32_t sa = cvt_e4m3x2(__fmul_rn(nvfp4_div6(ma), S), 0.f) & 0xFFu;
  const uint32_t sb = cvt_e4m3x2(__fmul_rn(nvfp4_div6(mb), S), 0.f) & 0xFFu;
  const uint64_t e2 = pack_f32x2(enc_tab[sa], enc_tab[sb]);
  float wa[16], wb[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint64_t p = mul_f32x2(x[i], e2);
    wa[i] = f32x2_lo(p);
    wb[i] = f32x2_hi(p);
  }
  qa[0] = cvt_e2m1x8(wa);
  qa[1] = cvt_e2m1x8(wa + 8);
  qb[0] = cvt_e2m1x8(wb);
  qb[1] = cvt_e2m1x8(wb + 8);
  return sa | (sb << 8);
}

// RHT of 16 values held by one thread (index = row within the block).
MOE_DEVICE void rht16_regs(float (&v)[16], uint32_t mask) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if ((mask >> i) & 1u) v[i] = -v[i];
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & m) continue;
      const float a = v[i], b = v[i | m];
      v[i] = a + b;
      v[i | m] = a - b;
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] *= 0.25f;
}

// RHT across the 16 lanes of a half-warp: lane l holds row (l & 15) of the block; returns the
// rotated value of that row. All 32 lanes must call it.
MOE_DEVICE float rht16_lanes(float x, uint32_t mask, int lane) {
  float v = ((mask >> (lane & 15)) & 1u) ? -x : x;
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) {
    const float o = __shfl_xor_sync(0xFFFFFFFFu, v, m);
    v = (lane & m) ? o - v : v + o;
  }
  return v * 0.25f;
}

// Running max of non-negative floats, merged into a global slot with one atomic per warp.
MOE_DEVICE void amax_flush_warp(float m, float* slot) {
  const uint32_t w = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m));
  if ((threadIdx.x & 31) == 0 && w != 0u) atomicMax(reinterpret_cast<unsigned int*>(slot), w);
}

}  // namespace moe
