// Helpers shared by the grouped GEMM kernels (BF16, MXFP8, NVFP4): fp32 activation math of the
// GLU epilogues, 32-wide bf16 load/store, and host-side TMA tensor-map construction.
#pragma once

#include <mutex>

#include "kernels.cuh"

namespace moe {

// ------------------------------------------------------------------ activations (fp32)
MOE_DEVICE float phi_cdf(float g) { return 0.5f * (1.0f + erff(g * 0.70710678118654752f)); }

template <int KIND>
MOE_DEVICE float act_fwd_k(const ActDev& a, float g, float l) {
  if (KIND == MOE_ACT_CLAMPED_SWIGLU) {
    const float gc = fminf(g, a.gate_max);
    const float lc = fminf(fmaxf(l, a.lin_lo), a.lin_hi);
    return (lc + a.lin_offset) * gc * sigmoidf_fast(a.beta * gc);
  }
  if (KIND == MOE_ACT_GEGLU) return l * g * phi_cdf(g);
  return l * g * sigmoidf_fast(a.beta * g);  // SwiGLU
}

// returns a (unscaled) and writes d_gate, d_lin for the upstream gradient dA
template <int KIND>
MOE_DEVICE float act_bwd_k(const ActDev& a, float g, float l, float dA, float& dg, float& dl) {
  if (KIND == MOE_ACT_CLAMPED_SWIGLU) {
    const float gc = fminf(g, a.gate_max);
    const float lc = fminf(fmaxf(l, a.lin_lo), a.lin_hi);
    const float s = sigmoidf_fast(a.beta * gc);
    const float sw = gc * s;
    dg = (g <= a.gate_max) ? dA * (lc + a.lin_offset) * s * (1.0f + a.beta * gc * (1.0f - s))
                           : 0.0f;
    dl = (l >= a.lin_lo && l <= a.lin_hi) ? dA * sw : 0.0f;
    return (lc + a.lin_offset) * sw;
  }
  if (KIND == MOE_ACT_GEGLU) {
    const float P = phi_cdf(g);
    const float pdf = 0.39894228040143268f * __expf(-0.5f * g * g);
    dg = dA * l * (P + g * pdf);
    dl = dA * g * P;
    return l * g * P;
  }
  const float s = sigmoidf_fast(a.beta * g);
  dg = dA * l * s * (1.0f + a.beta * g * (1.0f - s));
  dl = dA * g * s;
  return l * g * s;
}

MOE_DEVICE float act_fwd(const ActDev& a, float g, float l) {
  if (a.kind == MOE_ACT_CLAMPED_SWIGLU) return act_fwd_k<MOE_ACT_CLAMPED_SWIGLU>(a, g, l);
  if (a.kind == MOE_ACT_GEGLU) return act_fwd_k<MOE_ACT_GEGLU>(a, g, l);
  return act_fwd_k<MOE_ACT_SWIGLU>(a, g, l);
}

MOE_DEVICE float act_bwd(const ActDev& a, float g, float l, float dA, float& dg, float& dl) {
  if (a.kind == MOE_ACT_CLAMPED_SWIGLU) return act_bwd_k<MOE_ACT_CLAMPED_SWIGLU>(a, g, l, dA, dg, dl);
  if (a.kind == MOE_ACT_GEGLU) return act_bwd_k<MOE_ACT_GEGLU>(a, g, l, dA, dg, dl);
  return act_bwd_k<MOE_ACT_SWIGLU>(a, g, l, dA, dg, dl);
}

// 32-wide forms with the activation chosen once per block (keeps the unrolled code of one
// activation contiguous instead of interleaving all three per element).
// v[i] = prob * act(g[i], l[i])
MOE_DEVICE void glu_fwd32(const ActDev& a, float prob, const float* g, const float* l,
                          float (&v)[32]) {
  if (a.kind == MOE_ACT_CLAMPED_SWIGLU) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = prob * act_fwd_k<MOE_ACT_CLAMPED_SWIGLU>(a, g[i], l[i]);
  } else if (a.kind == MOE_ACT_GEGLU) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = prob * act_fwd_k<MOE_ACT_GEGLU>(a, g[i], l[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = prob * act_fwd_k<MOE_ACT_SWIGLU>(a, g[i], l[i]);
  }
}

// In place: g <- d_gate, l <- d_linear for dA = prob * das; returns sum_i das[i] * a[i].
template <int KIND>
MOE_DEVICE float glu_bwd32_k(const ActDev& a, float prob, const float (&das)[32],
                             float (&g)[32], float (&l)[32]) {
  float dp = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float dg, dl;
    const float av = act_bwd_k<KIND>(a, g[i], l[i], prob * das[i], dg, dl);
    dp += das[i] * av;
    g[i] = dg;
    l[i] = dl;
  }
  return dp;
}
MOE_DEVICE float glu_bwd32(const ActDev& a, float prob, const float (&das)[32], float (&g)[32],
                           float (&l)[32]) {
  if (a.kind == MOE_ACT_CLAMPED_SWIGLU)
    return glu_bwd32_k<MOE_ACT_CLAMPED_SWIGLU>(a, prob, das, g, l);
  if (a.kind == MOE_ACT_GEGLU) return glu_bwd32_k<MOE_ACT_GEGLU>(a, prob, das, g, l);
  return glu_bwd32_k<MOE_ACT_SWIGLU>(a, prob, das, g, l);
}

// 16-wide form of glu_bwd32 (packed bf16 inputs): g/l words hold the saved gate and linear
// values, das the upstream gradient; writes the packed bf16 d_gate / d_linear words and
// returns sum_i das[i] * a[i].
template <int KIND>
MOE_DEVICE float glu_bwd16_k(const ActDev& a, float prob, const uint32_t (&das)[16],
                             const uint32_t (&gw)[8], const uint32_t (&lw)[8], uint32_t (&dgw)[8],
                             uint32_t (&dlw)[8]) {
  float dp = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float dg0, dl0, dg1, dl1;
    const float d0 = __uint_as_float(das[2 * i]), d1 = __uint_as_float(das[2 * i + 1]);
    const float a0 = act_bwd_k<KIND>(a, bf16_lo(gw[i]), bf16_lo(lw[i]), prob * d0, dg0, dl0);
    const float a1 = act_bwd_k<KIND>(a, bf16_hi(gw[i]), bf16_hi(lw[i]), prob * d1, dg1, dl1);
    dp += d0 * a0 + d1 * a1;
    dgw[i] = pack_bf16x2(dg0, dg1);
    dlw[i] = pack_bf16x2(dl0, dl1);
  }
  return dp;
}
MOE_DEVICE float glu_bwd16(const ActDev& a, float prob, const uint32_t (&das)[16],
                           const uint32_t (&gw)[8], const uint32_t (&lw)[8], uint32_t (&dgw)[8],
                           uint32_t (&dlw)[8]) {
  if (a.kind == MOE_ACT_CLAMPED_SWIGLU)
    return glu_bwd16_k<MOE_ACT_CLAMPED_SWIGLU>(a, prob, das, gw, lw, dgw, dlw);
  if (a.kind == MOE_ACT_GEGLU) return glu_bwd16_k<MOE_ACT_GEGLU>(a, prob, das, gw, lw, dgw, dlw);
  return glu_bwd16_k<MOE_ACT_SWIGLU>(a, prob, das, gw, lw, dgw, dlw);
}
// Column sums over the warp's 32 rows: v[i] of every lane in, the sum of v[lane] out (a
// butterfly that halves the values each lane keeps: 31 shuffles for 32 columns). v is
// overwritten.
MOE_DEVICE float warp_colsum32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool hi = lane & w;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = hi ? v[i] : v[i + w];
      const float keep = hi ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, w);
    }
  }
  return v[0];
}

// Column sums of a warp's 32 rows (lane = row) for 16 columns: lanes l and l + 16 both
// return the sum of column l % 16 (the two half-warps are added first, then the same
// transpose-reduce as warp_colsum32 over the 16 columns).
MOE_DEVICE float warp_colsum16(float (&v)[16], int lane) {
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] += __shfl_xor_sync(0xFFFFFFFFu, v[i], 16);
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
    const bool hi = lane & w;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = hi ? v[i] : v[i + w];
      const float keep = hi ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, w);
    }
  }
  return v[0];
}

// 32 bytes at a 32-byte aligned global address, not allocated in L1.
MOE_DEVICE void ld_v8_noalloc(const void* src, uint32_t (&w)[8]) {
  asm volatile("ld.global.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                 "=r"(w[6]), "=r"(w[7])
               : "l"(src));
}

MOE_DEVICE void store_bf16x32(void* dst, const float (&v)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    d[i] = make_uint4(pack_bf16x2(v[8 * i + 0], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                      pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
}
// 32 fp32 -> 64 bytes of bf16 at a 32-byte aligned address: two 256-bit stores.
MOE_DEVICE void store_bf16x32_v8(void* dst, const float* v) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
  st_global_v8(dst, w);
  st_global_v8(static_cast<uint8_t*>(dst) + 32, w + 8);
}
// Either form: wide = dst is 32-byte aligned.
MOE_DEVICE void store_bf16x32w(void* dst, const float (&v)[32], bool wide) {
  if (wide) store_bf16x32_v8(dst, v);
  else store_bf16x32(dst, v);
}
MOE_DEVICE void load_bf16x32(const void* src, float (&v)[32]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 w = s[i];
    v[8 * i + 0] = bf16_lo(w.x); v[8 * i + 1] = bf16_hi(w.x);
    v[8 * i + 2] = bf16_lo(w.y); v[8 * i + 3] = bf16_hi(w.y);
    v[8 * i + 4] = bf16_lo(w.z); v[8 * i + 5] = bf16_hi(w.z);
    v[8 * i + 6] = bf16_lo(w.w); v[8 * i + 7] = bf16_hi(w.w);
  }
}
// 32 bf16 at a 32-byte aligned address in two 256-bit loads, unpacked to fp32.
MOE_DEVICE void load_bf16x32_v8(const void* src, float (&v)[32]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t w[8];
    asm volatile("ld.global.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                   "=r"(w[6]), "=r"(w[7])
                 : "l"(static_cast<const uint8_t*>(src) + 32 * h));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[16 * h + 2 * i] = bf16_lo(w[i]);
      v[16 * h + 2 * i + 1] = bf16_hi(w[i]);
    }
  }
}
MOE_DEVICE void store_zero_bf16x32(void* dst) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] = make_uint4(0, 0, 0, 0);
}


// dGLU: this lane's row of one chunk of saved Z (32 columns of gate and of linear values),
// copied into the warp's 4 KB shared buffer with cp.async. Pieces 0-3 (16 bytes each) come from src0 (gate columns, or the only half when not
// gated), pieces 4-7 from src1 (linear columns). Piece c of row r sits at r*128 +
// ((c ^ (r & 7)) * 16), so 8 rows reading the same piece touch 8 different bank groups.
MOE_DEVICE void zst_issue(uint32_t buf, const uint16_t* src0, const uint16_t* src1, int lane,
                          bool two, bool valid = true) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    if (c >= 4 && !two) break;
    const uint16_t* src = c < 4 ? src0 + 8 * c : src1 + 8 * (c - 4);
    // an invalid row copies nothing and reads no global memory (zero fill)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     buf + lane * 128 + ((c ^ (lane & 7)) * 16)),
                 "l"(valid ? src : src0), "r"(valid ? 16 : 0)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}
MOE_DEVICE void zst_piece(const uint8_t* buf, int c, int lane, uint32_t* w) {
  const uint4 v = *reinterpret_cast<const uint4*>(buf + lane * 128 + ((c ^ (lane & 7)) * 16));
  w[0] = v.x;
  w[1] = v.y;
  w[2] = v.z;
  w[3] = v.w;
}

// ------------------------------------------------------------------ tensor maps (host)
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// bf16 tensor map, 128-byte swizzle. dims/box innermost first; strides in bytes for dims 1..
inline bool make_tmap(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
               const uint64_t* strides, const uint32_t* box, CUtensorMapDataType dt,
               CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void*>(base),
                  reinterpret_cast<const cuuint64_t*>(dims),
                  reinterpret_cast<const cuuint64_t*>(strides),
                  reinterpret_cast<const cuuint32_t*>(box), estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

inline bool tmap_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_in,
             uint32_t box_out) {
  uint64_t dims[2] = {inner, outer};
  uint64_t strides[1] = {inner * 2};
  uint32_t box[2] = {box_in, box_out};
  return make_tmap(m, base, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}
inline bool tmap_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
             uint32_t b0, uint32_t b1) {
  uint64_t dims[3] = {d0, d1, d2};
  uint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  uint32_t box[3] = {b0, b1, 1};
  return make_tmap(m, base, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}


}  // namespace moe
