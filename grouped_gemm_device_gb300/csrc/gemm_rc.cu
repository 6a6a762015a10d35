// FC2 dgrad with the FC1 output recomputed instead of saved (activation recomputation, listed
// among the ongoing kernel optimisations in [NV-blog] "What's next"): the forward keeps no Z,
// and this kernel rebuilds each tile's Z next to dA_s.
//
// Per 128-row x 128-column tile of dA_s (columns over F) two GEMMs with the same reduction
// over H share one k-loop:
//   dA_s[rows, f0..f0+127]       = dY_perm[rows] . W2_e[f0..f0+127]^T       (128 x 128)
//   Z[rows, 2 f0 .. 2 f0 + 255]  = X_perm[rows]  . W1p_e[2 f0 .. 2 f0+255]^T (128 x 256)
// (the packed W1 rows 2 f0 .. 2 f0 + 255 are exactly the gate and linear columns of dA_s
// columns f0 .. f0 + 127, because the interleave divides 128). For sReLU (not gated, N1 = F)
// the Z tile is Z[rows, f0 .. f0 + 127] (128 x 128) and the epilogue is
// dZ = p dA_s 2 relu(Z), d_prob += dA_s relu(Z)^2. Both accumulate in TMEM (columns 0-127
// and from 128); the epilogue reads dA_s and the fp32 Z from TMEM and writes dZ (bf16,
// packed order) and the per-row d_prob partial of the tile.
//
// CTA = 10 warps: warp 0 TMA, warp 1 TMEM owner + MMA issuer, warps 2-9 epilogue (two per
// TMEM lane quadrant, 64 dA columns each). A stage holds the four k-blocks (dY, W2, X, W1p:
// 80 KB); two stages. One accumulator pair: the next tile's MMAs start when the epilogue has
// read this one. Every wait is bounded (4 s) and raises the device error word.
#include "gemm_common.cuh"

namespace moe {

namespace {

constexpr int BM = 128;
constexpr int BNA = 128;  // dA_s columns per tile
constexpr int BNZ = 256;  // Z columns per tile (gate + linear)
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int STAGES = 2;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kMaxE = 256;

constexpr int A1_BYTES = BM * BK * 2;   // dY
constexpr int B1_BYTES = BNA * BK * 2;  // W2 rows
constexpr int A2_BYTES = BM * BK * 2;   // X
constexpr int B2_BYTES = BNZ * BK * 2;  // W1p rows (gated: 256; sReLU uses the first 128)
constexpr int STAGE_BYTES = A1_BYTES + B1_BYTES + A2_BYTES + B2_BYTES;
constexpr int DATA = STAGES * STAGE_BYTES;
constexpr int SMEM_TOTAL = DATA + 4096 + 1024;
constexpr int kZCol = BNA;  // first TMEM column of the Z accumulator

struct RcArgs {
  CUtensorMap tmDy;  // dY_perm [R_cap, H], box {64, 128}
  CUtensorMap tmW2;  // W2 [E][F][H], box {64, 128, 1}
  CUtensorMap tmX;   // X_perm [R_cap, H], box {64, 128}
  CUtensorMap tmW1;  // W1p [E][N1][H], box {64, 256, 1}
  const int32_t* offsets;
  int E, R_cap, H, F, N1, ilv;
  const float* row_prob;
  uint16_t* dz;  // [R_cap, N1]
  float* dprob_part;
  int nparts;
  int wide;
  ActDev act;
  int* err;
};

struct Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull;
  uint64_t tempty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int off[kMaxE + 1];
  int prefix[kMaxE + 1];
};

struct Tile {
  int e, m0, n0, row_end;
};

MOE_DEVICE void decode(int tile, const RcArgs& p, const Ctrl& c, int NT, Tile& t) {
  int lo = 0, hi = p.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (c.prefix[mid] <= tile) lo = mid; else hi = mid;
  }
  const int local = tile - c.prefix[lo];
  const int mt = (c.off[lo + 1] - c.off[lo] + BM - 1) / BM;
  t.e = lo;
  t.m0 = c.off[lo] + (local % mt) * BM;
  t.n0 = (local / mt) * BNA;
  t.row_end = c.off[lo + 1];
}

MOE_DEVICE void st16(uint16_t* dst, const uint32_t (&w)[8], bool wide) {
  if (wide) {
    st_global_v8(dst, w);
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
    d[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

template <int KIND>
MOE_DEVICE float dglu16(const ActDev& a, float prob, const uint32_t (&da)[16],
                        const uint32_t (&g)[16], const uint32_t (&l)[16], uint32_t (&dgw)[8],
                        uint32_t (&dlw)[8]) {
  float dp = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    // dA_s and Z come from TMEM in fp32
    const float d0 = __uint_as_float(da[2 * i]), d1 = __uint_as_float(da[2 * i + 1]);
    float dg0, dl0, dg1, dl1;
    const float a0 = act_bwd_k<KIND>(a, __uint_as_float(g[2 * i]), __uint_as_float(l[2 * i]),
                                     prob * d0, dg0, dl0);
    const float a1 = act_bwd_k<KIND>(a, __uint_as_float(g[2 * i + 1]),
                                     __uint_as_float(l[2 * i + 1]), prob * d1, dg1, dl1);
    dp += d0 * a0 + d1 * a1;
    dgw[i] = pack_bf16x2(dg0, dg1);
    dlw[i] = pack_bf16x2(dl0, dl1);
  }
  return dp;
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    fc2_dgrad_recompute_kernel(const __grid_constant__ RcArgs p) {
  MOE_GRIDDEP_ENTRY();
  constexpr bool kGated = KIND != MOE_ACT_SRELU;
  constexpr int ZN = kGated ? BNZ : BNA;                        // Z columns per tile
  constexpr int kStageTx = STAGE_BYTES - (BNZ - ZN) * BK * 2;   // bytes a stage receives
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  Ctrl& c = *reinterpret_cast<Ctrl*>(smem + DATA);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &c.abort;
  const int NT = (p.F + BNA - 1) / BNA;
  const int nkb = (p.H + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], 1);
    }
    mbar_init(&c.tfull, 1);
    mbar_init(&c.tempty, kEpiWarps);
    mbar_init(&c.drain, 1);
    fence_mbar_init();
    c.abort = 0;
    bool ok = p.E >= 1 && p.E <= kMaxE;
    int prev = 0;
    for (int e = 0; ok && e <= p.E; ++e) {
      const int o = p.offsets[e];
      if (o < prev || o > p.R_cap || (e == 0 && o != 0)) ok = false;
      c.off[e] = o;
      prev = o;
    }
    int total = 0;
    if (ok) {
      for (int e = 0; e < p.E; ++e) {
        c.prefix[e] = total;
        total += ((c.off[e + 1] - c.off[e] + BM - 1) / BM) * NT;
      }
      c.prefix[p.E] = total;
    } else {
      set_error(p.err, MOE_DEVERR_CAPACITY);
    }
    c.total_tiles = total;
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmDy);
    tma_prefetch_desc(&p.tmW2);
    tma_prefetch_desc(&p.tmX);
    tma_prefetch_desc(&p.tmW1);
  }
  if (warp == 1) {
    tmem_alloc(&c.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = c.tmem_base;
  const int total = c.total_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int armed[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) armed[s] = -1;
      for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x) {
        Tile t;
        decode(tile, p, c, NT, t);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&c.empty[stage], phase ^ 1, abort, p.err)) break;
          uint8_t* s0 = smem + stage * STAGE_BYTES;
          uint64_t* bar = &c.full[stage];
          mbar_arrive_expect_tx(bar, kStageTx);
#pragma unroll
          for (int s = 0; s < STAGES; ++s)
            if (s == stage) armed[s] = (int)phase;
          const int k0 = kb * BK;
          tma_load_2d(s0, &p.tmDy, bar, k0, t.m0);
          tma_load_3d(s0 + A1_BYTES, &p.tmW2, bar, k0, t.n0, t.e);
          tma_load_2d(s0 + A1_BYTES + B1_BYTES, &p.tmX, bar, k0, t.m0);
          tma_load_3d(s0 + A1_BYTES + B1_BYTES + A2_BYTES, &p.tmW1, bar, k0,
                      kGated ? 2 * t.n0 : t.n0, t.e);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
#pragma unroll
      for (int s = 0; s < STAGES; ++s) {
        if (armed[s] >= 0) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(smem_u32(&c.full[s]), (uint32_t)armed[s]) &&
                 globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDA = idesc_bf16(BM, BNA, false, false);
      constexpr uint32_t IDZ = idesc_bf16(BM, ZN, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int acc_i = 0;
      bool issued_any = false;
      for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x) {
        if (!mbar_wait(&c.tempty, (acc_i & 1) ^ 1, abort, p.err)) break;
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&c.full[stage], phase, abort, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t s0 = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sB1 = s0 + A1_BYTES, sA2 = sB1 + B1_BYTES, sB2 = sA2 + A2_BYTES;
          for (int ks = 0; ks < BK / UMMA_K; ++ks) {
            const uint32_t koff = ks * UMMA_K * 2;  // K-major: 32 bytes along the swizzled row
            const uint32_t acc = (kb | ks) != 0 ? 1u : 0u;
            mma_bf16_ss(tmem_base, smem_desc_sw128(s0 + koff, 16, 1024),
                        smem_desc_sw128(sB1 + koff, 16, 1024), IDA, acc);
            mma_bf16_ss(tmem_base + kZCol, smem_desc_sw128(sA2 + koff, 16, 1024),
                        smem_desc_sw128(sB2 + koff, 16, 1024), IDZ, acc);
          }
          issued_any = true;
          mma_commit(&c.empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(&c.tfull);
        ++acc_i;
      }
      if (issued_any) {
        mma_commit(&c.drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&c.drain), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps 2..9
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;  // dA_s columns [64 * half, 64 * half + 64) of the tile
    const int ilv = p.ilv;
    int acc_i = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      // every give-up decision is warp-uniform (full-warp TMEM loads and __syncwarp)
      if (__shfl_sync(0xFFFFFFFFu, *abort, 0)) break;
      Tile t;
      decode(tile, p, c, NT, t);
      const int row = t.m0 + q * 32 + lane;
      const bool row_ok = row < t.row_end;
      const float prob = row_ok ? p.row_prob[row] : 0.f;
      const bool got = mbar_wait(&c.tfull, acc_i & 1, abort, p.err);
      if (!__all_sync(0xFFFFFFFFu, got)) break;
      tc_fence_after();
      const uint32_t tl = tmem_base + ((uint32_t)(q * 32) << 16);
      uint16_t* dzrow = p.dz + (int64_t)row * p.N1 + (kGated ? 2 * t.n0 : t.n0);
      float dp = 0.f;
#pragma unroll 1
      for (int cc = half * 64; cc < half * 64 + 64; cc += 16) {
        if (t.n0 + cc >= p.F) break;
        if constexpr (!kGated) {
          uint32_t da[16], z[16], dzw[8];
          tmem_ld_32x32b_x16(tl + cc, da);
          tmem_ld_32x32b_x16(tl + kZCol + cc, z);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float d0 = __uint_as_float(da[2 * i]), d1 = __uint_as_float(da[2 * i + 1]);
            const float r0 = fmaxf(__uint_as_float(z[2 * i]), 0.f);
            const float r1 = fmaxf(__uint_as_float(z[2 * i + 1]), 0.f);
            dp += d0 * r0 * r0 + d1 * r1 * r1;
            dzw[i] = pack_bf16x2(prob * d0 * 2.f * r0, prob * d1 * 2.f * r1);
          }
          if (row_ok) st16(dzrow + cc, dzw, p.wide);
          continue;
        }
        const int gc = (cc / ilv) * 2 * ilv + (cc % ilv);  // within the tile's 256 Z columns
        uint32_t da[16], g[16], l[16];
        tmem_ld_32x32b_x16(tl + cc, da);
        tmem_ld_32x32b_x16(tl + kZCol + gc, g);
        tmem_ld_32x32b_x16(tl + kZCol + gc + ilv, l);
        tmem_ld_wait();
        uint32_t dgw[8], dlw[8];
        dp += dglu16<KIND>(p.act, prob, da, g, l, dgw, dlw);
        if (row_ok) {
          st16(dzrow + gc, dgw, p.wide);
          st16(dzrow + gc + ilv, dlw, p.wide);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.tempty);
      ++acc_i;
      if (row_ok) p.dprob_part[(int64_t)row * p.nparts + (t.n0 / BNA) * 2 + half] = dp;
    }
  }

  griddep_launch_dependents();  // this CTA's tiles are done
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

template <int KIND>
cudaError_t launch_kind(const RcArgs& a, int grid, cudaStream_t s) {
  auto kern = fc2_dgrad_recompute_kernel<KIND>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), SMEM_TOTAL);
  if (e != cudaSuccess) return e;
  launch_kernel(kern, grid, kThreads, SMEM_TOTAL, s, nullptr, 0, a);
  count_launch(s, MOE_K_GEMM_FC2_DGRAD);
  return cudaGetLastError();
}

}  // namespace

int dprob_parts_recompute(int F) { return 2 * ((F + BNA - 1) / BNA); }

cudaError_t launch_fc2_dgrad_recompute(const GemmProblem& p, cudaStream_t s) {
  if (p.gated && p.ilv != 32 && p.ilv != 64 && p.ilv != 128) return cudaErrorInvalidValue;
  RcArgs a;
  memset(&a, 0, sizeof(a));
  const uint64_t R = (uint64_t)p.R_cap;
  bool ok = true;
  ok &= tmap_2d(&a.tmDy, p.dy_perm, p.H, R, 64, BM);
  ok &= tmap_3d(&a.tmW2, p.w2, p.H, p.F, p.E, 64, BNA);
  ok &= tmap_2d(&a.tmX, p.x_perm, p.H, R, 64, BM);
  ok &= tmap_3d(&a.tmW1, p.w1p, p.H, p.N1, p.E, 64, p.gated ? BNZ : BNA);
  if (!ok) return cudaErrorInvalidValue;
  a.offsets = p.offsets;
  a.E = p.E;
  a.R_cap = (int)p.R_cap;
  a.H = p.H;
  a.F = p.F;
  a.N1 = p.N1;
  a.ilv = p.ilv;
  a.row_prob = p.row_prob;
  a.dz = static_cast<uint16_t*>(p.out);
  a.dprob_part = p.dprob_part;
  a.nparts = dprob_parts_recompute(p.F);
  a.wide = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0 && p.N1 % 16 == 0;
  a.act = p.act;
  a.err = p.err;
  const int grid = p.num_ctas;
  switch (p.act.kind) {
    case MOE_ACT_SWIGLU: return launch_kind<MOE_ACT_SWIGLU>(a, grid, s);
    case MOE_ACT_CLAMPED_SWIGLU: return launch_kind<MOE_ACT_CLAMPED_SWIGLU>(a, grid, s);
    case MOE_ACT_GEGLU: return launch_kind<MOE_ACT_GEGLU>(a, grid, s);
    case MOE_ACT_SRELU: return launch_kind<MOE_ACT_SRELU>(a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
