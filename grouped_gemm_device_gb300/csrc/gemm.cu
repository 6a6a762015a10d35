// Persistent grouped GEMM for sm_103a: TMA -> shared-memory ring -> tcgen05.mma (fp32
// accumulators in tensor memory) -> warp-specialised epilogue, over a device-resident group
// table (the padded per-expert row offsets), so the host never learns the token counts.
//
// [NV-blog] kernel families: (1) GroupGemm + quantise (FC2 fprop, FC1 dgrad, wgrads),
// (2) GroupGemm + activation (+ quantise/transpose) for FC1, (3) GroupGemm + dActivation
// (+ quantise/transpose) for FC2 dgrad; the GLU epilogue relies on the repacked W1 so one
// 256-column tile holds 128 gate and 128 linear columns (GLU-epilogue section, Figure 2);
// the persistent tile loop over device offsets is the host-sync section's design; the
// `num_ctas` cap is the configurable SM margin.
//
// CTA = 10 warps: warp 0 issues TMA loads, warp 1 owns the TMEM allocation and issues the
// MMAs (one thread), warps 2..9 drain the accumulator (warp w reads TMEM lanes 32*(w%4)..
// and one half of the tile's columns).
// Two TMEM accumulators of BN fp32 columns let the epilogue of tile i overlap the mainloop
// of tile i+1. Tiles are 128 x BN; k-blocks are 64 bf16 (one 128-byte swizzle row).
//
// Two tile spaces:
//   row-grouped (fprop, dgrad): each expert's padded row segment is cut into 128-row tiles;
//     K is the same for all experts. Output rows beyond the segment end are not stored.
//   k-grouped (wgrad): every expert has the same M x N output; K is the expert's row segment.
//     A k-block that crosses the segment end issues only the in-segment 16-row MMA steps
//     (segments are 32-row aligned); an expert with no rows gets an all-zero tile.
#include <mutex>

#include "gemm_common.cuh"

namespace moe {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;  // TMA warp, MMA warp, epilogue warps
constexpr int kMaxE = 256;

enum { EPI_STORE = 0, EPI_GLU = 1, EPI_DGLU = 2 };

struct GemmArgs {
  CUtensorMap tmA;
  CUtensorMap tmB;
  const int32_t* offsets;
  int E;
  int R_cap;
  int M;   // k-grouped: output rows per expert
  int N;   // output columns
  int K;   // row-grouped: reduction length
  void* out;
  int64_t ldo;
  int64_t out_estride;
  void* out2;
  int64_t ldo2;
  const float* row_prob;
  const uint16_t* z;
  int64_t ldz;
  float* dprob_part;
  int nparts;
  int gated;
  int ilv;
  int F;
  int wide;  // out and out2 are 32-byte aligned with 16-element strides: 256-bit stores
  // epilogue extras (gated BF16): FC1 bias [E, N1] in logical [gate | linear] order and
  // feature scale [E, F] (fp32, NULL when absent); the dGLU epilogue writes per-32-row column
  // sums of dZ and of p * dA_s * a into ext_part [R_cap / 32, N1 + F]
  const float* fc1_bias;
  const float* fscale;
  float* ext_part;
  int N1;  // FC1 output columns (2F gated)
  ActDev act;
  int* err;
  int stall_loads;   // self-test: the producer issues no loads
  uint64_t wait_ns;  // limit of every barrier wait
};

// PAIR: the CTA holds half of the B tile (the pair's MMA reads both halves).
template <int BN, int STAGES, bool PAIR = false>
struct Smem {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int DATA = STAGES * STAGE_BYTES;
  static constexpr int CTRL = 4096;
  static constexpr int TOTAL = DATA + CTRL + 1024;  // + alignment slack
};

struct Ctrl {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int off[kMaxE + 1];
  int prefix[kMaxE + 1];
};

struct TileInfo {
  int e, m0, n0, kbeg, klen, nkb, row_end;
};

// Tiles are TM rows (128, or 256 for a CTA pair) by BN columns.
template <int BN, bool KG, int TM = BM>
MOE_DEVICE void decode_tile(int tile, const GemmArgs& p, const Ctrl& c, int MT, int NT,
                            TileInfo& t) {
  if (!KG) {
    int lo = 0, hi = p.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (c.prefix[mid] <= tile) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int local = tile - c.prefix[e];
    const int seg = c.off[e + 1] - c.off[e];
    const int mt = (seg + TM - 1) / TM;
    t.e = e;
    t.m0 = c.off[e] + (local % mt) * TM;
    t.n0 = (local / mt) * BN;
    t.kbeg = 0;
    t.klen = p.K;
    t.nkb = p.K / BK;
    t.row_end = c.off[e + 1];
  } else {
    // n fastest: the CTAs of one wave share a few 128-column slices of A (read once from
    // DRAM) and re-read the expert's narrow B (the N side, few tiles) from L2
    const int per = MT * NT;
    const int e = tile / per;
    const int local = tile - e * per;
    t.e = e;
    t.m0 = (local / NT) * TM;
    t.n0 = (local % NT) * BN;
    t.kbeg = c.off[e];
    t.klen = c.off[e + 1] - c.off[e];
    t.nkb = (t.klen + BK - 1) / BK;
    t.row_end = p.M;
  }
}

// dGLU with the epilogue extras for one 16-column step: the feature scale s enters as
// dA = p * s * dA_s and d_prob += dA_s * s * a; the step's column sums over the warp's rows of
// dZ (bias gradient) and of p * dA_s * a (scale gradient) are stored to the row group's
// partials (gate columns at f, linear at F + f, scale at N1 + f).
template <int KIND>
MOE_DEVICE float dglu16_extras(const GemmArgs& p, float prob, const uint32_t (&das)[16],
                               const uint32_t (&gw)[8], const uint32_t (&lw)[8], int e, int f,
                               uint32_t (&dgw)[8], uint32_t (&dlw)[8], float* part, int lane) {
  float v[32], t[32];
  float dp = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float d = __uint_as_float(das[i]);
    const float sc = p.fscale ? p.fscale[(int64_t)e * p.F + f + i] : 1.f;
    const float g = (i & 1) ? bf16_hi(gw[i >> 1]) : bf16_lo(gw[i >> 1]);
    const float l = (i & 1) ? bf16_hi(lw[i >> 1]) : bf16_lo(lw[i >> 1]);
    float dg, dl;
    const float a = act_bwd_k<KIND>(p.act, g, l, prob * sc * d, dg, dl);
    dp += d * sc * a;
    v[i] = dg;
    v[16 + i] = dl;
    t[i] = prob * d * a;
    t[16 + i] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    dgw[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    dlw[i] = pack_bf16x2(v[16 + 2 * i], v[16 + 2 * i + 1]);
  }
  if (part) {
    const float sb = warp_colsum32(v, lane);
    part[lane < 16 ? f + lane : p.F + f + lane - 16] = sb;
    const float ss = warp_colsum32(t, lane);
    if (lane < 16) part[p.N1 + f + lane] = ss;
  }
  return dp;
}
MOE_DEVICE float dglu16_extras_any(const GemmArgs& p, float prob, const uint32_t (&das)[16],
                                   const uint32_t (&gw)[8], const uint32_t (&lw)[8], int e, int f,
                                   uint32_t (&dgw)[8], uint32_t (&dlw)[8], float* part, int lane) {
  if (p.act.kind == MOE_ACT_CLAMPED_SWIGLU)
    return dglu16_extras<MOE_ACT_CLAMPED_SWIGLU>(p, prob, das, gw, lw, e, f, dgw, dlw, part, lane);
  if (p.act.kind == MOE_ACT_GEGLU)
    return dglu16_extras<MOE_ACT_GEGLU>(p, prob, das, gw, lw, e, f, dgw, dlw, part, lane);
  return dglu16_extras<MOE_ACT_SWIGLU>(p, prob, das, gw, lw, e, f, dgw, dlw, part, lane);
}

// dGLU: the saved Z (packed bf16) of dA columns f0 .. f0+15 of one row: the gate columns into
// g and, when gated, the linear columns into l (one 256-bit load each).
MOE_DEVICE void z_load16(const GemmArgs& p, const uint16_t* zrow, int f0, uint32_t (&g)[8],
                         uint32_t (&l)[8]) {
  const int gcol = p.gated ? (f0 / p.ilv) * 2 * p.ilv + (f0 % p.ilv) : f0;
  ld_v8_noalloc(zrow + gcol, g);
  if (p.gated) ld_v8_noalloc(zrow + gcol + p.ilv, l);
}
// 16 bf16 (8 packed words) at dst: one 256-bit store when 32-byte aligned.
MOE_DEVICE void st_bf16x16(void* dst, const uint32_t (&w)[8], bool wide) {
  if (wide) {
    st_global_v8(dst, w);
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
    d[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// EXT: the GLU / dGLU epilogue with the bias and feature-scale extras (a separate
// instantiation, so the plain kernels carry none of its code or registers).
//
// PAIR: the kernel runs as clusters of two CTAs on neighbouring SMs, each pair computing
// 256 x BN tiles with one cta_group::2 MMA per K step: CTA rank r loads rows 128r.. of the
// tile's A and columns (BN/2)r.. of its B, and keeps rows 128r.. of the accumulator in its
// own TMEM. Per K step a CTA moves 2/3 of the bytes a 128 x BN tile needs, for the same MMA
// work per SM. The even-ranked (leader) CTA issues every MMA. Both CTAs' TMA loads of a stage
// complete on the leader's full[s] barrier, which the leader arms with the pair's bytes; the
// follower's epilogue warps free the accumulator on the leader's tempty barrier; the leader's
// MMA commits reach both CTAs' empty / tfull barriers by multicast. Before it exits the
// follower waits until the MMAs have consumed its last loads, the leader until the last
// stages it armed have landed.
template <int BN, int STAGES, bool A_MN, bool B_MN, int EPI, bool KG, bool B3D, bool EXT = false,
          bool PAIR = false>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ GemmArgs p) {
  MOE_GRIDDEP_ENTRY();
  using L = Smem<BN, STAGES, PAIR>;
  constexpr int TM = PAIR ? 2 * BM : BM;    // tile rows
  constexpr int BNH = PAIR ? BN / 2 : BN;   // B columns this CTA loads
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  Ctrl& c = *reinterpret_cast<Ctrl*>(smem + L::DATA);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &c.abort;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int tile0 = PAIR ? (int)cluster_id_x() : (int)blockIdx.x;
  const int tstep = PAIR ? (int)nclusters_x() : (int)gridDim.x;

  const int NT = (p.N + BN - 1) / BN;
  const int MT = KG ? (p.M + TM - 1) / TM : 0;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c.tfull[i], 1);
      mbar_init(&c.tempty[i], PAIR ? 2 * kEpiWarps : kEpiWarps);
    }
    mbar_init(&c.drain, 1);
    fence_mbar_init();
    c.abort = 0;
    // group table: validate, then tile prefix
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
        if (KG) total += MT * NT;
        else total += ((c.off[e + 1] - c.off[e] + TM - 1) / TM) * NT;
      }
      c.prefix[p.E] = total;
    } else {
      set_error(p.err, MOE_DEVERR_CAPACITY);
    }
    c.total_tiles = total;
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA);
    tma_prefetch_desc(&p.tmB);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(&c.tmem_base, 2 * BN);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&c.tmem_base, 2 * BN);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  // both CTAs' barriers are initialised before either signals the other
  if constexpr (PAIR) cluster_sync_all();
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
      // pair: every load completes on the leader's full barrier
      const uint32_t full_leader = PAIR ? mapa_shared(smem_u32(&c.full[0]), 0) : 0u;
      for (int tile = tile0; tile < total && !*abort && !p.stall_loads; tile += tstep) {
        TileInfo t;
        decode_tile<BN, KG, TM>(tile, p, c, MT, NT, t);
        const int am0 = t.m0 + BM * (int)rank;    // this CTA's A rows
        const int bn0 = t.n0 + BNH * (int)rank;   // this CTA's B columns
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!mbar_wait(&c.empty[stage], phase ^ 1, abort, p.err, p.wait_ns)) break;
          uint8_t* sA = smem + stage * L::STAGE_BYTES;
          uint8_t* sB = sA + L::A_BYTES;
          uint64_t* bar = &c.full[stage];
          const uint32_t bar_c = full_leader + stage * (uint32_t)sizeof(uint64_t);
          if (!PAIR) mbar_arrive_expect_tx(bar, L::STAGE_BYTES);
          else if (rank == 0) mbar_arrive_expect_tx(bar, 2 * L::STAGE_BYTES);
#pragma unroll
          for (int s = 0; s < STAGES; ++s)
            if (s == stage) armed[s] = (int)phase;
          const int k0 = t.kbeg + kb * BK;
          auto ld2 = [&](void* dst, const CUtensorMap* m, int x, int y) {
            if constexpr (PAIR) tma_load_2d_pair(dst, m, bar_c, x, y);
            else tma_load_2d(dst, m, bar, x, y);
          };
          auto ld3 = [&](void* dst, const CUtensorMap* m, int x, int y, int z) {
            if constexpr (PAIR) tma_load_3d_pair(dst, m, bar_c, x, y, z);
            else tma_load_3d(dst, m, bar, x, y, z);
          };
          if (!A_MN) {
            ld2(sA, &p.tmA, k0, am0);
          } else {
            ld2(sA, &p.tmA, am0, k0);
            ld2(sA + 64 * 128, &p.tmA, am0 + 64, k0);
          }
          if (!B_MN) {
            if (B3D) ld3(sB, &p.tmB, k0, bn0, t.e);
            else ld2(sB, &p.tmB, k0, bn0);
          } else {
#pragma unroll
            for (int i = 0; i < BNH / 64; ++i) {
              if (B3D) ld3(sB + i * 64 * 128, &p.tmB, bn0 + 64 * i, k0, t.e);
              else ld2(sB + i * 64 * 128, &p.tmB, bn0 + 64 * i, k0);
            }
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // let every load this thread issued land before the CTA can exit: the leader (or a
      // single CTA) waits on the full barriers it armed, which also count a pair follower's
      // bytes; a pair follower waits until the MMAs have consumed its last load of each stage
      // (the consuming commit also arrives in its shared memory)
#pragma unroll
      for (int s = 0; s < STAGES; ++s) {
        if (armed[s] >= 0) {
          const uint32_t bar_s = (PAIR && rank != 0) ? smem_u32(&c.empty[s]) : smem_u32(&c.full[s]);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(bar_s, (uint32_t)armed[s]) &&
                 globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1 && PAIR && rank != 0) {
    // pair follower: no MMAs to issue (the leader issues the pair's)
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16(TM, BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int acc_i = 0;
      bool issued_any = false;
      for (int tile = tile0; tile < total && !*abort; tile += tstep) {
        TileInfo t;
        decode_tile<BN, KG, TM>(tile, p, c, MT, NT, t);
        if (t.nkb == 0) continue;
        const int acc = acc_i & 1;
        const uint32_t acc_phase = (acc_i >> 1) & 1;
        if (!mbar_wait(&c.tempty[acc], acc_phase ^ 1, abort, p.err, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!mbar_wait(&c.full[stage], phase, abort, p.err, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + stage * L::STAGE_BYTES);
          const uint32_t sB = sA + L::A_BYTES;
          int nsub = BK / UMMA_K;
          if (KG) {
            const int rem = t.klen - kb * BK;
            if (rem < BK) nsub = (rem + UMMA_K - 1) / UMMA_K;
          }
          for (int ks = 0; ks < nsub; ++ks) {
            const uint64_t ad = A_MN ? smem_desc_sw128(sA + ks * (UMMA_K * 128), 64 * 128, 1024)
                                     : smem_desc_sw128(sA + ks * (UMMA_K * 2), 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(sB + ks * (UMMA_K * 128), 64 * 128, 1024)
                                     : smem_desc_sw128(sB + ks * (UMMA_K * 2), 16, 1024);
            if constexpr (PAIR) mma_bf16_ss_pair(d_tmem, ad, bd, IDESC, (kb | ks) != 0 ? 1u : 0u);
            else mma_bf16_ss(d_tmem, ad, bd, IDESC, (kb | ks) != 0 ? 1u : 0u);
          }
          issued_any = true;
          if constexpr (PAIR) mma_commit_pair_mc(&c.empty[stage], 0x3);
          else mma_commit(&c.empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if constexpr (PAIR) mma_commit_pair_mc(&c.tfull[acc], 0x3);
        else mma_commit(&c.tfull[acc]);
        ++acc_i;
      }
      // drain: every MMA this thread issued completes before TMEM is released
      if (issued_any) {
        if constexpr (PAIR) mma_commit_pair_mc(&c.drain, 0x1);
        else mma_commit(&c.drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&c.drain), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps 2..9
    // warp w reads TMEM lanes 32*(w%4).. (its lane quadrant) and half (w-2)/4 of the columns
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    int acc_i = 0;
    // the accumulator is freed on the leader's barrier (a pair's MMAs write both CTAs' TMEM)
    const uint32_t tempty_leader = PAIR ? mapa_shared(smem_u32(&c.tempty[0]), 0) : 0u;
    for (int tile = tile0; tile < total; tile += tstep) {
      // every give-up decision is warp-uniform: the epilogue uses full-warp TMEM loads,
      // shuffles and __syncwarp, which all 32 lanes must reach together
      if (__shfl_sync(0xFFFFFFFFu, *abort, 0)) break;
      TileInfo t;
      decode_tile<BN, KG, TM>(tile, p, c, MT, NT, t);
      t.m0 += BM * (int)rank;                    // this CTA's 128 rows of the tile
      const int row = t.m0 + q * 32 + lane;
      const bool row_ok = row < t.row_end;
      const int c0 = half * (BN / 2), c1 = c0 + BN / 2;  // this warp's accumulator columns
      if (t.nkb == 0) {
        // k-grouped tile of an expert with no rows: exact zeros
        if (row_ok) {
          uint16_t* o = static_cast<uint16_t*>(p.out) + (int64_t)t.e * p.out_estride +
                        (int64_t)row * p.ldo;
          for (int cc = c0; cc < c1 && t.n0 + cc < p.N; cc += 32) store_zero_bf16x32(o + t.n0 + cc);
        }
        continue;
      }
      // dGLU: the saved Z of the first two 16-column steps is requested while the MMAs run
      const uint16_t* zrow = p.z + (int64_t)row * p.ldz;
      uint32_t z0g[8], z0l[8], z1g[8], z1l[8], z2g[8], z2l[8];
      if constexpr (EPI == EPI_DGLU) {
        if (row_ok && t.n0 + c0 < p.N) z_load16(p, zrow, t.n0 + c0, z0g, z0l);
        if (row_ok && t.n0 + c0 + 16 < p.N) z_load16(p, zrow, t.n0 + c0 + 16, z1g, z1l);
      }
      const int acc = acc_i & 1;
      const uint32_t acc_phase = (acc_i >> 1) & 1;
      const bool got = mbar_wait(&c.tfull[acc], acc_phase, abort, p.err, p.wait_ns);
      if (!__all_sync(0xFFFFFFFFu, got)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      uint32_t r[32];
      float v[32];
      bool released = false;
      if constexpr (EPI == EPI_STORE) {
        // drain this warp's 128 columns as packed bf16 and free the accumulator before any
        // store of this tile; the signal is a relaxed arrive (the TMEM loads have completed,
        // no memory access needs ordering), so it does not wait for the stores of earlier
        // tiles either
        uint32_t pk[64];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          tmem_ld_32x32b_x32(taddr + c0 + 32 * j, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[16 * j + i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)
            mbar_arrive_cluster_relaxed(tempty_leader + acc * (uint32_t)sizeof(uint64_t));
          else mbar_arrive_relaxed(&c.tempty[acc]);
        }
        released = true;
        if (row_ok) {
          uint16_t* o = static_cast<uint16_t*>(p.out) + (KG ? (int64_t)t.e * p.out_estride : 0) +
                        (int64_t)row * p.ldo + t.n0 + c0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (t.n0 + c0 + 32 * j >= p.N) break;
            if (p.wide) {
              st_global_v8(o + 32 * j, &pk[16 * j]);
              st_global_v8(o + 32 * j + 16, &pk[16 * j + 8]);
            } else {
              uint4* d = reinterpret_cast<uint4*>(o + 32 * j);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                d[i] = make_uint4(pk[16 * j + 4 * i], pk[16 * j + 4 * i + 1],
                                  pk[16 * j + 4 * i + 2], pk[16 * j + 4 * i + 3]);
            }
          }
        }
      } else if (EPI == EPI_GLU) {
        const float prob = row_ok ? p.row_prob[row] : 0.f;
        uint16_t* zrow = static_cast<uint16_t*>(p.out) + (int64_t)row * p.ldo;
        uint16_t* arow = static_cast<uint16_t*>(p.out2) + (int64_t)row * p.ldo2;
        if (p.gated) {
          // a-columns [half*BN/4, (half+1)*BN/4) of the tile's BN/2 GLU outputs
          for (int cc = half * (BN / 4); cc < (half + 1) * (BN / 4); cc += 32) {
            const int gcol = (cc / p.ilv) * 2 * p.ilv + (cc % p.ilv);
            const int lcol = gcol + p.ilv;
            if (t.n0 + gcol >= p.N) break;
            uint32_t rl[32];
            tmem_ld_32x32b_x32(taddr + gcol, r);
            tmem_ld_32x32b_x32(taddr + lcol, rl);
            tmem_ld_wait();
            float g[32], l[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              g[i] = __uint_as_float(r[i]);
              l[i] = __uint_as_float(rl[i]);
            }
            const int fa = t.n0 / 2 + cc;  // logical activation column of g[0] / l[0]
            if (EXT && p.fc1_bias) {
              const float* b = p.fc1_bias + (int64_t)t.e * p.N;
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                g[i] += b[fa + i];
                l[i] += b[p.F + fa + i];
              }
            }
            glu_fwd32(p.act, prob, g, l, v);
            if (EXT && p.fscale) {
              const float* sc = p.fscale + (int64_t)t.e * p.F;
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] *= sc[fa + i];
            }
            if (row_ok) {
              if (p.out) {  // the saved Z (absent when the backward recomputes it)
                store_bf16x32w(zrow + t.n0 + gcol, g, p.wide);
                store_bf16x32w(zrow + t.n0 + lcol, l, p.wide);
              }
              store_bf16x32w(arow + t.n0 / 2 + cc, v, p.wide);
            }
          }
        } else {
          for (int cc = c0; cc < c1; cc += 32) {
            if (t.n0 + cc >= p.N) break;
            tmem_ld_32x32b_x32(taddr + cc, r);
            tmem_ld_wait();
            float zz[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              zz[i] = __uint_as_float(r[i]);
              const float rr = fmaxf(zz[i], 0.f);
              v[i] = prob * rr * rr;
            }
            if (row_ok) {
              if (p.out) store_bf16x32w(zrow + t.n0 + cc, zz, p.wide);  // saved Z, if kept
              store_bf16x32w(arow + t.n0 + cc, v, p.wide);
            }
          }
        }
      } else {  // EPI_DGLU: accumulator = dA_s over F columns
        // 16-column steps with the saved Z of the next two steps already requested (8 + 8
        // packed words each), so its load latency overlaps two steps of dGLU math
        const float prob = row_ok ? p.row_prob[row] : 0.f;
        float dp = 0.f;
        uint16_t* dzrow = static_cast<uint16_t*>(p.out) + (int64_t)row * p.ldo;
        // the accumulator columns of the next step are loaded from TMEM while this one computes
        uint32_t das[16], nxt[16];
        tmem_ld_32x32b_x16(taddr + c0, das);
        tmem_ld_wait();
#pragma unroll 1
        for (int cc = c0; cc < c1; cc += 16) {
          const int f0 = t.n0 + cc;
          if (f0 >= p.N) break;
          const bool more = cc + 16 < c1 && f0 + 16 < p.N;
          if (more) tmem_ld_32x32b_x16(taddr + cc + 16, nxt);
          if (row_ok && cc + 32 < c1 && f0 + 32 < p.N) z_load16(p, zrow, f0 + 32, z2g, z2l);
          if (EXT && p.gated) {
            // extras: every lane of the warp takes part in the column sums; the warp's 32 rows
            // are all inside the segment or all outside (32-row aligned), and only inside
            // groups own their partials
            const int gcol = (f0 / p.ilv) * 2 * p.ilv + (f0 % p.ilv);
            uint32_t dgw[8], dlw[8];
            float* part = (t.m0 + q * 32 < t.row_end)
                              ? p.ext_part + (int64_t)((t.m0 + q * 32) >> 5) * (p.N1 + p.F)
                              : nullptr;
            dp += dglu16_extras_any(p, prob, das, z0g, z0l, t.e, f0, dgw, dlw, part, lane);
            if (row_ok) {
              st_bf16x16(dzrow + gcol, dgw, p.wide);
              st_bf16x16(dzrow + gcol + p.ilv, dlw, p.wide);
            }
          } else if (row_ok) {
            const int gcol = p.gated ? (f0 / p.ilv) * 2 * p.ilv + (f0 % p.ilv) : f0;
            uint32_t dgw[8], dlw[8];
            if (p.gated) {
              dp += glu_bwd16(p.act, prob, das, z0g, z0l, dgw, dlw);
              st_bf16x16(dzrow + gcol, dgw, p.wide);
              st_bf16x16(dzrow + gcol + p.ilv, dlw, p.wide);
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float d0 = __uint_as_float(das[2 * i]), d1 = __uint_as_float(das[2 * i + 1]);
                const float r0 = fmaxf(bf16_lo(z0g[i]), 0.f), r1 = fmaxf(bf16_hi(z0g[i]), 0.f);
                dp += d0 * r0 * r0 + d1 * r1 * r1;
                dgw[i] = pack_bf16x2(prob * d0 * 2.f * r0, prob * d1 * 2.f * r1);
              }
              st_bf16x16(dzrow + f0, dgw, p.wide);
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            z0g[i] = z1g[i]; z0l[i] = z1l[i];
            z1g[i] = z2g[i]; z1l[i] = z2l[i];
          }
          if (more) {
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) das[i] = nxt[i];
          }
        }
        if (row_ok) p.dprob_part[(int64_t)row * p.nparts + (t.n0 / BN) * 2 + half] = dp;
      }
      if (!released) {
        // every TMEM load of this warp has completed (each was waited for): the accumulator
        // is free, and the signal need not wait for this thread's global stores
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)
            mbar_arrive_cluster_relaxed(tempty_leader + acc * (uint32_t)sizeof(uint64_t));
          else mbar_arrive_relaxed(&c.tempty[acc]);
        }
      }
      ++acc_i;
    }
  }

  griddep_launch_dependents();  // this CTA's tiles are done
  tc_fence_before();
  __syncthreads();
  // a pair: neither CTA leaves while the other may still read its shared memory (the
  // leader's MMAs) or signal its barriers
  if constexpr (PAIR) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, 2 * BN);
    else tmem_dealloc(tmem_base, 2 * BN);
  }
}

template <int BN, int STAGES, bool A_MN, bool B_MN, int EPI, bool KG, bool B3D, bool EXT = false>
cudaError_t launch_instance(const GemmArgs& a, int grid, cudaStream_t s, int kid) {
  auto kern = grouped_gemm_kernel<BN, STAGES, A_MN, B_MN, EPI, KG, B3D, EXT>;
  constexpr int smem = Smem<BN, STAGES>::TOTAL;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  launch_kernel(kern, grid, kThreads, smem, s, nullptr, 0, a);
  count_launch(s, kid);
  return cudaGetLastError();
}

// Clusters of two CTAs; `ctas` (the SMs the caller allows, SM margin applied) is rounded down
// to whole pairs and capped by the number of pairs that can be resident at once.
template <int BN, int STAGES, bool A_MN, bool B_MN, int EPI, bool KG, bool B3D, bool EXT = false>
cudaError_t launch_pair_instance(const GemmArgs& a, int ctas, int64_t tiles, cudaStream_t s,
                                 int kid) {
  auto kern = grouped_gemm_kernel<BN, STAGES, A_MN, B_MN, EPI, KG, B3D, EXT, true>;
  constexpr int smem = Smem<BN, STAGES, true>::TOTAL;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int pairs = std::max(1, ctas / 2);
  const int resident = max_resident_pairs(reinterpret_cast<const void*>(kern), &cfg);
  if (resident > 0) pairs = std::min(pairs, resident);
  pairs = (int)std::max<int64_t>(1, std::min<int64_t>(pairs, tiles));
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  e = launch_kernel(kern, cfg.gridDim, cfg.blockDim, cfg.dynamicSmemBytes, s, attr, 1, a);
  count_launch(s, kid);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

constexpr int kBN = 256;
constexpr int kStages = 4;
constexpr int kPairStages = 6;   // 32 KB per stage and CTA
// the grouped GEMMs run as CTA pairs (256-row tiles, cta_group::2 MMAs); 0 selects the
// one-CTA kernels (128-row tiles)
#ifndef MOE_GEMM_PAIR
#define MOE_GEMM_PAIR 1
#endif
constexpr bool kUsePairs = MOE_GEMM_PAIR != 0;
// weight gradients (k-grouped) on CTA pairs too (same-box A/B: FC1 wgrad 2.79 -> 2.67 ms on
// the Mixtral BF16 layer, 2.09 -> 1.96 on GPT-OSS); 0: one-CTA 128 x 256 tiles
#ifndef MOE_WGRAD_PAIR
#define MOE_WGRAD_PAIR 1
#endif
constexpr bool kWgradPairs = kUsePairs && MOE_WGRAD_PAIR != 0;

}  // namespace

int gemm_bn(int) { return kBN; }

// two epilogue warps (column halves) contribute a partial d_prob per 256-column tile
int dprob_parts(int F) { return 2 * ((F + kBN - 1) / kBN); }

cudaError_t launch_grouped_gemm(const GemmProblem& p, cudaStream_t s) {
  GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.offsets = p.offsets;
  a.E = p.E;
  a.R_cap = (int)p.R_cap;
  a.gated = p.gated;
  a.ilv = p.ilv;
  a.F = p.F;
  a.N1 = p.N1;
  a.fc1_bias = p.fc1_bias;
  a.fscale = p.fscale;
  a.ext_part = p.ext_part;
  a.act = p.act;
  a.err = p.err;
  a.stall_loads = p.stall_loads;
  a.wait_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;
  a.row_prob = p.row_prob;
  static const int kKid[6] = {MOE_K_GEMM_FC1_FPROP, MOE_K_GEMM_FC2_FPROP, MOE_K_GEMM_FC2_DGRAD,
                              MOE_K_GEMM_FC2_WGRAD, MOE_K_GEMM_FC1_DGRAD, MOE_K_GEMM_FC1_WGRAD};
  if (p.role < 0 || p.role > 5) return cudaErrorInvalidValue;
  const int kid = kKid[p.role];
  const uint64_t R = (uint64_t)p.R_cap;
  auto aligned32 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 31) == 0; };
  const int H = p.H, F = p.F, N1 = p.N1, E = p.E;
  bool ok = true;
  const int ctas = p.num_ctas;
  // K-major weight tiles: one box of the B columns a CTA loads (half the tile for a pair)
  constexpr int kBRows = kUsePairs ? kBN / 2 : kBN;
  const int64_t any_tiles = INT64_MAX;  // row-grouped tile count lives on the device
#define MOE_LAUNCH(A_MN, B_MN, EPI, KG, B3D, EXT, TILES)                                        \
  (kUsePairs                                                                                   \
       ? launch_pair_instance<kBN, kPairStages, A_MN, B_MN, EPI, KG, B3D, EXT>(a, ctas, TILES, \
                                                                               s, kid)         \
       : launch_instance<kBN, kStages, A_MN, B_MN, EPI, KG, B3D, EXT>(                         \
             a, (int)std::min<int64_t>(ctas, TILES), s, kid))
  switch (p.role) {
    case ROLE_FC1_FPROP:
      ok &= tmap_2d(&a.tmA, p.x_perm, H, R, 64, BM);
      ok &= tmap_3d(&a.tmB, p.w1p, H, N1, E, 64, kBRows);
      a.K = H; a.N = N1;
      a.out = p.out; a.ldo = N1;
      a.out2 = p.out2; a.ldo2 = F;
      if (!ok) return cudaErrorInvalidValue;
      a.wide = aligned32(a.out) && aligned32(a.out2) && a.ldo % 16 == 0 && a.ldo2 % 16 == 0 &&
               a.out_estride % 16 == 0;
      if (a.fc1_bias || a.fscale) return MOE_LAUNCH(false, false, EPI_GLU, false, true, true, any_tiles);
      return MOE_LAUNCH(false, false, EPI_GLU, false, true, false, any_tiles);
    case ROLE_FC2_FPROP:
      ok &= tmap_2d(&a.tmA, p.a_s, F, R, 64, BM);
      ok &= tmap_3d(&a.tmB, p.w2, H, F, E, 64, 64);
      a.K = F; a.N = H;
      a.out = p.out; a.ldo = H;
      if (!ok) return cudaErrorInvalidValue;
      a.wide = aligned32(a.out) && aligned32(a.out2) && a.ldo % 16 == 0 && a.ldo2 % 16 == 0 &&
               a.out_estride % 16 == 0;
      return MOE_LAUNCH(false, true, EPI_STORE, false, true, false, any_tiles);
    case ROLE_FC2_DGRAD:
      ok &= tmap_2d(&a.tmA, p.dy_perm, H, R, 64, BM);
      ok &= tmap_3d(&a.tmB, p.w2, H, F, E, 64,
                    (kUsePairs && p.rows_per_expert >= 1024) ? kBRows : kBN);
      a.K = H; a.N = F;
      a.out = p.out; a.ldo = N1;
      a.z = static_cast<const uint16_t*>(p.z); a.ldz = N1;
      a.dprob_part = p.dprob_part; a.nparts = dprob_parts(F);
      if (!ok) return cudaErrorInvalidValue;
      a.wide = aligned32(a.out) && aligned32(a.out2) && a.ldo % 16 == 0 && a.ldo2 % 16 == 0 &&
               a.out_estride % 16 == 0;
      // pairs pay for up to 255 rows past each expert's segment end, and this kernel's dGLU
      // epilogue makes those rows expensive: pairs only when the experts average at least 1024
      // rows (measured: Mixtral-shaped, ~2048 rows, 1.40 -> 1.34 ms on pairs; GPT-OSS-shaped,
      // ~512 rows, 0.98 -> 1.03 ms)
      if (kUsePairs && p.rows_per_expert >= 1024) {
        if (a.ext_part) return MOE_LAUNCH(false, false, EPI_DGLU, false, true, true, any_tiles);
        return MOE_LAUNCH(false, false, EPI_DGLU, false, true, false, any_tiles);
      }
      if (a.ext_part)
        return launch_instance<kBN, kStages, false, false, EPI_DGLU, false, true, true>(a, ctas, s,
                                                                                       kid);
      return launch_instance<kBN, kStages, false, false, EPI_DGLU, false, true>(a, ctas, s, kid);
    case ROLE_FC1_DGRAD:
      ok &= tmap_2d(&a.tmA, p.dz, N1, R, 64, BM);
      ok &= tmap_3d(&a.tmB, p.w1p, H, N1, E, 64, 64);
      a.K = N1; a.N = H;
      a.out = p.out; a.ldo = H;
      if (!ok) return cudaErrorInvalidValue;
      a.wide = aligned32(a.out) && aligned32(a.out2) && a.ldo % 16 == 0 && a.ldo2 % 16 == 0 &&
               a.out_estride % 16 == 0;
      return MOE_LAUNCH(false, true, EPI_STORE, false, true, false, any_tiles);
    case ROLE_FC2_WGRAD:
    case ROLE_FC1_WGRAD: {
      const bool fc2 = p.role == ROLE_FC2_WGRAD;
      const int M = fc2 ? F : N1;
      ok &= tmap_2d(&a.tmA, fc2 ? p.a_s : p.dz, M, R, 64, 64);
      ok &= tmap_2d(&a.tmB, fc2 ? p.dy_perm : p.x_perm, H, R, 64, 64);
      a.M = M; a.N = H;
      a.out = p.out; a.ldo = H; a.out_estride = (int64_t)M * H;
      if (!ok) return cudaErrorInvalidValue;
      a.wide = aligned32(a.out) && a.ldo % 16 == 0 && a.out_estride % 16 == 0;
      if constexpr (kWgradPairs) {
        const int64_t tiles = (int64_t)E * ((M + 2 * BM - 1) / (2 * BM)) * ((H + kBN - 1) / kBN);
        return launch_pair_instance<kBN, kPairStages, true, true, EPI_STORE, true, false>(
            a, ctas, tiles, s, kid);
      } else {
        const int64_t tiles = (int64_t)E * ((M + BM - 1) / BM) * ((H + kBN - 1) / kBN);
        return launch_instance<kBN, kStages, true, true, EPI_STORE, true, false>(
            a, (int)std::min<int64_t>(ctas, tiles), s, kid);
      }
    }
  }
#undef MOE_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace moe
