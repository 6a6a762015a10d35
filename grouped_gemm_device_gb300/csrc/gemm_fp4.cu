// Persistent block-scaled NVFP4 grouped GEMM for sm_103a.
//
// [NV-blog] kernel families with NVFP4 operands: (1) GroupGemm (FC2 fprop, FC1 dgrad, wgrads),
// (2) FC1 + activation, (3) FC2 dgrad + dActivation; section "fused MXFP8 and NVFP4
// quantisation": for NVFP4 the FC1 kernel emits its BF16 output plus the per-tensor amax and
// the FC2-dgrad kernel the amax of its output's Hadamard-rotated transpose, so the NVFP4
// quantiser that follows needs no pass of its own to find them. Here both epilogues emit
// both amaxes (plain, for the row-wise copy of the next GEMM; rotated, for the transposed
// weight-gradient copy), as one atomic max per warp at the end of the kernel.
//
// Operands are NVFP4 copies (nvfp4.cuh), all K-major (sub-byte MMA operands have no MN-major
// form): packed E2M1 [rows, K/2] and E4M3 scales in the slab layout. A CTA:
//   warp 0   TMA of the A (128 x 128 B = 256 values) and B (256 x 128 B) k-blocks and eight
//            1-D bulk copies of their scale slabs (4 x 512 + 4 x 1024 bytes), one mbarrier;
//   warp 1   TMEM owner; one thread copies the stage's scales into TMEM (tcgen05.cp, 48
//            columns a stage) and issues four tcgen05.mma.kind::mxf4nvf4.block_scale
//            (scale_vec::4X) 128x256x64, each with its own 512-byte scale slab per 128 rows;
//   warps 2-9 epilogue: drain the accumulator into registers (warp w takes TMEM lanes
//            32*(w%4).. and 128 of the 256 columns) times 1 / (S_a S_b), release TMEM, then
//            bf16 store, GLU or dGLU.
// TMEM: one 256-column fp32 accumulator plus 4 x 48 scale columns. Expert segments are padded
// to 128 rows, so every row-grouped tile lies inside one segment (padding rows carry
// probability 0 and zero operands) and every weight-gradient k range starts on a scale slab.
#include "gemm_common.cuh"
#include "nvfp4.cuh"

namespace moe {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 256;       // E2M1 values per k-block: one 128-byte swizzle row
constexpr int BKB = BK / 2;   // bytes per k-block row
constexpr int MMA_K = 64;     // values per MMA: 32 bytes along the swizzled row
constexpr int STAGES = 4;
constexpr int ILV = 64;       // gate/linear interleave of the packed FC1 columns
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kMaxE = 256;
constexpr int kSfCol = BN;              // first TMEM column of the scale factors
constexpr int kSfColsPerMma = 12;       // 4 (A, 128 rows) + 8 (B, 256 rows)
constexpr int kSfColsPerStage = 4 * kSfColsPerMma;
constexpr int kTmemCols = 512;
static_assert(kSfCol + STAGES * kSfColsPerStage <= kTmemCols, "TMEM map");

enum { EPI_STORE = 0, EPI_GLU = 1, EPI_DGLU = 2 };

constexpr int A_BYTES = BM * BKB;
constexpr int B_BYTES = BN * BKB;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SFA_SLAB = 512;    // 128 rows x 4 blocks of 16 values
constexpr int SFB_SLAB = 1024;   // 256 rows x 4 blocks
constexpr int SF_STAGE = 4 * (SFA_SLAB + SFB_SLAB);
constexpr int SF_OFF = STAGES * STAGE_BYTES;
constexpr int CTRL_OFF = SF_OFF + STAGES * SF_STAGE;
constexpr int SMEM_TOTAL = CTRL_OFF + 4096 + 1024;
static_assert(SMEM_TOTAL <= 232448, "shared memory above the per-block limit");

struct Fp4Args {
  CUtensorMap tmA;
  CUtensorMap tmB;
  const uint8_t* sfa;
  int64_t sfa_pad;
  const uint8_t* sfb;
  int64_t sfb_pad;
  const int32_t* offsets;
  int E;
  int R_cap;
  int M, N, K;
  int a_row_e, a_k_e, b_row_e, b_k_e;  // per-expert row / k offsets of A and B
  void* out;                           // bf16: STORE output, GLU saved Z, dGLU dZ
  int64_t ldo;
  int64_t out_estride;
  void* out2;                          // GLU: bf16 a_s
  int64_t ldo2;
  const float* row_prob;
  const uint16_t* z;                   // dGLU: saved Z (bf16, packed columns)
  int64_t ldz;
  float* dprob_part;
  int nparts;
  const float* amax_a;                 // per-tensor amax of the A and B copies
  const float* amax_b;
  float* amax_out;                     // GLU / dGLU: amax of the bf16 output
  float* amax_out_rht;                 //   and of its 16-row rotation along the rows
  uint32_t rht_mask;
  int wide;                            // STORE: out is 32-byte aligned (256-bit stores)
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
static_assert(sizeof(Ctrl) <= 4096, "control block");

struct TileInfo {
  int e, m0, n0, kbeg, klen, nkb, row_end;
};

template <bool KG>
MOE_DEVICE void decode_tile(int tile, const Fp4Args& p, const Ctrl& c, int MT, int NT,
                            TileInfo& t) {
  if (!KG) {
    int lo = 0, hi = p.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (c.prefix[mid] <= tile) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int local = tile - c.prefix[e];
    const int mt = (c.off[e + 1] - c.off[e] + BM - 1) / BM;
    t.e = e;
    t.m0 = c.off[e] + (local % mt) * BM;
    t.n0 = (local / mt) * BN;
    t.kbeg = 0;
    t.klen = p.K;
    t.nkb = (p.K + BK - 1) / BK;
    t.row_end = c.off[e + 1];
  } else {
    const int per = MT * NT;
    const int e = tile / per;
    const int local = tile - e * per;
    t.e = e;
    t.m0 = (local / NT) * BM;
    t.n0 = (local % NT) * BN;
    t.kbeg = c.off[e];
    t.klen = c.off[e + 1] - c.off[e];
    t.nkb = (t.klen + BK - 1) / BK;
    t.row_end = p.M;
  }
}

// Instruction descriptor of tcgen05.mma.kind::mxf4nvf4: A and B E2M1 (format 1), K-major,
// N >> 3 at bit 17, scale type UE4M3 (bit 23 clear), M >> 4 at bit 24, scale ids 0 (the
// 4X form takes a whole 32-bit scale word per row).
constexpr uint32_t idesc_nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= (A . SFA) (B . SFB)^T over K = 64: E2M1 operands in shared memory, one E4M3
// scale per 16 values of each row in TMEM.
MOE_DEVICE void mma_nvf4_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

MOE_DEVICE float bf16r(float x) { return bf16_lo(pack_bf16x2(x, 0.f)); }

// 16 floats (already bf16 values) -> 32 bytes of bf16 at a 32-byte aligned address.
MOE_DEVICE void store_bf16x16_v8(void* dst, const float (&v)[16]) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
  st_global_v8(dst, w);
}

// Gate column of dA column f in the packed Z layout (blocks of ILV gate columns followed by
// ILV linear columns).
MOE_DEVICE int gate_col(int f) { return ((f & ~(ILV - 1)) << 1) | (f & (ILV - 1)); }

template <int EPI, int KIND, bool KG>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_fp4_kernel(const __grid_constant__ Fp4Args p) {
  constexpr bool kGated = KIND != MOE_ACT_SRELU;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  Ctrl& c = *reinterpret_cast<Ctrl*>(smem + CTRL_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &c.abort;
  const int NT = (p.N + BN - 1) / BN;
  const int MT = KG ? (p.M + BM - 1) / BM : 0;

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
      // segments must start on 128-row boundaries (scale slabs)
      if (o < prev || o > p.R_cap || (o & (BM - 1)) || (e == 0 && o != 0)) ok = false;
      c.off[e] = o;
      prev = o;
    }
    int total = 0;
    if (ok) {
      for (int e = 0; e < p.E; ++e) {
        c.prefix[e] = total;
        total += KG ? MT * NT : ((c.off[e + 1] - c.off[e] + BM - 1) / BM) * NT;
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
    tmem_alloc(&c.tmem_base, kTmemCols);
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
        TileInfo t;
        decode_tile<KG>(tile, p, c, MT, NT, t);
        const int a_row = t.m0 + t.e * p.a_row_e;
        const int b_row = t.n0 + t.e * p.b_row_e;
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!mbar_wait(&c.empty[stage], phase ^ 1, abort, p.err)) break;
          uint8_t* sA = smem + stage * STAGE_BYTES;
          uint8_t* sB = sA + A_BYTES;
          uint8_t* sf = smem + SF_OFF + stage * SF_STAGE;
          uint64_t* bar = &c.full[stage];
          mbar_arrive_expect_tx(bar, STAGE_BYTES + SF_STAGE);
#pragma unroll
          for (int s = 0; s < STAGES; ++s)
            if (s == stage) armed[s] = (int)phase;
          const int k0 = t.kbeg + kb * BK;  // a multiple of 128 (of 256 when row-grouped)
          const int a_k = k0 + t.e * p.a_k_e;
          const int b_k = k0 + t.e * p.b_k_e;
          // boxes of 128 rows x 128 bytes at byte column k / 2 (a multiple of 32)
          tma_load_2d(sA, &p.tmA, bar, a_k / 2, a_row);
          tma_load_2d(sB, &p.tmB, bar, b_k / 2, b_row);
          tma_load_2d(sB + B_BYTES / 2, &p.tmB, bar, b_k / 2, b_row + 128);
          // four 64-value scale slabs of each operand: A's 128 rows, B's 256 rows
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            bulk_load(sf + s * SFA_SLAB,
                      p.sfa + ((int64_t)(a_k / MMA_K + s) * p.sfa_pad + a_row) * 4, SFA_SLAB,
                      bar);
            bulk_load(sf + 4 * SFA_SLAB + s * SFB_SLAB,
                      p.sfb + ((int64_t)(b_k / MMA_K + s) * p.sfb_pad + b_row) * 4, SFB_SLAB,
                      bar);
          }
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
    // ------------------------------------------------------------ scale copy + MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_nvf4(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc_i = 0;
      bool issued_any = false;
      for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x) {
        TileInfo t;
        decode_tile<KG>(tile, p, c, MT, NT, t);
        if (t.nkb == 0) continue;
        // the single accumulator is free once every epilogue warp drained the last tile
        if (!mbar_wait(&c.tempty, (acc_i & 1) ^ 1, abort, p.err)) break;
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!mbar_wait(&c.full[stage], phase, abort, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sB = sA + A_BYTES;
          const uint32_t sf = smem_u32(smem + SF_OFF + stage * SF_STAGE);
          const uint32_t sft = tmem_base + kSfCol + stage * kSfColsPerStage;
          const int rem = t.klen - kb * BK;
          const int nsub = rem >= BK ? BK / MMA_K : (rem + MMA_K - 1) / MMA_K;
          for (int s = 0; s < nsub; ++s) {
            const uint32_t col = sft + s * kSfColsPerMma;
            tmem_cp_32x128b_warpx4(col, smem_desc_noswizzle(sf + s * SFA_SLAB, 0, 128));
            tmem_cp_32x128b_warpx4(col + 4, smem_desc_noswizzle(sf + 4 * SFA_SLAB + s * SFB_SLAB,
                                                                0, 128));
            tmem_cp_32x128b_warpx4(col + 8, smem_desc_noswizzle(
                                                sf + 4 * SFA_SLAB + s * SFB_SLAB + 512, 0, 128));
          }
          for (int s = 0; s < nsub; ++s) {
            const uint32_t col = sft + s * kSfColsPerMma;
            mma_nvf4_ss(tmem_base, smem_desc_sw128(sA + s * (MMA_K / 2), 16, 1024),
                        smem_desc_sw128(sB + s * (MMA_K / 2), 16, 1024), IDESC, col, col + 4,
                        (kb | s) != 0 ? 1u : 0u);
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
    // Control flow stays warp-uniform (the rotation amax exchanges values across lanes).
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;  // columns [128*half, 128*half + 128) of the tile
    const float alpha =
        __frcp_rn(__fmul_rn(nvfp4_encode_scale(*p.amax_a), nvfp4_encode_scale(*p.amax_b)));
    float m_out = 0.f, m_rht = 0.f;
    int acc_i = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      if (__shfl_sync(0xFFFFFFFFu, *abort, 0)) break;
      TileInfo t;
      decode_tile<KG>(tile, p, c, MT, NT, t);
      const int row0 = t.m0 + q * 32;
      const int row = row0 + lane;
      const bool row_ok = row < t.row_end;
      const int cb = half * 128;
      if (t.nkb == 0) {
        if (row_ok) {
          uint16_t* o = static_cast<uint16_t*>(p.out) + (int64_t)t.e * p.out_estride +
                        (int64_t)row * p.ldo;
          for (int cc = cb; cc < cb + 128 && t.n0 + cc < p.N; cc += 32)
            store_zero_bf16x32(o + t.n0 + cc);
        }
        continue;
      }
      const float prob = EPI == EPI_STORE ? 0.f : p.row_prob[row];
      const bool got = mbar_wait(&c.tfull, acc_i & 1, abort, p.err);
      if (!__all_sync(0xFFFFFFFFu, got)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + cb;
      if constexpr (EPI == EPI_STORE) {
        uint32_t pk[64];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tacc + 32 * j, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[16 * j + i] = pack_bf16x2(alpha * __uint_as_float(r[2 * i]),
                                         alpha * __uint_as_float(r[2 * i + 1]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.tempty);
        ++acc_i;
        if (row_ok) {
          uint16_t* o = static_cast<uint16_t*>(p.out) + (KG ? (int64_t)t.e * p.out_estride : 0) +
                        (int64_t)row * p.ldo + t.n0 + cb;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (t.n0 + cb + 32 * j < p.N) {
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
        }
      } else {
      // GLU / dGLU: the 128 columns as fp32 (activation math from the fp32 accumulator)
      float acc[128];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tacc + 32 * j, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[32 * j + i] = alpha * __uint_as_float(r[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.tempty);
      ++acc_i;
      // row-grouped segments are 128-row aligned: every row of the tile is in its segment
      if constexpr (EPI == EPI_GLU) {
        uint16_t* zout = static_cast<uint16_t*>(p.out) + (int64_t)row * p.ldo + t.n0 + cb;
#pragma unroll
        for (int j = 0; j < 4; ++j)  // the saved Z (bf16)
          if (t.n0 + cb + 32 * j < p.N) store_bf16x32_v8(zout + 32 * j, &acc[32 * j]);
        uint16_t* aout = static_cast<uint16_t*>(p.out2) + (int64_t)row * p.ldo2;
        // gated: this half holds 64 gate and 64 linear columns, two 32-wide output blocks;
        // sReLU: four 32-wide blocks
#pragma unroll
        for (int c32 = 0; c32 < (kGated ? 2 : 4); ++c32) {
          const int g_off = c32 * 32;
          const int acol = kGated ? (t.n0 + cb) / 2 + c32 * 32 : t.n0 + cb + c32 * 32;
          if (t.n0 + cb + g_off >= p.N) break;
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float a;
            if constexpr (kGated) {
              a = act_fwd_k<KIND>(p.act, acc[g_off + i], acc[g_off + ILV + i]);
            } else {
              const float rr = fmaxf(acc[g_off + i], 0.f);
              a = rr * rr;
            }
            v[i] = bf16r(prob * a);
          }
          store_bf16x32_v8(aout + acol, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            m_out = fmaxf(m_out, fabsf(v[i]));
            m_rht = fmaxf(m_rht, fabsf(rht16_lanes(v[i], p.rht_mask, lane)));
          }
        }
      } else {  // EPI_DGLU: accumulator = dA_s over F columns
        const uint16_t* zrow = p.z + (int64_t)row * p.ldz;
        uint16_t* dzrow = static_cast<uint16_t*>(p.out) + (int64_t)row * p.ldo;
        float dp = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int f0 = t.n0 + cb + 16 * j;
          if (f0 >= p.N) break;
          const int gc = kGated ? gate_col(f0) : f0;
          uint32_t gw[8], lw[8];
          ld_v8_noalloc(zrow + gc, gw);
          if constexpr (kGated) ld_v8_noalloc(zrow + gc + ILV, lw);
          float dg[16], dl[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float d = acc[16 * j + i];
            const float g = (i & 1) ? bf16_hi(gw[i >> 1]) : bf16_lo(gw[i >> 1]);
            if constexpr (kGated) {
              const float l = (i & 1) ? bf16_hi(lw[i >> 1]) : bf16_lo(lw[i >> 1]);
              dp += d * act_bwd_k<KIND>(p.act, g, l, prob * d, dg[i], dl[i]);
              dl[i] = bf16r(dl[i]);
            } else {
              const float rr = fmaxf(g, 0.f);
              dp += d * rr * rr;
              dg[i] = prob * d * 2.f * rr;
            }
            dg[i] = bf16r(dg[i]);
          }
          store_bf16x16_v8(dzrow + gc, dg);
          if constexpr (kGated) store_bf16x16_v8(dzrow + gc + ILV, dl);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            m_out = fmaxf(m_out, fabsf(dg[i]));
            m_rht = fmaxf(m_rht, fabsf(rht16_lanes(dg[i], p.rht_mask, lane)));
            if constexpr (kGated) {
              m_out = fmaxf(m_out, fabsf(dl[i]));
              m_rht = fmaxf(m_rht, fabsf(rht16_lanes(dl[i], p.rht_mask, lane)));
            }
          }
        }
        p.dprob_part[(int64_t)row * p.nparts + (t.n0 / BN) * 2 + half] = dp;
      }
      }  // GLU / dGLU
    }
    if constexpr (EPI != EPI_STORE) {
      amax_flush_warp(m_out, p.amax_out);
      amax_flush_warp(m_rht, p.amax_out_rht);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// K-major NVFP4 operand: packed codes [rows, cols / 2] bytes, boxes of 128 rows x 128 bytes.
bool tmap_fp4(CUtensorMap* m, const MxOperand& t) {
  uint64_t dims[2] = {(uint64_t)(t.cols / 2), (uint64_t)t.rows};
  uint64_t strides[1] = {(uint64_t)(t.cols / 2)};
  uint32_t box[2] = {128, 128};
  return make_tmap(m, t.q, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

template <int EPI, int KIND, bool KG>
cudaError_t launch_fp4(const Fp4Args& a, int grid, cudaStream_t s, int kid) {
  auto kern = grouped_gemm_fp4_kernel<EPI, KIND, KG>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), SMEM_TOTAL);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, SMEM_TOTAL, s>>>(a);
  count_launch(s, kid);
  return cudaGetLastError();
}

template <int EPI>
cudaError_t launch_act_family(const Fp4Args& a, int kind, int grid, cudaStream_t s, int kid) {
  switch (kind) {
    case MOE_ACT_SWIGLU: return launch_fp4<EPI, MOE_ACT_SWIGLU, false>(a, grid, s, kid);
    case MOE_ACT_CLAMPED_SWIGLU:
      return launch_fp4<EPI, MOE_ACT_CLAMPED_SWIGLU, false>(a, grid, s, kid);
    case MOE_ACT_GEGLU: return launch_fp4<EPI, MOE_ACT_GEGLU, false>(a, grid, s, kid);
    case MOE_ACT_SRELU: return launch_fp4<EPI, MOE_ACT_SRELU, false>(a, grid, s, kid);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int dprob_parts_fp4(int F) { return 2 * ((F + BN - 1) / BN); }

cudaError_t launch_grouped_gemm_fp4(const Fp4Problem& p, cudaStream_t s) {
  static const int kKid[6] = {MOE_K_GEMM_FC1_FPROP, MOE_K_GEMM_FC2_FPROP, MOE_K_GEMM_FC2_DGRAD,
                              MOE_K_GEMM_FC2_WGRAD, MOE_K_GEMM_FC1_DGRAD, MOE_K_GEMM_FC1_WGRAD};
  if (p.role < 0 || p.role > 5) return cudaErrorInvalidValue;
  if (p.gated && p.ilv != ILV) return cudaErrorInvalidValue;
  if (p.gated != (p.act.kind != MOE_ACT_SRELU)) return cudaErrorInvalidValue;
  Fp4Args a;
  memset(&a, 0, sizeof(a));
  a.offsets = p.offsets;
  a.E = p.E;
  a.R_cap = (int)p.R_cap;
  a.act = p.act;
  a.err = p.err;
  a.row_prob = p.row_prob;
  a.rht_mask = p.rht_mask;
  const int H = p.H, F = p.F, N1 = p.N1;
  const MxOperand *A = nullptr, *B = nullptr;
  int grid = p.num_ctas;
  switch (p.role) {
    case ROLE_FC1_FPROP:  // X x W1 (rows e*N1p + n), K = H
      A = &p.x; B = &p.w1;
      a.K = H; a.N = N1; a.b_row_e = p.N1p;
      a.out = p.out; a.ldo = N1;
      a.out2 = p.out2; a.ldo2 = F;
      a.amax_a = p.amax + AM_X; a.amax_b = p.amax + AM_W1;
      a.amax_out = p.amax + AM_A; a.amax_out_rht = p.amax + AM_AT;
      break;
    case ROLE_FC2_FPROP:  // a_s x W2^T copy ([H, E*Fp]), K = F
      A = &p.a; B = &p.w2t;
      a.K = F; a.N = H; a.b_k_e = p.Fp;
      a.out = p.out; a.ldo = H;
      a.amax_a = p.amax + AM_A; a.amax_b = p.amax + AM_W2;
      break;
    case ROLE_FC2_DGRAD:  // dY x W2 (rows e*Fp + f), K = H
      A = &p.dy; B = &p.w2;
      a.K = H; a.N = F; a.b_row_e = p.Fp;
      a.z = static_cast<const uint16_t*>(p.z); a.ldz = N1;
      a.out = p.out; a.ldo = N1;
      a.dprob_part = p.dprob_part; a.nparts = dprob_parts_fp4(F);
      a.amax_a = p.amax + AM_DY; a.amax_b = p.amax + AM_W2;
      a.amax_out = p.amax + AM_DZ; a.amax_out_rht = p.amax + AM_DZT;
      break;
    case ROLE_FC1_DGRAD:  // dZ x W1^T copy ([H, E*N1p]), K = N1
      A = &p.dz; B = &p.w1t;
      a.K = N1; a.N = H; a.b_k_e = p.N1p;
      a.out = p.out; a.ldo = H;
      a.amax_a = p.amax + AM_DZ; a.amax_b = p.amax + AM_W1;
      break;
    case ROLE_FC2_WGRAD:  // dW2_e [F, H] = a_s^T dY over the expert's rows (rotated copies)
      A = &p.at; B = &p.dyt;
      a.M = F; a.N = H;
      a.out = p.out; a.ldo = H; a.out_estride = (int64_t)F * H;
      a.amax_a = p.amax + AM_AT; a.amax_b = p.amax + AM_DYT;
      break;
    case ROLE_FC1_WGRAD:  // dW1_e [N1, H] = dZ^T X over the expert's rows (rotated copies)
      A = &p.dzt; B = &p.xt;
      a.M = N1; a.N = H;
      a.out = p.out; a.ldo = H; a.out_estride = (int64_t)N1 * H;
      a.amax_a = p.amax + AM_DZT; a.amax_b = p.amax + AM_XT;
      break;
  }
  if (!tmap_fp4(&a.tmA, *A) || !tmap_fp4(&a.tmB, *B)) return cudaErrorInvalidValue;
  a.sfa = A->s; a.sfa_pad = A->s_pad;
  a.sfb = B->s; a.sfb_pad = B->s_pad;
  a.wide = (reinterpret_cast<uintptr_t>(a.out) & 31) == 0 && a.ldo % 16 == 0 &&
           a.out_estride % 16 == 0;
  const int kid = kKid[p.role];
  switch (p.role) {
    case ROLE_FC1_FPROP: return launch_act_family<EPI_GLU>(a, p.act.kind, grid, s, kid);
    case ROLE_FC2_DGRAD: return launch_act_family<EPI_DGLU>(a, p.act.kind, grid, s, kid);
    case ROLE_FC2_FPROP:
    case ROLE_FC1_DGRAD:
      return launch_fp4<EPI_STORE, 0, false>(a, grid, s, kid);
    default: {
      const int64_t tiles = (int64_t)p.E * ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
      grid = (int)std::min<int64_t>(grid, std::max<int64_t>(tiles, 1));
      return launch_fp4<EPI_STORE, 0, true>(a, grid, s, kid);
    }
  }
}

}  // namespace moe
