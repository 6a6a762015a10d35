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
//   warps 2-9 epilogue (warp w reads TMEM lanes 32*(w%4)..): results times 1 / (S_a S_b).
// Two tile shapes:
//   STORE and GLU (FC2 fprop, FC1 dgrad, wgrads; FC1 fprop): 128 x 256 tiles (a 128 x 256 x 64
//     MMA costs about what a 128-wide one does), one 256-column accumulator that the epilogue
//     drains into registers (128 columns a warp) and releases at once; 4 stages;
//   dGLU (FC2 dgrad), whose epilogue is several times heavier than its mainloop: 128 x 128
//     tiles and two 128-column accumulators, so that the epilogue reads TMEM step by step with
//     no accumulator in registers while the next tile's MMAs run; 4 stages, the fifth stage's
//     space holding the saved-Z staging and the rotation transposes.
// The rotated amax goes across lanes by shuffles in the GLU epilogue (64 values a thread and
// tile) and through a per-warp shared-memory transpose in the dGLU epilogue (each lane rotates
// a column of 16 rows in registers); both perform the quantiser's fp32 butterflies.
// TMEM: 256 accumulator columns, then the scale columns of every stage. Expert segments are
// padded to 128 rows, so every row-grouped tile lies inside one segment (padding rows carry
// probability 0 and zero operands) and every weight-gradient k range starts on a scale slab.
#include "gemm_common.cuh"
#include "nvfp4.cuh"

namespace moe {

namespace {

constexpr int BM = 128;
constexpr int BK = 256;       // E2M1 values per k-block: one 128-byte swizzle row
constexpr int BKB = BK / 2;   // bytes per k-block row
constexpr int MMA_K = 64;     // values per MMA: 32 bytes along the swizzled row
constexpr int kMaxStages = 5;
constexpr int ILV = 64;       // gate/linear interleave of the packed FC1 columns
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
#ifndef FP4_DGLU_WARPS
#define FP4_DGLU_WARPS 8
#endif
constexpr int kMaxE = 256;
constexpr int kTmemCols = 512;

enum { EPI_STORE = 0, EPI_GLU = 1, EPI_DGLU = 2 };

constexpr int A_BYTES = BM * BKB;
constexpr int SFA_SLAB = 512;            // 128 rows x 4 blocks of 16 values
constexpr int ZQ_BUF = 32 * 64;          // dGLU: one 16-column step of saved Z, 32 rows
constexpr int ZQ_WARP = 2 * ZQ_BUF;      //   double-buffered per epilogue warp
constexpr int XT_PITCH = 20;             // words per row of the rotation transpose tile
constexpr int XT_WARP = (32 * XT_PITCH + 16) * 4;  // rows 16..31 shifted by 16 words

// Tile shape, pipeline depth and shared-memory / TMEM maps of one epilogue kind.
template <int EPI>
struct Fp4Cfg {
  static constexpr int BN = 256;
  static constexpr int NACC = 1;
  // the dGLU epilogue (saved-Z loads, activation gradient, rotated amax) outlasts the tile's
  // MMAs with eight warps: it takes FP4_DGLU_WARPS, each lane quadrant's warps dealing the
  // tile's 16-column chunks round-robin, with one stage fewer to make room for their buffers
  static constexpr int EW = EPI == EPI_DGLU ? FP4_DGLU_WARPS : kEpiWarps;
  static constexpr int EWQ = EW / 4;  // warps per lane quadrant
  static constexpr int THREADS = 64 + 32 * EW;
  static constexpr int STAGES = EPI == EPI_DGLU ? (EW > 8 ? 2 : 3) : 4;
  static constexpr int B_BYTES = BN * BKB;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int SFB_SLAB = BN * 4;
  static constexpr int SF_STAGE = 4 * (SFA_SLAB + SFB_SLAB);
  static constexpr int SF_COLS_MMA = 4 + 4 * (BN / 128);  // A's 128 rows + B's BN rows
  static constexpr int SF_COLS_STAGE = 4 * SF_COLS_MMA;
  // TMEM: the fp32 accumulator, then the stages' scale columns; the dGLU keeps instead a
  // bf16-packed copy of its accumulator (128 columns, so the accumulator is freed for the next
  // tile's MMAs while the epilogue works) and two scale buffers of half a k-block each, reused
  // once the MMAs that read them have completed
  static constexpr int PACK_COL = BN;
  static constexpr int SF_COL0 = EPI == EPI_DGLU ? BN + BN / 2 : NACC * BN;
  static constexpr int SF_HALF = 2 * SF_COLS_MMA;
  static constexpr int SF_OFF = STAGES * STAGE_BYTES;
  static constexpr int ZQ_OFF = SF_OFF + STAGES * SF_STAGE;
  static constexpr int XT_OFF = ZQ_OFF + (EPI == EPI_DGLU ? EW * ZQ_WARP : 0);
  static constexpr int CTRL_OFF = XT_OFF + (EPI == EPI_DGLU ? EW * XT_WARP : 0);
  static constexpr int TOTAL = CTRL_OFF + 4096 + 1024;
  static_assert(TOTAL <= 232448, "shared memory above the per-block limit");
  static_assert(SF_COL0 + (EPI == EPI_DGLU ? 2 * SF_HALF : STAGES * SF_COLS_STAGE) <= kTmemCols,
                "TMEM map");
  static_assert(EPI != EPI_DGLU || PACK_COL + BN / 2 <= SF_COL0, "TMEM map: packed copy");
  static_assert(STAGES <= kMaxStages, "barrier arrays");
  static_assert(EWQ * 4 == EW && THREADS <= 1024, "whole lane quadrants");
  static_assert(ZQ_OFF % 16 == 0 && XT_OFF % 16 == 0 && CTRL_OFF % 8 == 0, "alignment");
};

struct Fp4Args {
  CUtensorMap tmA;
  CUtensorMap tmB;
  CUtensorMap tmSFA;  // A's scale slabs: boxes of 128 rows x the four slabs of a k-block
  CUtensorMap tmSFB;  // B's: BN rows x four slabs
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
  // EXT kernels: FC1 bias [E, N1] (logical [gate | linear] order), feature scale [E, F], and
  // the dGLU's per-32-row column sums of dZ and of p * dA_s * a into ext_part [., N1 + F]
  const float* fc1_bias;
  const float* fscale;
  float* ext_part;
  int F, N1;
};

struct Ctrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t sfh[2];  // dGLU: the MMAs that read scale buffer h have completed
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

template <int BN, bool KG>
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

// dGLU saved-Z staging: each lane copies its own row's 16 gate (and 16 linear) values of one
// 16-column step, four 16-byte pieces, into a 64-byte slot of the warp's buffer (pieces
// XOR-rotated by lane so that the 16-byte reads of eight lanes hit distinct banks).
MOE_DEVICE uint32_t zq_slot(int lane, int piece) {
  return lane * 64 + ((piece ^ ((lane >> 1) & 3)) * 16);
}
MOE_DEVICE void zq_issue(uint32_t buf, const uint16_t* src, bool gated, int lane) {
#pragma unroll
  for (int pc = 0; pc < 4; ++pc) {
    if (pc >= 2 && !gated) break;
    const uint16_t* g = src + (pc >= 2 ? ILV : 0) + (pc & 1) * 8;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(buf + zq_slot(lane, pc)),
                 "l"(g)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Max |rotated value| of the warp's 32 rows x 32 bf16 columns (lane = row; w = its 32 values
// as bf16 pairs): the tile goes through shared memory, then lane l rotates columns
// 2 (l % 16) and 2 (l % 16) + 1 over rows 16 (l / 16) .. + 15 with the register butterflies.
MOE_DEVICE float rht_amax_tile32(uint32_t* xt, const uint32_t (&w)[16], uint32_t mask,
                                 int lane) {
  uint32_t* row = xt + lane * XT_PITCH + (lane >= 16 ? 16 : 0);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    *reinterpret_cast<uint4*>(row + 4 * k) =
        make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
  __syncwarp();
  const int cw = lane & 15, h = lane >> 4;
  const uint32_t* col = xt + (16 * h) * XT_PITCH + 16 * h + cw;
  float a[16], b[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t v = col[i * XT_PITCH];
    a[i] = bf16_lo(v);
    b[i] = bf16_hi(v);
  }
  __syncwarp();  // every lane has read the tile before the next call rewrites it
  rht16_regs(a, mask);
  rht16_regs(b, mask);
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fmaxf(fabsf(a[i]), fabsf(b[i])));
  return m;
}

// Gate column of dA column f in the packed Z layout (blocks of ILV gate columns followed by
// ILV linear columns).
MOE_DEVICE int gate_col(int f) { return ((f & ~(ILV - 1)) << 1) | (f & (ILV - 1)); }

template <int EPI, int KIND, bool KG, bool EXT = false>
__global__ void __launch_bounds__(Fp4Cfg<EPI>::THREADS, 1)
    grouped_gemm_fp4_kernel(const __grid_constant__ Fp4Args p) {
  MOE_GRIDDEP_ENTRY();
  constexpr bool kGated = KIND != MOE_ACT_SRELU;
  static_assert(!EXT || (kGated && EPI != EPI_STORE), "extras: gated GLU / dGLU epilogues");
  using L = Fp4Cfg<EPI>;
  constexpr int BN = L::BN;
  constexpr int NACC = L::NACC;
  constexpr int STAGES = L::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  Ctrl& c = *reinterpret_cast<Ctrl*>(smem + L::CTRL_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &c.abort;
  const int NT = (p.N + BN - 1) / BN;
  const int MT = KG ? (p.M + BM - 1) / BM : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c.tfull[i], 1);
      mbar_init(&c.tempty[i], L::EW);
      mbar_init(&c.sfh[i], 1);
    }
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
    tma_prefetch_desc(&p.tmSFA);
    tma_prefetch_desc(&p.tmSFB);
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
        decode_tile<BN, KG>(tile, p, c, MT, NT, t);
        const int a_row = t.m0 + t.e * p.a_row_e;
        const int b_row = t.n0 + t.e * p.b_row_e;
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!mbar_wait(&c.empty[stage], phase ^ 1, abort, p.err)) break;
          uint8_t* sA = smem + stage * L::STAGE_BYTES;
          uint8_t* sB = sA + A_BYTES;
          uint8_t* sf = smem + L::SF_OFF + stage * L::SF_STAGE;
          uint64_t* bar = &c.full[stage];
          mbar_arrive_expect_tx(bar, L::STAGE_BYTES + L::SF_STAGE);
#pragma unroll
          for (int s = 0; s < STAGES; ++s)
            if (s == stage) armed[s] = (int)phase;
          const int k0 = t.kbeg + kb * BK;  // a multiple of 128 (of 256 when row-grouped)
          const int a_k = k0 + t.e * p.a_k_e;
          const int b_k = k0 + t.e * p.b_k_e;
          // boxes of 128 rows x 128 bytes at byte column k / 2 (a multiple of 32)
          tma_load_2d(sA, &p.tmA, bar, a_k / 2, a_row);
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)
            tma_load_2d(sB + h * (128 * BKB), &p.tmB, bar, b_k / 2, b_row + 128 * h);
          // the four 64-value scale slabs of each operand in one copy each (A's 128 rows,
          // B's BN rows; slab s lands at s x rows x 4 bytes)
          tma_load_2d(sf, &p.tmSFA, bar, a_row, a_k / MMA_K);
          tma_load_2d(sf + 4 * SFA_SLAB, &p.tmSFB, bar, b_row, b_k / MMA_K);
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
      int sf_use[2] = {0, 0};  // dGLU: half k-blocks whose scales have gone through buffer h
      bool issued_any = false;
      for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x) {
        TileInfo t;
        decode_tile<BN, KG>(tile, p, c, MT, NT, t);
        if (t.nkb == 0) continue;
        const int acc = acc_i % NACC;
        const uint32_t acc_phase = (acc_i / NACC) & 1;
        // the accumulator is free once every epilogue warp has finished with its last tile
        if (!mbar_wait(&c.tempty[acc], acc_phase ^ 1, abort, p.err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!mbar_wait(&c.full[stage], phase, abort, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + stage * L::STAGE_BYTES);
          const uint32_t sB = sA + A_BYTES;
          const uint32_t sf = smem_u32(smem + L::SF_OFF + stage * L::SF_STAGE);
          const int rem = t.klen - kb * BK;
          const int nsub = rem >= BK ? BK / MMA_K : (rem + MMA_K - 1) / MMA_K;
          if constexpr (EPI == EPI_DGLU) {
            for (int h = 0; h < 2 && 2 * h < nsub; ++h) {
              // buffer h is free once the MMAs of its previous half k-block have completed
              // (the tensor pipe gets there while the other half's MMAs keep it busy)
              if (sf_use[h] > 0 && !mbar_wait(&c.sfh[h], (uint32_t)(sf_use[h] - 1) & 1u, abort,
                                              p.err)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t hb = tmem_base + L::SF_COL0 + L::SF_HALF * h;
              const int s_end = nsub < 2 * h + 2 ? nsub : 2 * h + 2;
              for (int s = 2 * h; s < s_end; ++s) {
                const uint32_t col = hb + (s - 2 * h) * L::SF_COLS_MMA;
                tmem_cp_32x128b_warpx4(col, smem_desc_noswizzle(sf + s * SFA_SLAB, 0, 128));
#pragma unroll
                for (int hh = 0; hh < BN / 128; ++hh)
                  tmem_cp_32x128b_warpx4(
                      col + 4 + 4 * hh,
                      smem_desc_noswizzle(sf + 4 * SFA_SLAB + s * L::SFB_SLAB + 512 * hh, 0, 128));
              }
              for (int s = 2 * h; s < s_end; ++s) {
                const uint32_t col = hb + (s - 2 * h) * L::SF_COLS_MMA;
                mma_nvf4_ss(d_tmem, smem_desc_sw128(sA + s * (MMA_K / 2), 16, 1024),
                            smem_desc_sw128(sB + s * (MMA_K / 2), 16, 1024), IDESC, col, col + 4,
                            (kb | s) != 0 ? 1u : 0u);
              }
              issued_any = true;
              mma_commit(&c.sfh[h]);
              ++sf_use[h];
            }
            if (!ok) break;
            mma_commit(&c.empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          const uint32_t sft = tmem_base + L::SF_COL0 + stage * L::SF_COLS_STAGE;
          for (int s = 0; s < nsub; ++s) {
            const uint32_t col = sft + s * L::SF_COLS_MMA;
            tmem_cp_32x128b_warpx4(col, smem_desc_noswizzle(sf + s * SFA_SLAB, 0, 128));
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              tmem_cp_32x128b_warpx4(
                  col + 4 + 4 * h,
                  smem_desc_noswizzle(sf + 4 * SFA_SLAB + s * L::SFB_SLAB + 512 * h, 0, 128));
          }
          for (int s = 0; s < nsub; ++s) {
            const uint32_t col = sft + s * L::SF_COLS_MMA;
            mma_nvf4_ss(d_tmem, smem_desc_sw128(sA + s * (MMA_K / 2), 16, 1024),
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
        mma_commit(&c.tfull[acc]);
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
    // ------------------------------------------------------------ epilogue warps 2..
    // Control flow stays warp-uniform (the shared-memory transposes are warp-wide).
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;  // STORE and GLU: which 128 (BN / 2) columns
    const int ws = (warp - 2) >> 2;    // dGLU: this warp's slot among its quadrant's EWQ
    const uint32_t zq = smem_u32(smem + L::ZQ_OFF + (warp - 2) * ZQ_WARP);
    const uint8_t* zq_ptr = smem + L::ZQ_OFF + (warp - 2) * ZQ_WARP;
    uint32_t* xt = reinterpret_cast<uint32_t*>(smem + L::XT_OFF + (warp - 2) * XT_WARP);
    const float alpha =
        __frcp_rn(__fmul_rn(nvfp4_encode_scale(*p.amax_a), nvfp4_encode_scale(*p.amax_b)));
    float m_out = 0.f, m_rht = 0.f;
    int acc_i = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      if (__shfl_sync(0xFFFFFFFFu, *abort, 0)) break;
      TileInfo t;
      decode_tile<BN, KG>(tile, p, c, MT, NT, t);
      const int row0 = t.m0 + q * 32;
      const int row = row0 + lane;
      const bool row_ok = row < t.row_end;
      if (t.nkb == 0) {
        if (row_ok) {
          const int cb = half * (BN / 2);
          uint16_t* o = static_cast<uint16_t*>(p.out) + (int64_t)t.e * p.out_estride +
                        (int64_t)row * p.ldo;
          for (int cc = cb; cc < cb + BN / 2 && t.n0 + cc < p.N; cc += 32)
            store_zero_bf16x32(o + t.n0 + cc);
        }
        continue;
      }
      const float prob = EPI == EPI_STORE ? 0.f : p.row_prob[row];
      if constexpr (EPI == EPI_DGLU) {
        // the first step's saved Z comes in while the MMAs run
        const int f0 = t.n0 + 16 * ws;
        if (f0 < p.N)
          zq_issue(zq, p.z + (int64_t)row * p.ldz + (kGated ? gate_col(f0) : f0), kGated, lane);
      }
      const int acc = acc_i % NACC;
      const uint32_t acc_phase = (acc_i / NACC) & 1;
      const bool got = mbar_wait(&c.tfull[acc], acc_phase, abort, p.err);
      if (!__all_sync(0xFFFFFFFFu, got)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      if constexpr (EPI == EPI_STORE) {
        // drain 128 columns as packed bf16 and release the accumulator at once
        const int cb = half * 128;
        uint32_t pk[64];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tacc + cb + 32 * j, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[16 * j + i] = pack_bf16x2(alpha * __uint_as_float(r[2 * i]),
                                         alpha * __uint_as_float(r[2 * i + 1]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.tempty[acc]);
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
      } else if constexpr (EPI == EPI_GLU) {
        // drain the 128 columns as fp32 (the activation is computed from the fp32
        // accumulator), free TMEM, then work from registers. Row-grouped segments are 128-row
        // aligned: every row of the tile is in its segment.
        const int cb = half * 128;
        float acc_r[128];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tacc + cb + 32 * j, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) acc_r[32 * j + i] = alpha * __uint_as_float(r[i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.tempty[acc]);
        ++acc_i;
        if constexpr (EXT) {
          // the bias joins Z before the activation (and is part of the saved Z); packed
          // column n0 + cb + c has logical column (block / 2) ILV + c % ILV (+ F if linear)
          if (p.fc1_bias) {
            const float* b = p.fc1_bias + (int64_t)t.e * p.N1;
#pragma unroll
            for (int c = 0; c < 128; ++c) {
              const int pc = t.n0 + cb + c;
              const int blk = pc / ILV;
              const int lc = (blk >> 1) * ILV + pc % ILV + ((blk & 1) ? p.F : 0);
              if (pc < p.N) acc_r[c] += b[lc];
            }
          }
        }
        uint16_t* zout = static_cast<uint16_t*>(p.out) + (int64_t)row * p.ldo + t.n0 + cb;
        if (p.out) {  // the saved Z (bf16); absent when the backward recomputes it
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (t.n0 + cb + 32 * j < p.N) store_bf16x32_v8(zout + 32 * j, &acc_r[32 * j]);
        }
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
              a = act_fwd_k<KIND>(p.act, acc_r[g_off + i], acc_r[g_off + ILV + i]);
            } else {
              const float rr = fmaxf(acc_r[g_off + i], 0.f);
              a = rr * rr;
            }
            if constexpr (EXT) {
              if (p.fscale) a *= p.fscale[(int64_t)t.e * p.F + acol + i];
            }
            v[i] = bf16_lo(pack_bf16x2(prob * a, 0.f));
          }
          store_bf16x32_v8(aout + acol, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            m_out = fmaxf(m_out, fabsf(v[i]));
            m_rht = fmaxf(m_rht, fabsf(rht16_lanes(v[i], p.rht_mask, lane)));
          }
        }
      } else {  // EPI_DGLU: accumulator = dA_s over F columns; chunks ws, ws + EWQ, ...
        const uint16_t* zrow = p.z + (int64_t)row * p.ldz;
        uint16_t* dzrow = static_cast<uint16_t*>(p.out) + (int64_t)row * p.ldo;
        float dp = 0.f;
        constexpr int EWQ = L::EWQ;
        // this warp's 16-column chunks of dA_s, scaled and rounded to bf16, into the packed
        // copy (8 columns a chunk); then the accumulator is free for the next tile's MMAs
        const uint32_t tpk = tmem_base + ((uint32_t)(q * 32) << 16) + L::PACK_COL;
#pragma unroll 1
        for (int j = ws; j < BN / 16; j += EWQ) {
          if (t.n0 + 16 * j >= p.N) break;
          uint32_t r[16];
          tmem_ld_32x32b_x16(tacc + 16 * j, r);
          tmem_ld_wait();
          uint32_t w8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            w8[i] = pack_bf16x2(alpha * __uint_as_float(r[2 * i]),
                                alpha * __uint_as_float(r[2 * i + 1]));
          tmem_st_32x32b_x8(tpk + 8 * j, w8);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.tempty[acc]);
        ++acc_i;
#pragma unroll 1
        for (int j = ws, step = 0; j < BN / 16; j += EWQ, ++step) {
          const int f0 = t.n0 + 16 * j;
          if (f0 >= p.N) break;
          const int gc = kGated ? gate_col(f0) : f0;
          // next step's Z into the other buffer (this lane finished reading it in the previous
          // step), then wait for this step's
          const int fn = f0 + 16 * EWQ;
          const bool more = j + EWQ < BN / 16 && fn < p.N;
          if (more) {
            zq_issue(zq + ((step + 1) & 1) * ZQ_BUF, zrow + (kGated ? gate_col(fn) : fn), kGated,
                     lane);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
          } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
          }
          uint32_t dr[8];  // dA_s of the chunk as bf16 pairs
          tmem_ld_32x32b_x8(tpk + 8 * j, dr);
          uint32_t gw[8], lw[8];
          {
            const uint8_t* b = zq_ptr + (step & 1) * ZQ_BUF;
            const uint4 g0 = *reinterpret_cast<const uint4*>(b + zq_slot(lane, 0));
            const uint4 g1 = *reinterpret_cast<const uint4*>(b + zq_slot(lane, 1));
            gw[0] = g0.x; gw[1] = g0.y; gw[2] = g0.z; gw[3] = g0.w;
            gw[4] = g1.x; gw[5] = g1.y; gw[6] = g1.z; gw[7] = g1.w;
            if constexpr (kGated) {
              const uint4 l0 = *reinterpret_cast<const uint4*>(b + zq_slot(lane, 2));
              const uint4 l1 = *reinterpret_cast<const uint4*>(b + zq_slot(lane, 3));
              lw[0] = l0.x; lw[1] = l0.y; lw[2] = l0.z; lw[3] = l0.w;
              lw[4] = l1.x; lw[5] = l1.y; lw[6] = l1.z; lw[7] = l1.w;
            }
          }
          tmem_ld_wait();
          uint32_t w[16];  // dG pairs in w[0..7], dL pairs in w[8..15]
          // extras: this row's dG, dL and p * dA_s * a for the column sums
          float xg[EXT ? 16 : 1], xl[EXT ? 16 : 1], xs[EXT ? 16 : 1];
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            float dg[2], dl[2] = {0.f, 0.f};
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const float d = u ? bf16_hi(dr[i >> 1]) : bf16_lo(dr[i >> 1]);
              const float g = u ? bf16_hi(gw[i >> 1]) : bf16_lo(gw[i >> 1]);
              if constexpr (EXT) {
                // the feature scale s enters as dA = p * s * dA_s and d_prob += dA_s * s * a
                const float l = u ? bf16_hi(lw[i >> 1]) : bf16_lo(lw[i >> 1]);
                const float sc = p.fscale ? p.fscale[(int64_t)t.e * p.F + f0 + i + u] : 1.f;
                const float a = act_bwd_k<KIND>(p.act, g, l, prob * sc * d, dg[u], dl[u]);
                dp += d * sc * a;
                xg[i + u] = dg[u];
                xl[i + u] = dl[u];
                xs[i + u] = prob * d * a;
              } else if constexpr (kGated) {
                const float l = u ? bf16_hi(lw[i >> 1]) : bf16_lo(lw[i >> 1]);
                dp += d * act_bwd_k<KIND>(p.act, g, l, prob * d, dg[u], dl[u]);
              } else {
                const float rr = fmaxf(g, 0.f);
                dp += d * rr * rr;
                dg[u] = prob * d * 2.f * rr;
              }
            }
            w[i >> 1] = pack_bf16x2(dg[0], dg[1]);
            w[8 + (i >> 1)] = pack_bf16x2(dl[0], dl[1]);
          }
#pragma unroll
          for (int i = 0; i < 16; ++i)
            m_out = fmaxf(m_out, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
          st_global_v8(dzrow + gc, w);
          if constexpr (EXT) {
            // column sums over the warp's 32 rows (one expert's: segments are 128-row
            // aligned) into the row group's partials: gate column f at f, linear at F + f,
            // scale at N1 + f
            float* part = p.ext_part + (int64_t)(row0 >> 5) * (p.N1 + p.F);
            const float sg = warp_colsum16(xg, lane);
            const float sl = warp_colsum16(xl, lane);
            const float ss = warp_colsum16(xs, lane);
            if (lane < 16) {
              part[f0 + lane] = sg;
              part[p.F + f0 + lane] = sl;
              part[p.N1 + f0 + lane] = ss;
            }
          }
          if constexpr (kGated) {
            st_global_v8(dzrow + gc + ILV, w + 8);
            m_rht = fmaxf(m_rht, rht_amax_tile32(xt, w, p.rht_mask, lane));
          } else {
            // sReLU: no linear half; rotate the 16 dG columns (the other 16 are zero)
            uint32_t w2[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) w2[i] = i < 8 ? w[i] : 0u;
            m_rht = fmaxf(m_rht, rht_amax_tile32(xt, w2, p.rht_mask, lane));
          }
        }
        p.dprob_part[(int64_t)row * p.nparts + (t.n0 / BN) * EWQ + ws] = dp;
      }
    }
    if constexpr (EPI == EPI_DGLU) asm volatile("cp.async.wait_all;" ::: "memory");
    if constexpr (EPI != EPI_STORE) {
      amax_flush_warp(m_out, p.amax_out);
      amax_flush_warp(m_rht, p.amax_out_rht);
    }
  }

  griddep_launch_dependents();  // this CTA's tiles are done
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// The E4M3 scales of a K-major NVFP4 operand: slab g (64 values of K) holds 4 bytes a row for
// s_pad rows, slabs back to back. As a 2-D tensor of 32-bit words [slabs, s_pad], boxes of
// box_rows words x 4 slabs: one copy brings the four slabs of a 256-value k-block, in the
// same order in shared memory. Slabs past the operand's K read as zeros.
bool tmap_fp4_sf(CUtensorMap* m, const MxOperand& t, uint32_t box_rows) {
  uint64_t dims[2] = {(uint64_t)t.s_pad, (uint64_t)((t.cols + 63) / 64)};
  uint64_t strides[1] = {(uint64_t)t.s_pad * 4};
  uint32_t box[2] = {box_rows, 4};
  return make_tmap(m, t.s, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT32,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
}

// K-major NVFP4 operand: packed codes [rows, cols / 2] bytes, boxes of 128 rows x 128 bytes.
bool tmap_fp4(CUtensorMap* m, const MxOperand& t) {
  uint64_t dims[2] = {(uint64_t)(t.cols / 2), (uint64_t)t.rows};
  uint64_t strides[1] = {(uint64_t)(t.cols / 2)};
  uint32_t box[2] = {128, 128};
  return make_tmap(m, t.q, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

template <int EPI, int KIND, bool KG, bool EXT = false>
cudaError_t launch_fp4(const Fp4Args& a, int grid, cudaStream_t s, int kid) {
  auto kern = grouped_gemm_fp4_kernel<EPI, KIND, KG, EXT>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), Fp4Cfg<EPI>::TOTAL);
  if (e != cudaSuccess) return e;
  launch_kernel(kern, grid, Fp4Cfg<EPI>::THREADS, Fp4Cfg<EPI>::TOTAL, s, nullptr, 0, a);
  count_launch(s, kid);
  return cudaGetLastError();
}

template <int EPI>
cudaError_t launch_act_family(const Fp4Args& a, int kind, int grid, cudaStream_t s, int kid) {
  if (a.fc1_bias || a.fscale || a.ext_part) {  // extras: gated activations only
    switch (kind) {
      case MOE_ACT_SWIGLU: return launch_fp4<EPI, MOE_ACT_SWIGLU, false, true>(a, grid, s, kid);
      case MOE_ACT_CLAMPED_SWIGLU:
        return launch_fp4<EPI, MOE_ACT_CLAMPED_SWIGLU, false, true>(a, grid, s, kid);
      case MOE_ACT_GEGLU: return launch_fp4<EPI, MOE_ACT_GEGLU, false, true>(a, grid, s, kid);
      default: return cudaErrorInvalidValue;
    }
  }
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

int dprob_parts_fp4(int F) {
  using L = Fp4Cfg<EPI_DGLU>;
  return L::EWQ * ((F + L::BN - 1) / L::BN);
}

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
  a.F = p.F;
  a.N1 = p.N1;
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
      a.fc1_bias = p.fc1_bias; a.fscale = p.fscale;
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
      a.fscale = p.fscale; a.ext_part = p.ext_part;
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
  constexpr int bn_max = Fp4Cfg<EPI_STORE>::BN, bn_dglu = Fp4Cfg<EPI_DGLU>::BN;
  const uint32_t sfb_rows = p.role == ROLE_FC2_DGRAD ? bn_dglu : bn_max;
  if (!tmap_fp4(&a.tmA, *A) || !tmap_fp4(&a.tmB, *B) || !tmap_fp4_sf(&a.tmSFA, *A, BM) ||
      !tmap_fp4_sf(&a.tmSFB, *B, sfb_rows))
    return cudaErrorInvalidValue;
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
      constexpr int bn = Fp4Cfg<EPI_STORE>::BN;
      const int64_t tiles = (int64_t)p.E * ((a.M + BM - 1) / BM) * ((a.N + bn - 1) / bn);
      grid = (int)std::min<int64_t>(grid, std::max<int64_t>(tiles, 1));
      return launch_fp4<EPI_STORE, 0, true>(a, grid, s, kid);
    }
  }
}


// ----------------------------------------------------------------------------------------
// FC2 dgrad with the FC1 output recomputed (activation recomputation, [NV-blog] "What's
// next"), NVFP4 operands. Per 128-row x 128-column tile of dA_s two block-scaled FP4 GEMMs
// share one loop over H (k-blocks of 256 values, four MMAs of K = 64 each):
//   dA_s[rows, f0..f0+127]      = Q(dY)[rows] . Q_H(W2)[f0..f0+127]^T          (128 x 128)
//   Z[rows, 2f0 .. 2f0+255]     = Q(X)[rows]  . Q_H(W1p)[2f0 .. 2f0+255]^T     (128 x 256)
// (with the interleave of 64, packed W1 rows 2f0 .. 2f0+255 are the gate and linear columns of
// dA_s columns f0 .. f0+127, in blocks of 64; sReLU, not gated: Z[rows, f0..f0+127], 128 x
// 128). Both scaled by 1 / (S_a S_b) of their operands. TMEM: dA_s columns 0-127, Z 128-383
// and, from 384, two scale buffers of 40 columns, one per half k-block (its two MMAs x dY 4,
// W2 4, X 4, W1p 8 columns): a half k-block's copies wait (bounded) until the MMAs that read
// the buffer one k-block earlier have completed, which the tensor pipe reaches while the other
// half's MMAs keep it busy. Two stages of 80 KB operands and 10 KB of scale slabs. The epilogue
// reads dA_s and Z in fp32 from TMEM and writes dZ in BF16 (packed order) with its amax and
// the amax of its 16-row rotation, and the per-row d_prob partial of the tile, as the saved-Z
// dGLU kernel does. One accumulator set; every wait is bounded.
namespace {

constexpr int RC4_BNA = 128;                  // dA_s columns per tile
constexpr int RC4_STAGES = 2;
constexpr int RC4_A = BM * BKB;               // 16 KB: 128 rows x 128 bytes (dY, X)
constexpr int RC4_B1 = RC4_BNA * BKB;         // 16 KB: W2 rows
constexpr int RC4_B2 = 2 * RC4_BNA * BKB;     // 32 KB: W1p rows (gated; sReLU uses 16 KB)
constexpr int RC4_STAGE = RC4_A + RC4_B1 + RC4_A + RC4_B2;
// a stage's scale slabs: four 512-byte slabs each of dY, W2 and X, then W1p's four slabs of
// 256 rows (1 KB each; sReLU: 128 rows, 512 bytes)
constexpr int RC4_SF_W1 = 12 * SFA_SLAB;
constexpr int RC4_SF = RC4_SF_W1 + 4 * 2 * SFA_SLAB;
constexpr int RC4_SF_OFF = RC4_STAGES * RC4_STAGE;
constexpr int RC4_XT_OFF = RC4_SF_OFF + RC4_STAGES * RC4_SF;
constexpr int RC4_CTRL_OFF = RC4_XT_OFF + kEpiWarps * XT_WARP;
constexpr int RC4_TOTAL = RC4_CTRL_OFF + 4096 + 1024;
constexpr int RC4_ZCOL = RC4_BNA;             // first TMEM column of Z
constexpr int RC4_SFCOL = 384;                // first TMEM column of the two scale buffers
constexpr int RC4_SFH = 40;                   // columns of one buffer (half a k-block)
static_assert(RC4_TOTAL <= 232448, "shared memory");
static_assert(RC4_ZCOL + 2 * RC4_BNA <= RC4_SFCOL && RC4_SFCOL + 2 * RC4_SFH <= kTmemCols,
              "TMEM map");
static_assert(RC4_STAGE % 1024 == 0 && RC4_A % 1024 == 0 && RC4_B1 % 1024 == 0, "alignment");

struct Rc4Args {
  CUtensorMap tmDy;  // dY row-wise copy [R_cap, H/2 bytes], box {128 B, 128 rows}
  CUtensorMap tmW2;  // W2 row-wise copy [E*Fp, H/2], box {128 B, 128 rows}
  CUtensorMap tmX;   // X row-wise copy [R_cap, H/2], box {128 B, 128 rows}
  CUtensorMap tmW1;  // W1p row-wise copy [E*N1p, H/2], box {128 B, 256 (gated) / 128 rows}
  // their scales: boxes of 128 rows (W1p: 256 gated) x four slabs
  CUtensorMap tmSdy, tmSw2, tmSx, tmSw1;
  const float *amax_dy, *amax_w2, *amax_x, *amax_w1;
  const int32_t* offsets;
  int E, R_cap, H, F, N1, Fp, N1p;
  const float* row_prob;
  uint16_t* dz;           // [R_cap, N1] bf16, packed columns
  float* dprob_part;
  int nparts;
  float* amax_out;        // amax of dZ
  float* amax_out_rht;    //   and of its 16-row rotation
  uint32_t rht_mask;
  ActDev act;
  int* err;
};

struct Rc4Ctrl {
  uint64_t full[RC4_STAGES];
  uint64_t empty[RC4_STAGES];
  uint64_t sfh[2];  // the MMAs that read scale buffer h have completed
  uint64_t tfull;
  uint64_t tempty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int off[kMaxE + 1];
  int prefix[kMaxE + 1];
};
static_assert(sizeof(Rc4Ctrl) <= 4096, "control block");

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    fc2_dgrad_recompute_fp4_kernel(const __grid_constant__ Rc4Args p) {
  MOE_GRIDDEP_ENTRY();
  constexpr bool kGated = KIND != MOE_ACT_SRELU;
  constexpr int ZN = kGated ? 2 * RC4_BNA : RC4_BNA;        // Z columns per tile
  constexpr int kW1Slab = kGated ? 2 * SFA_SLAB : SFA_SLAB;   // W1p scale slab bytes
  constexpr uint32_t kStageTx = RC4_STAGE - (kGated ? 0 : RC4_B2 / 2) + RC4_SF_W1 + 4 * kW1Slab;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  Rc4Ctrl& c = *reinterpret_cast<Rc4Ctrl*>(smem + RC4_CTRL_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &c.abort;
  const int NT = (p.F + RC4_BNA - 1) / RC4_BNA;
  const int nkb = (p.H + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RC4_STAGES; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], 1);
    }
    mbar_init(&c.tfull, 1);
    mbar_init(&c.tempty, kEpiWarps);
    mbar_init(&c.drain, 1);
    mbar_init(&c.sfh[0], 1);
    mbar_init(&c.sfh[1], 1);
    fence_mbar_init();
    c.abort = 0;
    bool ok = p.E >= 1 && p.E <= kMaxE;
    int prev = 0;
    for (int e = 0; ok && e <= p.E; ++e) {
      const int o = p.offsets[e];
      if (o < prev || o > p.R_cap || (o & (BM - 1)) || (e == 0 && o != 0)) ok = false;
      c.off[e] = o;
      prev = o;
    }
    int total = 0;
    if (ok) {
      for (int e = 0; e < p.E; ++e) {
        c.prefix[e] = total;
        total += ((c.off[e + 1] - c.off[e]) / BM) * NT;
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
    tma_prefetch_desc(&p.tmSdy);
    tma_prefetch_desc(&p.tmSw2);
    tma_prefetch_desc(&p.tmSx);
    tma_prefetch_desc(&p.tmSw1);
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
  // tile -> expert, first row, first dA_s column (m fastest within an expert)
  auto decode = [&](int tile, int& e, int& m0, int& n0) {
    int lo = 0, hi = p.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (c.prefix[mid] <= tile) lo = mid; else hi = mid;
    }
    const int local = tile - c.prefix[lo];
    const int mt = (c.off[lo + 1] - c.off[lo]) / BM;
    e = lo;
    m0 = c.off[lo] + (local % mt) * BM;
    n0 = (local / mt) * RC4_BNA;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int armed[RC4_STAGES];
#pragma unroll
      for (int s = 0; s < RC4_STAGES; ++s) armed[s] = -1;
      for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x) {
        int e, m0, n0;
        decode(tile, e, m0, n0);
        // weight blocks start on 128-row scale slabs (Fp, N1p and n0 are multiples of 128)
        const int w2_row = e * p.Fp + n0, w1_row = e * p.N1p + (kGated ? 2 * n0 : n0);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&c.empty[stage], phase ^ 1, abort, p.err)) break;
          uint8_t* s0 = smem + stage * RC4_STAGE;
          uint8_t* sf = smem + RC4_SF_OFF + stage * RC4_SF;
          uint64_t* bar = &c.full[stage];
          mbar_arrive_expect_tx(bar, kStageTx);
#pragma unroll
          for (int s = 0; s < RC4_STAGES; ++s)
            if (s == stage) armed[s] = (int)phase;
          const int k0 = kb * BK;  // values; boxes start at byte column k0 / 2
          tma_load_2d(s0, &p.tmDy, bar, k0 / 2, m0);
          tma_load_2d(s0 + RC4_A, &p.tmW2, bar, k0 / 2, w2_row);
          tma_load_2d(s0 + RC4_A + RC4_B1, &p.tmX, bar, k0 / 2, m0);
          tma_load_2d(s0 + 2 * RC4_A + RC4_B1, &p.tmW1, bar, k0 / 2, w1_row);
          // the four 64-value scale slabs of each operand, one copy each
          const int kg = k0 / MMA_K;
          tma_load_2d(sf, &p.tmSdy, bar, m0, kg);
          tma_load_2d(sf + 4 * SFA_SLAB, &p.tmSw2, bar, w2_row, kg);
          tma_load_2d(sf + 8 * SFA_SLAB, &p.tmSx, bar, m0, kg);
          tma_load_2d(sf + RC4_SF_W1, &p.tmSw1, bar, w1_row, kg);
          if (++stage == RC4_STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
#pragma unroll
      for (int s = 0; s < RC4_STAGES; ++s) {
        if (armed[s] >= 0) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(smem_u32(&c.full[s]), (uint32_t)armed[s]) &&
                 globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ scale copies + MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDA = idesc_nvf4(BM, RC4_BNA);
      constexpr uint32_t IDZ = idesc_nvf4(BM, ZN);
      int stage = 0;
      uint32_t phase = 0;
      int acc_i = 0;
      int sf_use[2] = {0, 0};  // half k-blocks whose scales have gone through buffer h
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
          const uint32_t sA1 = smem_u32(smem + stage * RC4_STAGE);
          const uint32_t sB1 = sA1 + RC4_A, sA2 = sB1 + RC4_B1, sB2 = sA2 + RC4_A;
          const uint32_t sf = smem_u32(smem + RC4_SF_OFF + stage * RC4_SF);
          const int rem = p.H - kb * BK;
          const int nsub = rem >= BK ? BK / MMA_K : (rem + MMA_K - 1) / MMA_K;
          for (int h = 0; h < 2 && 2 * h < nsub; ++h) {
            // buffer h is free once the MMAs of the previous half k-block that used it are done
            if (sf_use[h] > 0 && !mbar_wait(&c.sfh[h], (uint32_t)(sf_use[h] - 1) & 1u, abort,
                                            p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t hb = tmem_base + RC4_SFCOL + RC4_SFH * h;
            const int s_end = nsub < 2 * h + 2 ? nsub : 2 * h + 2;
            for (int s = 2 * h; s < s_end; ++s) {
              const uint32_t col = hb + 20 * (s - 2 * h);
              tmem_cp_32x128b_warpx4(col, smem_desc_noswizzle(sf + s * SFA_SLAB, 0, 128));
              tmem_cp_32x128b_warpx4(col + 4,
                                     smem_desc_noswizzle(sf + (4 + s) * SFA_SLAB, 0, 128));
              tmem_cp_32x128b_warpx4(col + 8,
                                     smem_desc_noswizzle(sf + (8 + s) * SFA_SLAB, 0, 128));
              tmem_cp_32x128b_warpx4(col + 12,
                                     smem_desc_noswizzle(sf + RC4_SF_W1 + s * kW1Slab, 0, 128));
              if constexpr (kGated)  // W1p rows 128-255 of the tile
                tmem_cp_32x128b_warpx4(
                    col + 16, smem_desc_noswizzle(sf + RC4_SF_W1 + s * kW1Slab + SFA_SLAB, 0, 128));
            }
            for (int s = 2 * h; s < s_end; ++s) {
              const uint32_t col = hb + 20 * (s - 2 * h);
              const uint32_t acc = (kb | s) != 0 ? 1u : 0u;
              mma_nvf4_ss(tmem_base, smem_desc_sw128(sA1 + s * (MMA_K / 2), 16, 1024),
                          smem_desc_sw128(sB1 + s * (MMA_K / 2), 16, 1024), IDA, col, col + 4,
                          acc);
              mma_nvf4_ss(tmem_base + RC4_ZCOL, smem_desc_sw128(sA2 + s * (MMA_K / 2), 16, 1024),
                          smem_desc_sw128(sB2 + s * (MMA_K / 2), 16, 1024), IDZ, col + 8,
                          col + 12, acc);
            }
            issued_any = true;
            mma_commit(&c.sfh[h]);
            ++sf_use[h];
          }
          if (!ok) break;
          mma_commit(&c.empty[stage]);
          if (++stage == RC4_STAGES) {
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
    uint32_t* xt = reinterpret_cast<uint32_t*>(smem + RC4_XT_OFF + (warp - 2) * XT_WARP);
    const float alpha_a =
        __frcp_rn(__fmul_rn(nvfp4_encode_scale(*p.amax_dy), nvfp4_encode_scale(*p.amax_w2)));
    const float alpha_z =
        __frcp_rn(__fmul_rn(nvfp4_encode_scale(*p.amax_x), nvfp4_encode_scale(*p.amax_w1)));
    float m_out = 0.f, m_rht = 0.f;
    int acc_i = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      if (__shfl_sync(0xFFFFFFFFu, *abort, 0)) break;
      int e, m0, n0;
      decode(tile, e, m0, n0);
      const int row = m0 + q * 32 + lane;
      const float prob = p.row_prob[row];  // segments are 128-row aligned: every row is inside
      const bool got = mbar_wait(&c.tfull, acc_i & 1, abort, p.err);
      if (!__all_sync(0xFFFFFFFFu, got)) break;
      tc_fence_after();
      const uint32_t tl = tmem_base + ((uint32_t)(q * 32) << 16);
      uint16_t* dzrow = p.dz + (int64_t)row * p.N1;
      float dp = 0.f;
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        const int cc = half * 64 + 16 * j;  // dA_s column within the tile
        const int f0 = n0 + cc;
        if (f0 >= p.F) break;
        // gated: Z holds the packed W1p rows, blocks of 64 gate then 64 linear columns
        const int zc = kGated ? ((cc & ~63) << 1) + (cc & 63) : cc;
        uint32_t da[16], gz[16], lz[16];
        tmem_ld_32x32b_x16(tl + cc, da);
        tmem_ld_32x32b_x16(tl + RC4_ZCOL + zc, gz);
        if constexpr (kGated) tmem_ld_32x32b_x16(tl + RC4_ZCOL + zc + 64, lz);
        tmem_ld_wait();
        uint32_t w[16];  // dG pairs in w[0..7], dL pairs in w[8..15]
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          float dg[2], dl[2] = {0.f, 0.f};
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const float d = alpha_a * __uint_as_float(da[i + u]);
            const float g = alpha_z * __uint_as_float(gz[i + u]);
            if constexpr (kGated) {
              const float l = alpha_z * __uint_as_float(lz[i + u]);
              dp += d * act_bwd_k<KIND>(p.act, g, l, prob * d, dg[u], dl[u]);
            } else {
              const float rr = fmaxf(g, 0.f);
              dp += d * rr * rr;
              dg[u] = prob * d * 2.f * rr;
            }
          }
          w[i >> 1] = pack_bf16x2(dg[0], dg[1]);
          w[8 + (i >> 1)] = pack_bf16x2(dl[0], dl[1]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
          m_out = fmaxf(m_out, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
        const int gc = kGated ? gate_col(f0) : f0;
        st_global_v8(dzrow + gc, w);
        if constexpr (kGated) {
          st_global_v8(dzrow + gc + ILV, w + 8);
          m_rht = fmaxf(m_rht, rht_amax_tile32(xt, w, p.rht_mask, lane));
        } else {
          uint32_t w2[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) w2[i] = i < 8 ? w[i] : 0u;
          m_rht = fmaxf(m_rht, rht_amax_tile32(xt, w2, p.rht_mask, lane));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.tempty);
      ++acc_i;
      p.dprob_part[(int64_t)row * p.nparts + (n0 / RC4_BNA) * 2 + half] = dp;
    }
    amax_flush_warp(m_out, p.amax_out);
    amax_flush_warp(m_rht, p.amax_out_rht);
  }

  griddep_launch_dependents();  // this CTA's tiles are done
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// K-major NVFP4 copy [rows, cols] (cols/2 bytes a row) as TMA boxes of 128 bytes x box_rows
bool tmap_fp4_rows(CUtensorMap* m, const MxOperand& t, uint32_t box_rows) {
  uint64_t dims[2] = {(uint64_t)(t.cols / 2), (uint64_t)t.rows};
  uint64_t strides[1] = {(uint64_t)(t.cols / 2)};
  uint32_t box[2] = {128, box_rows};
  return make_tmap(m, t.q, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

template <int KIND>
cudaError_t launch_rc_fp4(const Rc4Args& a, int grid, cudaStream_t s) {
  auto kern = fc2_dgrad_recompute_fp4_kernel<KIND>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), RC4_TOTAL);
  if (e != cudaSuccess) return e;
  launch_kernel(kern, grid, kThreads, RC4_TOTAL, s, nullptr, 0, a);
  count_launch(s, MOE_K_GEMM_FC2_DGRAD);
  return cudaGetLastError();
}

}  // namespace

int dprob_parts_fp4_recompute(int F) { return 2 * ((F + RC4_BNA - 1) / RC4_BNA); }

cudaError_t launch_fc2_dgrad_recompute_fp4(const Fp4Problem& p, cudaStream_t s) {
  if (p.gated && p.ilv != ILV) return cudaErrorInvalidValue;
  if (p.gated != (p.act.kind != MOE_ACT_SRELU)) return cudaErrorInvalidValue;
  Rc4Args a;
  memset(&a, 0, sizeof(a));
  if (!tmap_fp4_rows(&a.tmDy, p.dy, BM) || !tmap_fp4_rows(&a.tmW2, p.w2, RC4_BNA) ||
      !tmap_fp4_rows(&a.tmX, p.x, BM) ||
      !tmap_fp4_rows(&a.tmW1, p.w1, p.gated ? 2 * RC4_BNA : RC4_BNA))
    return cudaErrorInvalidValue;
  if (!tmap_fp4_sf(&a.tmSdy, p.dy, BM) || !tmap_fp4_sf(&a.tmSw2, p.w2, RC4_BNA) ||
      !tmap_fp4_sf(&a.tmSx, p.x, BM) ||
      !tmap_fp4_sf(&a.tmSw1, p.w1, p.gated ? 2 * RC4_BNA : RC4_BNA))
    return cudaErrorInvalidValue;
  a.amax_dy = p.amax + AM_DY; a.amax_w2 = p.amax + AM_W2;
  a.amax_x = p.amax + AM_X; a.amax_w1 = p.amax + AM_W1;
  a.offsets = p.offsets;
  a.E = p.E;
  a.R_cap = (int)p.R_cap;
  a.H = p.H;
  a.F = p.F;
  a.N1 = p.N1;
  a.Fp = p.Fp;
  a.N1p = p.N1p;
  a.row_prob = p.row_prob;
  a.dz = static_cast<uint16_t*>(p.out);
  a.dprob_part = p.dprob_part;
  a.nparts = dprob_parts_fp4_recompute(p.F);
  a.amax_out = p.amax + AM_DZ;
  a.amax_out_rht = p.amax + AM_DZT;
  a.rht_mask = p.rht_mask;
  a.act = p.act;
  a.err = p.err;
  const int grid = std::max(1, p.num_ctas);
  switch (p.act.kind) {
    case MOE_ACT_SWIGLU: return launch_rc_fp4<MOE_ACT_SWIGLU>(a, grid, s);
    case MOE_ACT_CLAMPED_SWIGLU: return launch_rc_fp4<MOE_ACT_CLAMPED_SWIGLU>(a, grid, s);
    case MOE_ACT_GEGLU: return launch_rc_fp4<MOE_ACT_GEGLU>(a, grid, s);
    case MOE_ACT_SRELU: return launch_rc_fp4<MOE_ACT_SRELU>(a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
