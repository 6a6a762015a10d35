// Persistent block-scaled (MXFP8) grouped GEMM for sm_103a.
//
// [NV-blog] kernel families in the MXFP8 recipe: (1) GroupGemm + quantise, (2) FC1 +
// activation + quantise/transpose, (3) FC2 dgrad + dActivation + quantise/transpose; [TE-MoE]
// Challenge 2 (MXFP8: E4M3 with one E8M0 scale per 32 values, tensor-core accelerated).
//
// Every operand is an E4M3 matrix quantised along its own reduction dimension. A row-wise copy
// ([rows, K] row-major) is read K-major; a column-wise copy keeps its source's row-major
// layout ([K, rows]) and is read MN-major, so no copy is ever transposed in memory. Scales sit
// in the MMA slab layout (sf_mma_offset). A CTA:
//   warp 0   TMA of the A (128 x 128 B) and B (256 x 128 B) k-blocks and one 1-D bulk copy of
//            their 512 + 1024 bytes of scale slabs, all counted on one mbarrier,
//   warp 1   TMEM owner; one thread copies the stage's scales into TMEM (tcgen05.cp) and issues
//            four tcgen05.mma.kind::mxf8f6f4.block_scale 128x256x32 (scale byte = K step),
//   warps 2-9 epilogue: drain the accumulator into registers (warp w takes TMEM lanes
//            32*(w%4).. and 128 of the 256 columns), release TMEM, then bf16 store, or GLU /
//            dGLU with fused row-wise and column-wise MXFP8 quantisation. Every 32-byte E4M3
//            run and every 64-byte bf16 run leaves in 256-bit stores; the dGLU epilogue stages
//            the saved Z of its next 32 columns in shared memory (cp.async) while it quantises.
// The tile is 128 x 256 because a 128 x 256 x 32 MMA runs at the full fp8 rate while 128-wide
// ones do not; TMEM then holds one accumulator (256 columns) plus 12 scale columns per stage,
// and the register drain lets the next tile's MMAs start while the epilogue works. Expert
// segments are padded to 128 rows so that every tile starts on a scale slab. The activation
// is a template parameter, so each kernel carries the epilogue code of one activation only.
#include "gemm_common.cuh"

namespace moe {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;  // fp8 elements (bytes) per k-block: one 128-byte swizzle row
constexpr int MMA_K = 32;
constexpr int kMaxStages = 6;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
// epilogue warps of the one-CTA dGLU kernel, each lane quadrant's warps dealing the tile's
// eight 32-column chunks round-robin (measured: twelve warps, 128 registers a thread, ran the
// GPT-OSS-shaped dGLU 5% faster and the Mixtral-shaped one 4% slower than eight)
#ifndef MX_DGLU_WARPS
#define MX_DGLU_WARPS 8
#endif
constexpr int kMaxE = 256;
constexpr int kSfCol = BN;  // first TMEM column of the per-stage scale factors
constexpr int kPackCol = 320;  // dGLU: the drained accumulator as packed bf16 (128 columns)
constexpr int kTmemCols = 512;
static_assert(kPackCol + BN / 2 <= kTmemCols, "TMEM map");

enum { EPI_STORE = 0, EPI_GLU = 1, EPI_DGLU = 2 };

struct MxArgs {
  CUtensorMap tmA;
  CUtensorMap tmB;
  // TST kernels: the weight-gradient output [E][M][N] bf16, box 64 x 32 x 1, 128B swizzle
  CUtensorMap tmOut;
  // pair kernels: the scale buffers as [bytes / 16, 16] uint8 tensors, so that a CTA's scale
  // slabs are TMA loads that can complete on the pair leader's barrier
  CUtensorMap tmSFA;
  CUtensorMap tmSFB;
  const uint8_t* sfa;
  int64_t sfa_pad;
  const uint8_t* sfb;
  int64_t sfb_pad;
  const int32_t* offsets;
  int E;
  int R_cap;
  int M, N, K;
  int a_row_e, a_k_e, b_row_e, b_k_e;  // per-expert row / k offsets of A and B
  void* out;                           // bf16 output (STORE) or saved Z (GLU)
  int64_t ldo;
  int64_t out_estride;
  uint8_t* q_row;                      // GLU: a_s, DGLU: dZ, row-wise MXFP8 [R, ld_q_row]
  uint8_t* s_row;
  int64_t ld_q_row;
  int64_t s_row_pad;
  uint8_t* q_col;                      // column-wise MXFP8, natural layout [R, ld_q_col]
  uint8_t* s_col;
  int64_t ld_q_col;
  int64_t s_col_pad;
  const float* row_prob;
  const uint16_t* z;                   // DGLU: saved Z (bf16, packed columns)
  int64_t ldz;
  float* dprob_part;
  int nparts;
  int ilv;                             // gate/linear interleave of the packed columns
  int wide;                            // STORE: out is 32-byte aligned (256-bit stores)
  // epilogue extras (EXT kernels): FC1 bias [E, N1] (logical [gate | linear] order) and
  // feature scale [E, F], fp32, NULL when absent; the dGLU epilogue's per-32-row column sums
  // of dZ (bias gradient) and of p * dA_s * a (scale gradient) go to ext_part
  // [R_cap / 32, N1 + F]
  const float* fc1_bias;
  const float* fscale;
  float* ext_part;
  int F, N1;
  ActDev act;
  int* err;
};

constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int SFA_BYTES = 512;   // 128 rows x 4 k-blocks
constexpr int SFB_BYTES = 1024;  // 256 rows x 4 k-blocks
constexpr int kCtrlBytes = 2560;  // the control block (barriers, expert table), below

// per-warp 32 x 32 bf16 staging tile of the column-wise quantisation: 64-byte rows whose
// four 16-byte pieces are XOR-rotated by (row / 2) % 4, which spreads a warp's row writes over
// all banks without padding; then 32 column factors 2^-e
constexpr int XP_ROW = 64;
constexpr int XPOSE_WARP_BYTES = 32 * XP_ROW + 32 * 4;
MOE_DEVICE int xp_piece(int row, int piece) { return row * XP_ROW + ((piece ^ ((row >> 1) & 3)) << 4); }
constexpr int ZST_WARP_BYTES = 32 * 128;  // dGLU: saved Z of one chunk, 32 rows x 64 bf16
constexpr int TST_WARP_BYTES = 32 * 128;  // TMA-store staging: 32 rows x 64 bf16, 128B swizzle

// Shared-memory map of one kernel: four pipeline stages, except for the dGLU kernel, whose Z
// buffer takes the fourth stage's space. STORE kernels have no quantisation staging tiles.
// PAIR: a CTA of a pair holds half of the B tile (and all of its scale factors), so more
// stages fit: 6 (STORE), 5 (GLU, dGLU).
// TST: the weight-gradient STORE epilogue writes through shared memory and TMA stores (a
// 32 x 64-column bf16 box a warp at a time), which takes one stage's room.
template <int EPI, bool PAIR = false, bool TST = false>
struct MxSmem {
  static constexpr int EW = EPI == 2 && !PAIR ? MX_DGLU_WARPS : kEpiWarps;  // epilogue warps
  static constexpr int EWQ = EW / 4;                                        // per lane quadrant
  static constexpr int THREADS = 64 + 32 * EW;
  static constexpr int STAGES = TST ? 3 : PAIR ? (EPI == 0 ? 6 : 5) : (EPI == 2 ? 3 : 4);
  static constexpr int STAGE_BYTES_ = A_BYTES + (PAIR ? B_BYTES / 2 : B_BYTES);
  static constexpr int DATA = STAGES * STAGE_BYTES_;
  static constexpr int SF_OFF = DATA;
  static constexpr int XPOSE_OFF = SF_OFF + STAGES * (SFA_BYTES + SFB_BYTES);
  static constexpr int ZST_OFF = XPOSE_OFF + (EPI == 0 ? 0 : EW * XPOSE_WARP_BYTES);
  static constexpr int TST_OFF = (ZST_OFF + (EPI == 2 ? EW * ZST_WARP_BYTES : 0) + 1023) / 1024 * 1024;
  static constexpr int CTRL_OFF = TST_OFF + (TST ? EW * TST_WARP_BYTES : 0);
  static constexpr int TOTAL = CTRL_OFF + kCtrlBytes + 1024;
  static_assert(TOTAL <= 232448, "shared memory above the sm_100 per-block limit");
  static_assert(XPOSE_OFF % 16 == 0 && ZST_OFF % 128 == 0 && CTRL_OFF % 8 == 0, "alignment");
  static_assert(STAGES <= kMaxStages, "control barriers");
  static_assert(EWQ * 4 == EW && THREADS <= 1024, "whole lane quadrants");
  // scale columns of every stage below the dGLU's packed accumulator
  static_assert(EPI != 2 || kSfCol + 12 * STAGES <= kPackCol, "TMEM scale columns");
  static_assert(kSfCol + 12 * STAGES <= kTmemCols, "TMEM scale columns");
};

struct Ctrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull;
  uint64_t tempty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int off[kMaxE + 1];
  int prefix[kMaxE + 1];
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");

struct TileInfo {
  int e, m0, n0, kbeg, klen, nkb, row_end;
};

// Tiles are TM rows (128, or 256 for a CTA pair) by BN columns.
template <bool KG, int TM = BM>
MOE_DEVICE void decode_tile(int tile, const MxArgs& p, const Ctrl& c, int MT, int NT, TileInfo& t) {
  if (!KG) {
    int lo = 0, hi = p.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (c.prefix[mid] <= tile) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int local = tile - c.prefix[e];
    const int mt = (c.off[e + 1] - c.off[e] + TM - 1) / TM;
    t.e = e;
    t.m0 = c.off[e] + (local % mt) * TM;
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
    t.m0 = (local / NT) * TM;
    t.n0 = (local % NT) * BN;
    t.kbeg = c.off[e];
    t.klen = c.off[e + 1] - c.off[e];
    t.nkb = (t.klen + BK - 1) / BK;
    t.row_end = p.M;
  }
}

// Row-wise MXFP8 of one 32-column block held by this thread: one 32-byte run and its scale.
MOE_DEVICE void mx_row_block(const float (&v)[32], uint8_t* qdst, uint8_t* sdst) {
  uint32_t w[8];
  *sdst = (uint8_t)mx_quant_block(v, w);
  st_global_v8(qdst, w);
}

// Column-wise MXFP8 of the warp's 32 rows x 32 columns (this lane holds one row), stored in the
// natural row-major layout. A block's exponent depends only on the exponent bits of its
// maximum |v|, and truncating |v| to bf16 keeps those bits (values small enough to lose them
// clamp to e = -127 either way), so the column maxima are taken over a bf16 staging tile:
// lanes j and j + 16 scan column pair j over rows 0-15 and 16-31 with packed 16-bit maxima,
// one shuffle combines them, lane j publishes 2^-e of column 2j + (j >= 16) and writes its
// scale byte; every lane then quantises its own fp32 row with the 32 factors and stores one
// 32-byte run. The tile and the factors are rewritten only after every lane has passed the
// next call's first warp barrier, so two barriers per call suffice.
MOE_DEVICE void mx_col_block(const float (&v)[32], uint8_t* xs, uint8_t* qdst, uint8_t* s_col,
                             int64_t col0, int64_t kb, int64_t s_pad, int lane) {
  float* xinv = reinterpret_cast<float*>(xs + 32 * XP_ROW);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = __byte_perm(__float_as_uint(v[8 * k + 2 * i]), __float_as_uint(v[8 * k + 2 * i + 1]),
                         0x7632) & 0x7FFF7FFFu;
    *reinterpret_cast<uint4*>(xs + xp_piece(lane, k)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __syncwarp();
  const int jp = lane & 15, rh = lane >> 4;
  // column pair jp sits in piece jp / 4 of every row, word jp % 4 of it (rows rh*16 + r share
  // the piece rotation of row r, rh*16 being a multiple of 8)
  const uint8_t* col = xs + rh * 16 * XP_ROW + 4 * (jp & 3);
  uint32_t m0 = 0, m1 = 0;
#pragma unroll
  for (int r = 0; r < 16; r += 2) {
    uint32_t t0, t1;
    asm("max.u16x2 %0, %1, %2;" : "=r"(t0) : "r"(m0), "r"(*reinterpret_cast<const uint32_t*>(col + xp_piece(r, jp >> 2))));
    asm("max.u16x2 %0, %1, %2;" : "=r"(t1) : "r"(m1), "r"(*reinterpret_cast<const uint32_t*>(col + xp_piece(r + 1, jp >> 2))));
    m0 = t0;
    m1 = t1;
  }
  uint32_t m;
  asm("max.u16x2 %0, %1, %2;" : "=r"(m) : "r"(m0), "r"(m1));
  const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, m, 16);
  asm("max.u16x2 %0, %1, %2;" : "=r"(m) : "r"(m), "r"(other));
  const int c = 2 * jp + rh;  // this lane's column of the block
  const int e = mx_block_exponent(__uint_as_float(rh ? (m & 0xFFFF0000u) : (m << 16)));
  s_col[sf_mma_offset(col0 + c, kb, s_pad)] = (uint8_t)(e + 127);
  xinv[c] = mx_inv_scale(e);
  __syncwarp();
  uint32_t w[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float4 f = reinterpret_cast<const float4*>(xinv)[k];
    w[k] = cvt_e4m3x2(v[4 * k] * f.x, v[4 * k + 1] * f.y) |
           (cvt_e4m3x2(v[4 * k + 2] * f.z, v[4 * k + 3] * f.w) << 16);
  }
  st_global_v8(qdst, w);
}

// Gate and linear columns of dA column f in the packed Z layout (blocks of ilv gate columns
// followed by ilv linear columns; ilv a power of two).
MOE_DEVICE int gate_col(int f, int ilv) { return ((f & ~(ilv - 1)) << 1) | (f & (ilv - 1)); }

// A_MN / B_MN: the operand is a column-wise copy stored [K rows, M or N columns] (MN-major);
// otherwise it is [M or N rows, K] (K-major). KIND: the activation of the GLU / dGLU epilogue
// (moe_activation_t; unused by STORE). ILV: the gate/linear interleave of the GLU epilogue.
//
// PAIR: clusters of two CTAs compute 256 x 256 tiles with cta_group::2 block-scaled MMAs. CTA
// rank r loads rows 128r.. of A, rows 128r.. of the B tile (half of it) and the scale factors
// of its A rows and of all 256 B rows (each SM's tensor core needs the B scales in its own
// TMEM); it keeps rows 128r.. of the accumulator. Both CTAs' loads of a stage (operands and
// scale slabs, all TMA) complete on the leader's full barrier, which the leader arms with the
// pair's bytes; the leader (rank 0) then copies the scales into both CTAs' TMEM and issues the
// MMAs; MMA commits reach both CTAs by multicast; the follower's epilogue frees the
// accumulator on the leader's barrier. Expert segments are 128-row aligned, so each CTA's
// half of a tile lies wholly inside or wholly past its segment.
// EXT: the GLU / dGLU epilogues with the FC1 bias and feature-scale extras (a separate
// instantiation, so the plain kernels carry none of its code or registers).
//
// TST (k-grouped STORE only): the weight gradients of experts with few rows are bound by the
// epilogue's stores (per-lane row stores fill the load/store queue), so this variant writes
// each warp's 32 x 64-column bf16 chunk to shared memory (128-byte swizzle, conflict-free) and
// sends it with one TMA store; an expert without rows stores zeros the same way.
template <int EPI, int KIND, bool KG, int ILV, bool A_MN, bool B_MN, bool PAIR = false,
          bool EXT = false, bool TST = false>
__global__ void __launch_bounds__(MxSmem<EPI, PAIR, TST>::THREADS, 1)
    grouped_gemm_mx_kernel(const __grid_constant__ MxArgs p) {
  MOE_GRIDDEP_ENTRY();
  constexpr bool kGated = KIND != MOE_ACT_SRELU;
  static_assert(!TST || (EPI == EPI_STORE && KG && !PAIR), "TMA stores: weight gradients");
  using L = MxSmem<EPI, PAIR, TST>;
  constexpr int STAGES = L::STAGES;
  constexpr int SBYTES = L::STAGE_BYTES_;
  constexpr int TM = PAIR ? 2 * BM : BM;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  Ctrl& c = *reinterpret_cast<Ctrl*>(smem + L::CTRL_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &c.abort;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int tile0 = PAIR ? (int)cluster_id_x() : (int)blockIdx.x;
  const int tstep = PAIR ? (int)nclusters_x() : (int)gridDim.x;
  const int NT = (p.N + BN - 1) / BN;
  const int MT = KG ? (p.M + TM - 1) / TM : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&c.full[s], 1);
      mbar_init(&c.empty[s], 1);
    }
    mbar_init(&c.tfull, 1);
    mbar_init(&c.tempty, PAIR ? 2 * L::EW : L::EW);
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
        total += KG ? MT * NT : ((c.off[e + 1] - c.off[e] + TM - 1) / TM) * NT;
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
      tmem_alloc_pair(&c.tmem_base, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&c.tmem_base, kTmemCols);
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
      for (int tile = tile0; tile < total && !*abort; tile += tstep) {
        TileInfo t;
        decode_tile<KG, TM>(tile, p, c, MT, NT, t);
        const int a_row = t.m0 + BM * (int)rank + t.e * p.a_row_e;  // this CTA's A rows
        const int b_row_sf = t.n0 + t.e * p.b_row_e;                // the tile's B rows
        const int b_row = b_row_sf + (BN / 2) * (int)rank;           // pair: this CTA's half
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!mbar_wait(&c.empty[stage], phase ^ 1, abort, p.err)) break;
          uint8_t* sA = smem + stage * SBYTES;
          uint8_t* sB = sA + A_BYTES;
          uint8_t* sfA = smem + L::SF_OFF + stage * (SFA_BYTES + SFB_BYTES);
          uint64_t* bar = &c.full[stage];
          const uint32_t bar_c = full_leader + stage * (uint32_t)sizeof(uint64_t);
          if (!PAIR) mbar_arrive_expect_tx(bar, SBYTES + SFA_BYTES + SFB_BYTES);
          else if (rank == 0) mbar_arrive_expect_tx(bar, 2 * (SBYTES + SFA_BYTES + SFB_BYTES));
#pragma unroll
          for (int s = 0; s < STAGES; ++s)
            if (s == stage) armed[s] = (int)phase;
          const int k0 = t.kbeg + kb * BK;
          const int a_k = k0 + t.e * p.a_k_e;
          const int b_k = k0 + t.e * p.b_k_e;
          const int64_t sfa_off = ((int64_t)(a_k / BK) * p.sfa_pad + a_row) * 4;
          const int64_t sfb_off = ((int64_t)(b_k / BK) * p.sfb_pad + b_row_sf) * 4;
          // boxes are 128 x 128 bytes: K-major {k, row}, MN-major {mn, k}
          if constexpr (PAIR) {
            if (!A_MN) tma_load_2d_pair(sA, &p.tmA, bar_c, a_k, a_row);
            else tma_load_2d_pair(sA, &p.tmA, bar_c, a_row, a_k);
            if (!B_MN) tma_load_2d_pair(sB, &p.tmB, bar_c, b_k, b_row);
            else tma_load_2d_pair(sB, &p.tmB, bar_c, b_row, b_k);
            // scale slabs start on 512-byte boundaries: rows of 16 bytes
            tma_load_2d_pair(sfA, &p.tmSFA, bar_c, 0, (int)(sfa_off >> 4));
            tma_load_2d_pair(sfA + SFA_BYTES, &p.tmSFB, bar_c, 0, (int)(sfb_off >> 4));
          } else {
            if (!A_MN) tma_load_2d(sA, &p.tmA, bar, a_k, a_row);
            else tma_load_2d(sA, &p.tmA, bar, a_row, a_k);
            if (!B_MN) {
              tma_load_2d(sB, &p.tmB, bar, b_k, b_row);
              tma_load_2d(sB + B_BYTES / 2, &p.tmB, bar, b_k, b_row + 128);
            } else {
              tma_load_2d(sB, &p.tmB, bar, b_row, b_k);
              tma_load_2d(sB + B_BYTES / 2, &p.tmB, bar, b_row + 128, b_k);
            }
            bulk_load(sfA, p.sfa + sfa_off, SFA_BYTES, bar);
            bulk_load(sfA + SFA_BYTES, p.sfb + sfb_off, SFB_BYTES, bar);
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
#pragma unroll
      for (int s = 0; s < STAGES; ++s) {
        if (armed[s] >= 0) {
          const uint32_t bar_s = (PAIR && rank != 0) ? smem_u32(&c.empty[s]) : smem_u32(&c.full[s]);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(bar_s, (uint32_t)armed[s]) && globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1 && PAIR && rank != 0) {
    // pair follower: no MMAs to issue (the leader issues the pair's)
  } else if (warp == 1) {
    // ------------------------------------------------------------ scale copy + MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc_i = 0;
      bool issued_any = false;
      for (int tile = tile0; tile < total && !*abort; tile += tstep) {
        TileInfo t;
        decode_tile<KG, TM>(tile, p, c, MT, NT, t);
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
          const uint32_t sA = smem_u32(smem + stage * SBYTES);
          const uint32_t sB = sA + A_BYTES;
          const uint32_t sfA = smem_u32(smem + L::SF_OFF + stage * (SFA_BYTES + SFB_BYTES));
          const uint32_t sfa_t = tmem_base + kSfCol + stage * 12;
          const uint32_t sfb_t = sfa_t + 4;
          if constexpr (PAIR) {
            tmem_cp_32x128b_warpx4_pair(sfa_t, smem_desc_noswizzle(sfA, 0, 128));
            tmem_cp_32x128b_warpx4_pair(sfb_t, smem_desc_noswizzle(sfA + SFA_BYTES, 0, 128));
            tmem_cp_32x128b_warpx4_pair(sfb_t + 4,
                                        smem_desc_noswizzle(sfA + SFA_BYTES + 512, 0, 128));
          } else {
            tmem_cp_32x128b_warpx4(sfa_t, smem_desc_noswizzle(sfA, 0, 128));
            tmem_cp_32x128b_warpx4(sfb_t, smem_desc_noswizzle(sfA + SFA_BYTES, 0, 128));
            tmem_cp_32x128b_warpx4(sfb_t + 4, smem_desc_noswizzle(sfA + SFA_BYTES + 512, 0, 128));
          }
          const int rem = t.klen - kb * BK;
          const int nsub = rem >= BK ? BK / MMA_K : (rem + MMA_K - 1) / MMA_K;
          for (int ks = 0; ks < nsub; ++ks) {
            // K-major: a K step is 32 bytes along the swizzled row; MN-major: 32 rows of 128
            // bytes, with the 128-element MN chunks of B 16 KB apart (LBO) and 8-row groups
            // 1024 bytes apart (SBO)
            const uint64_t ad = A_MN ? smem_desc_sw128(sA + ks * (MMA_K * 128), A_BYTES, 1024)
                                     : smem_desc_sw128(sA + ks * MMA_K, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(sB + ks * (MMA_K * 128), B_BYTES / 2, 1024)
                                     : smem_desc_sw128(sB + ks * MMA_K, 16, 1024);
            if constexpr (PAIR)
              mma_mxf8_ss_pair(tmem_base, ad, bd, idesc_mxf8(TM, BN, ks, A_MN, B_MN), sfa_t,
                               sfb_t, (kb | ks) != 0 ? 1u : 0u);
            else
              mma_mxf8_ss(tmem_base, ad, bd, idesc_mxf8(BM, BN, ks, A_MN, B_MN), sfa_t, sfb_t,
                          (kb | ks) != 0 ? 1u : 0u);
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
        if constexpr (PAIR) mma_commit_pair_mc(&c.tfull, 0x3);
        else mma_commit(&c.tfull);
        ++acc_i;
      }
      if (issued_any) {
        if constexpr (PAIR) mma_commit_pair_mc(&c.drain, 0x1);
        else mma_commit(&c.drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&c.drain), 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps 2..
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;  // STORE, GLU: columns [128*half, 128*half + 128)
    // dGLU: this warp's slot among its lane quadrant's EWQ warps; it takes the tile's 32-column
    // chunks ws, ws + EWQ, ...
    constexpr int EWQ = L::EWQ;
    const int ws = (warp - 2) >> 2;
    uint8_t* xs = smem + L::XPOSE_OFF + (warp - 2) * XPOSE_WARP_BYTES;
    const uint8_t* zst = smem + L::ZST_OFF + (warp - 2) * ZST_WARP_BYTES;
    const uint32_t zst_a = smem_u32(zst);
    int acc_i = 0;
    // the accumulator is freed on the leader's barrier (a pair's MMAs write both CTAs' TMEM)
    const uint32_t tempty_leader = PAIR ? mapa_shared(smem_u32(&c.tempty), 0) : 0u;
    auto release_acc = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (PAIR) mbar_arrive_cluster(tempty_leader);
        else mbar_arrive(&c.tempty);
      }
    };
    for (int tile = tile0; tile < total; tile += tstep) {
      // every give-up decision is warp-uniform (full-warp TMEM loads, shuffles, __syncwarp)
      if (__shfl_sync(0xFFFFFFFFu, *abort, 0)) break;
      TileInfo t;
      decode_tile<KG, TM>(tile, p, c, MT, NT, t);
      t.m0 += BM * (int)rank;          // this CTA's 128 rows of the tile
      // a pair's second half can lie past the segment (segments are 128-row aligned, so a
      // half is wholly inside or wholly outside): it only frees the accumulator
      const bool half_live = t.m0 < t.row_end;
      const int row0 = t.m0 + q * 32;  // first row of this warp's 32-row block
      const int row = row0 + lane;
      const bool row_ok = row < t.row_end;
      const int cb = half * 128;       // first tile column of this warp
      if constexpr (TST) {
        // 128 columns of the warp's 32 rows as packed bf16 (zeros for an expert without rows)
        uint32_t pk[64];
        if (t.nkb == 0) {
#pragma unroll
          for (int i = 0; i < 64; ++i) pk[i] = 0u;
        } else {
          const bool got = mbar_wait(&c.tfull, acc_i & 1, abort, p.err);
          if (!__all_sync(0xFFFFFFFFu, got)) break;
          tc_fence_after();
          const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + cb;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tacc + 32 * j, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[16 * j + i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
          }
          release_acc();
          ++acc_i;
        }
        // two 32 x 64-column boxes: row `lane` of the box is 128 bytes, its 16-byte piece c at
        // piece c ^ (lane % 8) (the 128-byte swizzle), which keeps the shared stores free of
        // bank conflicts; rows past M and columns past N are clipped by the TMA store
        uint8_t* buf = smem + L::TST_OFF + (warp - 2) * TST_WARP_BYTES;
#pragma unroll
        for (int j2 = 0; j2 < 2; ++j2) {
          const int x = t.n0 + cb + 64 * j2;
          if (x >= p.N) break;
          if (lane == 0) bulk_wait_read0();  // the previous box has left the buffer
          __syncwarp();
#pragma unroll
          for (int cpc = 0; cpc < 8; ++cpc)
            *reinterpret_cast<uint4*>(buf + lane * 128 + ((cpc ^ (lane & 7)) << 4)) =
                make_uint4(pk[32 * j2 + 4 * cpc], pk[32 * j2 + 4 * cpc + 1],
                           pk[32 * j2 + 4 * cpc + 2], pk[32 * j2 + 4 * cpc + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&p.tmOut, buf, x, row0, t.e);
            bulk_commit();
          }
        }
        continue;
      }
      if (t.nkb == 0) {
        if (row_ok) {
          uint16_t* o = static_cast<uint16_t*>(p.out) + (int64_t)t.e * p.out_estride +
                        (int64_t)row * p.ldo;
          for (int cc = cb; cc < cb + 128 && t.n0 + cc < p.N; cc += 32)
            store_zero_bf16x32(o + t.n0 + cc);
        }
        continue;
      }
      const uint16_t* zrow = p.z + (int64_t)row * p.ldz;
      if constexpr (EPI == EPI_DGLU) {
        // the saved Z of the first chunk comes in while the MMAs run
        const int f0 = t.n0 + 32 * ws;
        if (f0 < p.N && half_live) {
          const int gc = kGated ? gate_col(f0, p.ilv) : f0;
          zst_issue(zst_a, zrow + gc, zrow + gc + p.ilv, lane, kGated);
        }
      }
      const float prob = (EPI == EPI_STORE || !half_live) ? 0.f : p.row_prob[row];
      const bool got = mbar_wait(&c.tfull, acc_i & 1, abort, p.err);
      if (!__all_sync(0xFFFFFFFFu, got)) break;
      tc_fence_after();
      if (!half_live) {
        release_acc();
        ++acc_i;
        continue;
      }
      if constexpr (EPI == EPI_GLU) {
        // GLU: drain the 128 columns as fp32 (the activation and its MXFP8 blocks are computed
        // from the fp32 accumulator), free TMEM, then work from registers
        float acc[128];
        {
          const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + cb;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + 32 * j, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[32 * j + i] = __uint_as_float(r[i]);
          }
        }
        release_acc();
        ++acc_i;
        if constexpr (EXT && kGated) {
          // the bias joins Z before the activation (and is part of the saved Z); acc[c] holds
          // packed column n0 + cb + c, whose logical column follows from the interleave
          if (p.fc1_bias) {
            const float* b = p.fc1_bias + (int64_t)t.e * p.N1;
#pragma unroll
            for (int c = 0; c < 128; ++c) {
              const int pc = t.n0 + cb + c;
              const int blk = pc / ILV;
              const int lc = (blk >> 1) * ILV + pc % ILV + ((blk & 1) ? p.F : 0);
              if (pc < p.N) acc[c] += b[lc];
            }
          }
        }
        // segments are 128-row aligned, so every row of the tile is inside its segment
        uint16_t* zout = static_cast<uint16_t*>(p.out) + (int64_t)row * p.ldo + t.n0 + cb;
        if (p.out) {  // the saved Z (bf16); absent when the backward recomputes it
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (t.n0 + cb + 32 * j < p.N) store_bf16x32_v8(zout + 32 * j, &acc[32 * j]);
        }
        uint8_t* qr = p.q_row + (int64_t)row * p.ld_q_row;
        uint8_t* qc = p.q_col + (int64_t)row * p.ld_q_col;
        if constexpr (kGated) {
          // this half holds 64 gate and 64 linear columns: two 32-wide output blocks
#pragma unroll
          for (int c32 = 0; c32 < 2; ++c32) {
            const int g_off = (c32 * 32 / ILV) * 2 * ILV + (c32 * 32) % ILV;  // within the half
            const int acol = (t.n0 + cb) / 2 + c32 * 32;
            if (t.n0 + cb + g_off >= p.N) break;
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
              v[i] = prob * act_fwd_k<KIND>(p.act, acc[g_off + i], acc[g_off + ILV + i]);
            if constexpr (EXT) {
              if (p.fscale) {
                const float* sc = p.fscale + (int64_t)t.e * p.F + acol;
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= sc[i];
              }
            }
            mx_row_block(v, qr + acol, p.s_row + sf_mma_offset(row, acol / 32, p.s_row_pad));
            mx_col_block(v, xs, qc + acol, p.s_col, acol, row0 / 32, p.s_col_pad, lane);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int acol = t.n0 + cb + 32 * j;
            if (acol >= p.N) break;
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float rr = fmaxf(acc[32 * j + i], 0.f);
              v[i] = prob * rr * rr;
            }
            mx_row_block(v, qr + acol, p.s_row + sf_mma_offset(row, acol / 32, p.s_row_pad));
            mx_col_block(v, xs, qc + acol, p.s_col, acol, row0 / 32, p.s_col_pad, lane);
          }
        }
        continue;
      }
      // STORE: drain 128 accumulator columns into registers as packed bf16; dGLU: pack them
      // into this warp's 64 columns of the TMEM packed area instead (registers stay free for
      // the dGLU math). Either way the fp32 accumulator is released before any other work.
      const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16);  // this lane quadrant
      uint32_t pk[EPI == EPI_STORE ? 64 : 1];
      if constexpr (EPI == EPI_STORE) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tq + cb + 32 * j, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[16 * j + i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
        }
      } else {
        // chunk c (32 columns) packs into TMEM columns kPackCol + 16 c
#pragma unroll 1
        for (int c = ws; c < BN / 32; c += EWQ) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tq + 32 * c, r);
          tmem_ld_wait();
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
          tmem_st_32x32b_x16(tq + kPackCol + 16 * c, w);
        }
        tmem_st_wait();
      }
      release_acc();
      ++acc_i;

      if constexpr (EPI == EPI_STORE) {
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
      } else {  // EPI_DGLU: accumulator = dA_s over F columns
        float dp0 = 0.f, dp1 = 0.f, dp2 = 0.f, dp3 = 0.f;
        uint8_t* qr = p.q_row + (int64_t)row * p.ld_q_row;
        uint8_t* qc = p.q_col + (int64_t)row * p.ld_q_col;
        // one copy of the chunk body (keeps the kernel inside the instruction cache); chunk c
        // of the packed accumulator comes back from TMEM
#pragma unroll 1
        for (int c = ws; c < BN / 32; c += EWQ) {
          const int f0 = t.n0 + 32 * c;
          if (f0 >= p.N) break;
          uint32_t cur[16];
          tmem_ld_32x32b_x16(tq + kPackCol + 16 * c, cur);
          tmem_ld_wait();
          const int gcol = kGated ? gate_col(f0, p.ilv) : f0;
          const int lcol = gcol + p.ilv;
          float dg[32], dl[32];
          float ts[EXT ? 32 : 1];  // extras: p * dA_s * a of this row, for the scale gradient
          // this lane's own pieces of the chunk (each lane reads only the row it copied)
          asm volatile("cp.async.wait_all;" ::: "memory");
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t gw[8], lw[8];
            zst_piece(zst, 2 * h, lane, gw);
            zst_piece(zst, 2 * h + 1, lane, gw + 4);
            if (kGated) {
              zst_piece(zst, 4 + 2 * h, lane, lw);
              zst_piece(zst, 5 + 2 * h, lane, lw + 4);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int k = 16 * h + i;
              const float d = (k & 1) ? bf16_hi(cur[k >> 1]) : bf16_lo(cur[k >> 1]);
              const float g = (i & 1) ? bf16_hi(gw[i >> 1]) : bf16_lo(gw[i >> 1]);
              float contrib;
              if constexpr (EXT && kGated) {
                // the feature scale s enters as dA = p * s * dA_s and d_prob += dA_s * s * a
                const float l = (i & 1) ? bf16_hi(lw[i >> 1]) : bf16_lo(lw[i >> 1]);
                const float sc = p.fscale ? p.fscale[(int64_t)t.e * p.F + f0 + k] : 1.f;
                const float a = act_bwd_k<KIND>(p.act, g, l, prob * sc * d, dg[k], dl[k]);
                contrib = d * sc * a;
                ts[k] = prob * d * a;
              } else if constexpr (kGated) {
                const float l = (i & 1) ? bf16_hi(lw[i >> 1]) : bf16_lo(lw[i >> 1]);
                contrib = d * act_bwd_k<KIND>(p.act, g, l, prob * d, dg[k], dl[k]);
              } else {
                const float rr = fmaxf(g, 0.f);
                contrib = d * rr * rr;
                dg[k] = prob * d * 2.f * rr;
              }
              if ((k & 3) == 0) dp0 += contrib;
              else if ((k & 3) == 1) dp1 += contrib;
              else if ((k & 3) == 2) dp2 += contrib;
              else dp3 += contrib;
            }
          }
          // the next chunk's Z goes into the same buffer: this lane has read its row already
          if (c + EWQ < BN / 32 && f0 + 32 * EWQ < p.N) {
            const int gn = kGated ? gate_col(f0 + 32 * EWQ, p.ilv) : f0 + 32 * EWQ;
            zst_issue(zst_a, zrow + gn, zrow + gn + p.ilv, lane, kGated);
          }
          mx_row_block(dg, qr + gcol, p.s_row + sf_mma_offset(row, gcol / 32, p.s_row_pad));
          if constexpr (kGated)
            mx_row_block(dl, qr + lcol, p.s_row + sf_mma_offset(row, lcol / 32, p.s_row_pad));
          mx_col_block(dg, xs, qc + gcol, p.s_col, gcol, row0 / 32, p.s_col_pad, lane);
          if constexpr (kGated)
            mx_col_block(dl, xs, qc + lcol, p.s_col, lcol, row0 / 32, p.s_col_pad, lane);
          if constexpr (EXT && kGated) {
            // column sums over the warp's 32 rows (one expert's, segments being 128-row
            // aligned) of dZ (bias gradient) and of p * dA_s * a (scale gradient), into the
            // row group's partials: gate column f at f, linear at F + f, scale at N1 + f
            float* part = p.ext_part + (int64_t)(row0 >> 5) * (p.N1 + p.F);
            const float sg = warp_colsum32(dg, lane);
            const float sl = warp_colsum32(dl, lane);
            const float ss = warp_colsum32(ts, lane);
            part[f0 + lane] = sg;
            part[p.F + f0 + lane] = sl;
            part[p.N1 + f0 + lane] = ss;
          }
        }
        p.dprob_part[(int64_t)row * p.nparts + (t.n0 / BN) * EWQ + ws] = (dp0 + dp1) + (dp2 + dp3);
      }
    }
    if constexpr (EPI == EPI_DGLU) asm volatile("cp.async.wait_all;" ::: "memory");
    if constexpr (TST) {
      if (lane == 0) bulk_wait0();  // every box this warp stored has landed
      __syncwarp();
    }
  }

  griddep_launch_dependents();  // this CTA's tiles are done
  tc_fence_before();
  __syncthreads();
  // a pair: neither CTA leaves while the other may still read its shared memory (the
  // leader's MMAs and scale copies) or signal its barriers
  if constexpr (PAIR) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

// An operand t has t.rows M/N indices and t.cols K indices. K-major data is [rows, cols]; the
// column-wise copies are MN-major, stored [cols (K), rows (M or N)].
bool tmap_fp8(CUtensorMap* m, const MxOperand& t, bool mn_major) {
  const uint64_t inner = mn_major ? t.rows : t.cols, outer = mn_major ? t.cols : t.rows;
  uint64_t dims[2] = {inner, outer};
  uint64_t strides[1] = {inner};
  uint32_t box[2] = {128, 128};
  return make_tmap(m, t.q, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

// The scale slabs of an operand as a [bytes / 16, 16] byte tensor (no swizzle); one box is
// `rows16` 16-byte rows (32 = one 512-byte slab of 128 rows, 64 = two). The extent is the
// workspace's scale buffer of the operand, its 1 KB of slack included.
bool tmap_sf(CUtensorMap* m, const MxOperand& t, uint32_t rows16) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t bytes =
      (uint64_t)((t.cols / 32 + 3) / 4) * (uint64_t)((t.rows + 127) / 128 * 128) * 4 + 1024;
  cuuint64_t dims[2] = {16, bytes / 16};
  cuuint64_t strides[1] = {16};
  cuuint32_t box[2] = {16, rows16};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, t.s, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 1: the block-scaled GEMMs run as CTA pairs (256-row tiles, cta_group::2 MMAs). Off: with a
// single TMEM accumulator per CTA (two do not fit beside the scale factors), every tile ends
// with the MMAs waiting until both CTAs' epilogues have drained it, and the cross-SM signals
// lengthen that wait; measured 2-20% slower than one-CTA tiles on the Mixtral and GPT-OSS
// layers, so the one-CTA kernels run.
#ifndef MOE_GEMM_MX_PAIR
#define MOE_GEMM_MX_PAIR 0
#endif
constexpr bool kMxPairs = MOE_GEMM_MX_PAIR != 0;

// `grid`: the CTAs the caller allows (SM margin applied) or, for a pair kernel, twice the pairs
// the tile count can use at most; pairs are further capped by how many fit at once.
template <int EPI, int KIND, bool KG, int ILV, bool A_MN, bool B_MN, bool EXT = false,
          bool TST = false>
cudaError_t launch_mx(const MxArgs& a, int grid, cudaStream_t s, int kid) {
  if constexpr (!kMxPairs || TST) {
    auto kern = grouped_gemm_mx_kernel<EPI, KIND, KG, ILV, A_MN, B_MN, false, EXT, TST>;
    constexpr int smem = MxSmem<EPI, false, TST>::TOTAL;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    launch_kernel(kern, grid, MxSmem<EPI, false, TST>::THREADS, smem, s, nullptr, 0, a);
    count_launch(s, kid);
    return cudaGetLastError();
  } else {
    auto kern = grouped_gemm_mx_kernel<EPI, KIND, KG, ILV, A_MN, B_MN, true, EXT>;
    constexpr int smem = MxSmem<EPI, true>::TOTAL;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(MxSmem<EPI, true>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int pairs = std::max(1, grid / 2);
    const int resident = max_resident_pairs(reinterpret_cast<const void*>(kern), &cfg);
    if (resident > 0) pairs = std::min(pairs, resident);
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    e = launch_kernel(kern, cfg.gridDim, cfg.blockDim, cfg.dynamicSmemBytes, s, attr, 1, a);
    count_launch(s, kid);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
}

// GLU / dGLU kernels for one activation. The dGLU epilogue takes the interleave at run time;
// the GLU epilogue indexes its registers with it, so it is compiled for 32 and 64. Layers with
// epilogue extras (gated activations) take the EXT instantiations.
template <int EPI, int KIND>
cudaError_t launch_act(const MxArgs& a, int grid, cudaStream_t s, int kid) {
  const bool ext = a.fc1_bias || a.fscale || a.ext_part;
  if constexpr (KIND == MOE_ACT_SRELU) {
    if (ext) return cudaErrorInvalidValue;
    return launch_mx<EPI, KIND, false, 64, false, false>(a, grid, s, kid);
  } else if constexpr (EPI == EPI_DGLU) {
    return ext ? launch_mx<EPI, KIND, false, 64, false, false, true>(a, grid, s, kid)
               : launch_mx<EPI, KIND, false, 64, false, false>(a, grid, s, kid);
  } else {
    if (ext)
      return a.ilv == 32 ? launch_mx<EPI, KIND, false, 32, false, false, true>(a, grid, s, kid)
                         : launch_mx<EPI, KIND, false, 64, false, false, true>(a, grid, s, kid);
    return a.ilv == 32 ? launch_mx<EPI, KIND, false, 32, false, false>(a, grid, s, kid)
                       : launch_mx<EPI, KIND, false, 64, false, false>(a, grid, s, kid);
  }
}

template <int EPI>
cudaError_t launch_glu_family(const MxArgs& a, int kind, int grid, cudaStream_t s, int kid) {
  switch (kind) {
    case MOE_ACT_SWIGLU: return launch_act<EPI, MOE_ACT_SWIGLU>(a, grid, s, kid);
    case MOE_ACT_CLAMPED_SWIGLU: return launch_act<EPI, MOE_ACT_CLAMPED_SWIGLU>(a, grid, s, kid);
    case MOE_ACT_GEGLU: return launch_act<EPI, MOE_ACT_GEGLU>(a, grid, s, kid);
    case MOE_ACT_SRELU: return launch_act<EPI, MOE_ACT_SRELU>(a, grid, s, kid);
    default: return cudaErrorInvalidValue;
  }
}


}  // namespace

int dprob_parts_mx(int F) { return MxSmem<EPI_DGLU, kMxPairs>::EWQ * ((F + BN - 1) / BN); }

// ------------------------------------------------------------------------------------------
// FC2 dgrad with the FC1 output recomputed (activation recomputation, [NV-blog] "What's
// next"), MXFP8 operands. Per 128-row x 128-column tile of dA_s two block-scaled GEMMs share
// one loop over H:
//   dA_s[rows, f0..f0+127]      = Q(dY)[rows] . Q_H(W2)[f0..f0+127]^T        (128 x 128)
//   Z[rows, 2f0 .. 2f0+255]     = Q(X)[rows]  . Q_H(W1p)[2f0 .. 2f0+255]^T   (128 x 256)
// (the packed W1 rows 2f0.. are the gate and linear columns of dA_s columns f0.., the
// interleave dividing 128; sReLU, not gated: Z[rows, f0..f0+127], a 128 x 128 GEMM with one
// W1 box and scale slab). TMEM: dA_s in columns 0-127, Z from 128 (to 383), the stages' scale
// factors from 384 (20 columns a stage). A stage holds four 128-byte k-blocks (80 KB) and
// their scale slabs; two stages. The dGLU epilogue reads dA_s and Z in fp32 straight from
// TMEM and writes dZ as row-wise and column-wise MXFP8 plus the per-row d_prob partials, like
// the saved-Z kernel's epilogue. One accumulator set: the next tile's MMAs start once every
// epilogue warp has read this one.
namespace {

constexpr int RC_BNA = 128;                 // dA_s columns per tile
constexpr int RC_BNZ = 256;                 // Z columns per tile
constexpr int RC_STAGES = 2;
constexpr int RC_A1 = BM * BK;              // dY k-block (16 KB)
constexpr int RC_B1 = RC_BNA * BK;          // W2 rows
constexpr int RC_A2 = BM * BK;              // X
constexpr int RC_B2 = RC_BNZ * BK;          // W1p rows
constexpr int RC_STAGE = RC_A1 + RC_B1 + RC_A2 + RC_B2;
constexpr int RC_SF = 512 + 512 + 512 + 1024;  // scale slabs of the four k-blocks
constexpr int RC_SF_OFF = RC_STAGES * RC_STAGE;
constexpr int RC_XPOSE_OFF = RC_SF_OFF + RC_STAGES * RC_SF;
constexpr int RC_CTRL_OFF = RC_XPOSE_OFF + kEpiWarps * XPOSE_WARP_BYTES;
constexpr int RC_TOTAL = RC_CTRL_OFF + 4096 + 1024;
constexpr int RC_ZCOL = RC_BNA;             // first TMEM column of Z
constexpr int RC_SFCOL = RC_BNA + RC_BNZ;   // first TMEM column of the scale factors
static_assert(RC_TOTAL <= 232448, "shared memory");
static_assert(RC_SFCOL + 20 * RC_STAGES <= kTmemCols, "TMEM map");

struct RcMxArgs {
  CUtensorMap tmDy, tmW2, tmX, tmW1;  // row-wise MXFP8 copies, 128 x 128-byte boxes
  const uint8_t *sf_dy, *sf_w2, *sf_x, *sf_w1;
  int64_t pad_dy, pad_w2, pad_x, pad_w1;
  const int32_t* offsets;
  int E, R_cap, H, F, N1, Fp, N1p, ilv;
  const float* row_prob;
  uint8_t *q_row, *s_row, *q_col, *s_col;  // dZ copies, as the saved-Z dGLU writes them
  int64_t s_row_pad, s_col_pad;
  float* dprob_part;
  int nparts;
  ActDev act;
  int* err;
};

struct RcCtrl {
  uint64_t full[RC_STAGES];
  uint64_t empty[RC_STAGES];
  uint64_t tfull;
  uint64_t tempty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int off[kMaxE + 1];
  int prefix[kMaxE + 1];
};

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    fc2_dgrad_recompute_mx_kernel(const __grid_constant__ RcMxArgs p) {
  MOE_GRIDDEP_ENTRY();
  constexpr bool kGated = KIND != MOE_ACT_SRELU;
  constexpr int ZN = kGated ? RC_BNZ : RC_BNA;  // Z columns per tile
  // bytes a stage receives: sReLU loads one 128-row W1 box and one 512-byte W1 scale slab
  constexpr uint32_t kStageTx = RC_STAGE + RC_SF - (kGated ? 0 : 128 * BK + 512);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  RcCtrl& c = *reinterpret_cast<RcCtrl*>(smem + RC_CTRL_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &c.abort;
  const int NT = (p.F + RC_BNA - 1) / RC_BNA;
  const int nkb = (p.H + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RC_STAGES; ++s) {
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
  // tile -> (expert, first row, first dA_s column)
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
    n0 = (local / mt) * RC_BNA;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int armed[RC_STAGES];
#pragma unroll
      for (int s = 0; s < RC_STAGES; ++s) armed[s] = -1;
      for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x) {
        int e, m0, n0;
        decode(tile, e, m0, n0);
        const int w2_row = e * p.Fp + n0, w1_row = e * p.N1p + (kGated ? 2 * n0 : n0);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&c.empty[stage], phase ^ 1, abort, p.err)) break;
          uint8_t* s0 = smem + stage * RC_STAGE;
          uint8_t* sf = smem + RC_SF_OFF + stage * RC_SF;
          uint64_t* bar = &c.full[stage];
          mbar_arrive_expect_tx(bar, kStageTx);
#pragma unroll
          for (int s = 0; s < RC_STAGES; ++s)
            if (s == stage) armed[s] = (int)phase;
          const int k0 = kb * BK;
          tma_load_2d(s0, &p.tmDy, bar, k0, m0);
          tma_load_2d(s0 + RC_A1, &p.tmW2, bar, k0, w2_row);
          tma_load_2d(s0 + RC_A1 + RC_B1, &p.tmX, bar, k0, m0);
          tma_load_2d(s0 + RC_A1 + RC_B1 + RC_A2, &p.tmW1, bar, k0, w1_row);
          if (kGated) tma_load_2d(s0 + RC_A1 + RC_B1 + RC_A2 + 128 * BK, &p.tmW1, bar, k0, w1_row + 128);
          const int64_t kg = kb;  // k-block index = group of four 32-element scale blocks
          bulk_load(sf, p.sf_dy + (kg * p.pad_dy + m0) * 4, 512, bar);
          bulk_load(sf + 512, p.sf_w2 + (kg * p.pad_w2 + w2_row) * 4, 512, bar);
          bulk_load(sf + 1024, p.sf_x + (kg * p.pad_x + m0) * 4, 512, bar);
          bulk_load(sf + 1536, p.sf_w1 + (kg * p.pad_w1 + w1_row) * 4, kGated ? 1024 : 512, bar);
          if (++stage == RC_STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
#pragma unroll
      for (int s = 0; s < RC_STAGES; ++s) {
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
          const uint32_t s0 = smem_u32(smem + stage * RC_STAGE);
          const uint32_t sB1 = s0 + RC_A1, sA2 = sB1 + RC_B1, sB2 = sA2 + RC_A2;
          const uint32_t sf = smem_u32(smem + RC_SF_OFF + stage * RC_SF);
          const uint32_t t_sf = tmem_base + RC_SFCOL + stage * 20;
          tmem_cp_32x128b_warpx4(t_sf, smem_desc_noswizzle(sf, 0, 128));              // dY
          tmem_cp_32x128b_warpx4(t_sf + 4, smem_desc_noswizzle(sf + 512, 0, 128));    // W2
          tmem_cp_32x128b_warpx4(t_sf + 8, smem_desc_noswizzle(sf + 1024, 0, 128));   // X
          tmem_cp_32x128b_warpx4(t_sf + 12, smem_desc_noswizzle(sf + 1536, 0, 128));  // W1
          if (kGated) tmem_cp_32x128b_warpx4(t_sf + 16, smem_desc_noswizzle(sf + 2048, 0, 128));
          const int rem = p.H - kb * BK;
          const int nsub = rem >= BK ? BK / MMA_K : (rem + MMA_K - 1) / MMA_K;
          for (int ks = 0; ks < nsub; ++ks) {
            const uint32_t acc = (kb | ks) != 0 ? 1u : 0u;
            mma_mxf8_ss(tmem_base, smem_desc_sw128(s0 + ks * MMA_K, 16, 1024),
                        smem_desc_sw128(sB1 + ks * MMA_K, 16, 1024),
                        idesc_mxf8(BM, RC_BNA, ks), t_sf, t_sf + 4, acc);
            mma_mxf8_ss(tmem_base + RC_ZCOL, smem_desc_sw128(sA2 + ks * MMA_K, 16, 1024),
                        smem_desc_sw128(sB2 + ks * MMA_K, 16, 1024),
                        idesc_mxf8(BM, ZN, ks), t_sf + 8, t_sf + 12, acc);
          }
          issued_any = true;
          mma_commit(&c.empty[stage]);
          if (++stage == RC_STAGES) {
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
    uint8_t* xs = smem + RC_XPOSE_OFF + (warp - 2) * XPOSE_WARP_BYTES;
    int acc_i = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      if (__shfl_sync(0xFFFFFFFFu, *abort, 0)) break;
      int e, m0, n0;
      decode(tile, e, m0, n0);
      const int row0 = m0 + q * 32;
      const int row = row0 + lane;
      const float prob = p.row_prob[row];  // segments are 128-row aligned: every row is inside
      const bool got = mbar_wait(&c.tfull, acc_i & 1, abort, p.err);
      if (!__all_sync(0xFFFFFFFFu, got)) break;
      tc_fence_after();
      const uint32_t tl = tmem_base + ((uint32_t)(q * 32) << 16);
      uint8_t* qr = p.q_row + (int64_t)row * p.N1;
      uint8_t* qc = p.q_col + (int64_t)row * p.N1;
      float dp = 0.f;
#pragma unroll 1
      for (int j = 0; j < 2; ++j) {
        const int cc = half * 64 + 32 * j;  // dA_s column within the tile
        if (n0 + cc >= p.F) break;
        if constexpr (!kGated) {
          // sReLU: dZ = p dA_s 2 relu(Z), d_prob += dA_s relu(Z)^2; dZ column = dA column
          float dz[32];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t da[16], z[16];
            tmem_ld_32x32b_x16(tl + cc + 16 * h, da);
            tmem_ld_32x32b_x16(tl + RC_ZCOL + cc + 16 * h, z);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float d = __uint_as_float(da[i]);
              const float rr = fmaxf(__uint_as_float(z[i]), 0.f);
              dp += d * rr * rr;
              dz[16 * h + i] = prob * d * 2.f * rr;
            }
          }
          const int col = n0 + cc;
          mx_row_block(dz, qr + col, p.s_row + sf_mma_offset(row, col / 32, p.s_row_pad));
          mx_col_block(dz, xs, qc + col, p.s_col, col, row0 / 32, p.s_col_pad, lane);
          continue;
        }
        const int gc = (cc / p.ilv) * 2 * p.ilv + (cc % p.ilv);  // gate column within the 256
        float dg[32], dl[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t da[16], g[16], l[16];
          tmem_ld_32x32b_x16(tl + cc + 16 * h, da);
          tmem_ld_32x32b_x16(tl + RC_ZCOL + gc + 16 * h, g);
          tmem_ld_32x32b_x16(tl + RC_ZCOL + gc + p.ilv + 16 * h, l);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float d = __uint_as_float(da[i]);
            const float a = act_bwd_k<KIND>(p.act, __uint_as_float(g[i]), __uint_as_float(l[i]),
                                            prob * d, dg[16 * h + i], dl[16 * h + i]);
            dp += d * a;
          }
        }
        const int gcol = 2 * n0 + gc, lcol = gcol + p.ilv;  // packed dZ columns
        mx_row_block(dg, qr + gcol, p.s_row + sf_mma_offset(row, gcol / 32, p.s_row_pad));
        mx_row_block(dl, qr + lcol, p.s_row + sf_mma_offset(row, lcol / 32, p.s_row_pad));
        mx_col_block(dg, xs, qc + gcol, p.s_col, gcol, row0 / 32, p.s_col_pad, lane);
        mx_col_block(dl, xs, qc + lcol, p.s_col, lcol, row0 / 32, p.s_col_pad, lane);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.tempty);
      ++acc_i;
      p.dprob_part[(int64_t)row * p.nparts + (n0 / RC_BNA) * 2 + half] = dp;
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

template <int KIND>
cudaError_t launch_rc_mx(const RcMxArgs& a, int grid, cudaStream_t s) {
  auto kern = fc2_dgrad_recompute_mx_kernel<KIND>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), RC_TOTAL);
  if (e != cudaSuccess) return e;
  launch_kernel(kern, grid, kThreads, RC_TOTAL, s, nullptr, 0, a);
  count_launch(s, MOE_K_GEMM_FC2_DGRAD);
  return cudaGetLastError();
}

}  // namespace

int dprob_parts_mx_recompute(int F) { return 2 * ((F + RC_BNA - 1) / RC_BNA); }

cudaError_t launch_fc2_dgrad_recompute_mx(const MxProblem& p, cudaStream_t s) {
  if (p.gated && p.ilv != 32 && p.ilv != 64) return cudaErrorInvalidValue;
  RcMxArgs a;
  memset(&a, 0, sizeof(a));
  if (!tmap_fp8(&a.tmDy, p.dy, false) || !tmap_fp8(&a.tmW2, p.w2, false) ||
      !tmap_fp8(&a.tmX, p.x, false) || !tmap_fp8(&a.tmW1, p.w1, false))
    return cudaErrorInvalidValue;
  a.sf_dy = p.dy.s; a.pad_dy = p.dy.s_pad;
  a.sf_w2 = p.w2.s; a.pad_w2 = p.w2.s_pad;
  a.sf_x = p.x.s; a.pad_x = p.x.s_pad;
  a.sf_w1 = p.w1.s; a.pad_w1 = p.w1.s_pad;
  a.offsets = p.offsets;
  a.E = p.E;
  a.R_cap = (int)p.R_cap;
  a.H = p.H;
  a.F = p.F;
  a.N1 = p.N1;
  a.Fp = p.Fp;
  a.N1p = p.N1p;
  a.ilv = p.ilv;
  a.row_prob = p.row_prob;
  a.q_row = p.dz.q; a.s_row = p.dz.s; a.s_row_pad = p.dz.s_pad;
  a.q_col = p.dzt.q; a.s_col = p.dzt.s; a.s_col_pad = p.dzt.s_pad;
  a.dprob_part = p.dprob_part;
  a.nparts = dprob_parts_mx_recompute(p.F);
  a.act = p.act;
  a.err = p.err;
  const int grid = std::max(1, p.num_ctas);
  switch (p.act.kind) {
    case MOE_ACT_SWIGLU: return launch_rc_mx<MOE_ACT_SWIGLU>(a, grid, s);
    case MOE_ACT_CLAMPED_SWIGLU: return launch_rc_mx<MOE_ACT_CLAMPED_SWIGLU>(a, grid, s);
    case MOE_ACT_GEGLU: return launch_rc_mx<MOE_ACT_GEGLU>(a, grid, s);
    case MOE_ACT_SRELU: return launch_rc_mx<MOE_ACT_SRELU>(a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_grouped_gemm_mx(const MxProblem& p, cudaStream_t s) {
  static const int kKid[6] = {MOE_K_GEMM_FC1_FPROP, MOE_K_GEMM_FC2_FPROP, MOE_K_GEMM_FC2_DGRAD,
                              MOE_K_GEMM_FC2_WGRAD, MOE_K_GEMM_FC1_DGRAD, MOE_K_GEMM_FC1_WGRAD};
  if (p.role < 0 || p.role > 5) return cudaErrorInvalidValue;
  if (p.gated && p.ilv != 32 && p.ilv != 64) return cudaErrorInvalidValue;
  if (p.gated != (p.act.kind != MOE_ACT_SRELU)) return cudaErrorInvalidValue;
  MxArgs a;
  memset(&a, 0, sizeof(a));
  a.offsets = p.offsets;
  a.E = p.E;
  a.R_cap = (int)p.R_cap;
  a.ilv = p.ilv;
  a.act = p.act;
  a.err = p.err;
  a.row_prob = p.row_prob;
  a.F = p.F;
  a.N1 = p.N1;
  if (p.role == ROLE_FC1_FPROP) {
    a.fc1_bias = p.fc1_bias;
    a.fscale = p.fscale;
  } else if (p.role == ROLE_FC2_DGRAD) {
    a.fscale = p.fscale;
    a.ext_part = p.ext_part;
  }
  const int H = p.H, F = p.F, N1 = p.N1;
  const MxOperand *A = nullptr, *B = nullptr;
  int grid = p.num_ctas;
  switch (p.role) {
    case ROLE_FC1_FPROP:  // X (rows) x W1 (rows e*N1p + n), K = H
      A = &p.x; B = &p.w1;
      a.K = H; a.N = N1; a.b_row_e = p.N1p;
      a.out = p.out; a.ldo = N1;
      a.q_row = p.a.q; a.s_row = p.a.s; a.ld_q_row = F; a.s_row_pad = p.a.s_pad;
      a.q_col = p.at.q; a.s_col = p.at.s; a.ld_q_col = F; a.s_col_pad = p.at.s_pad;
      break;
    case ROLE_FC2_FPROP:  // a_s x W2 (column-wise copy [E*Fp, H], MN-major), K = F
      A = &p.a; B = &p.w2t;
      a.K = F; a.N = H; a.b_k_e = p.Fp;
      a.out = p.out; a.ldo = H;
      break;
    case ROLE_FC2_DGRAD:  // dY x W2 (rows e*Fp + f), K = H
      A = &p.dy; B = &p.w2;
      a.K = H; a.N = F; a.b_row_e = p.Fp;
      a.z = static_cast<const uint16_t*>(p.z); a.ldz = N1;
      a.q_row = p.dz.q; a.s_row = p.dz.s; a.ld_q_row = N1; a.s_row_pad = p.dz.s_pad;
      a.q_col = p.dzt.q; a.s_col = p.dzt.s; a.ld_q_col = N1; a.s_col_pad = p.dzt.s_pad;
      a.dprob_part = p.dprob_part; a.nparts = dprob_parts_mx(F);
      break;
    case ROLE_FC1_DGRAD:  // dZ x W1 (column-wise copy [E*N1p, H], MN-major), K = N1
      A = &p.dz; B = &p.w1t;
      a.K = N1; a.N = H; a.b_k_e = p.N1p;
      a.out = p.out; a.ldo = H;
      break;
    case ROLE_FC2_WGRAD:  // dW2_e [F, H] = a_s^T dY over the expert's rows
      A = &p.at; B = &p.dyt;
      a.M = F; a.N = H;
      a.out = p.out; a.ldo = H; a.out_estride = (int64_t)F * H;
      break;
    case ROLE_FC1_WGRAD:  // dW1_e [N1, H] = dZ^T X over the expert's rows
      A = &p.dzt; B = &p.xt;
      a.M = N1; a.N = H;
      a.out = p.out; a.ldo = H; a.out_estride = (int64_t)N1 * H;
      break;
  }
  const bool kg = p.role == ROLE_FC2_WGRAD || p.role == ROLE_FC1_WGRAD;
  const bool b_mn = kg || p.role == ROLE_FC2_FPROP || p.role == ROLE_FC1_DGRAD;
  if (!tmap_fp8(&a.tmA, *A, kg) || !tmap_fp8(&a.tmB, *B, b_mn)) return cudaErrorInvalidValue;
  if (kMxPairs && (!tmap_sf(&a.tmSFA, *A, SFA_BYTES / 16) || !tmap_sf(&a.tmSFB, *B, SFB_BYTES / 16)))
    return cudaErrorInvalidValue;
  a.sfa = A->s; a.sfa_pad = A->s_pad;
  a.sfb = B->s; a.sfb_pad = B->s_pad;
  a.wide = (reinterpret_cast<uintptr_t>(a.out) & 31) == 0 && a.ldo % 16 == 0 &&
           a.out_estride % 16 == 0;
  const int kid = kKid[p.role];
  switch (p.role) {
    case ROLE_FC1_FPROP: return launch_glu_family<EPI_GLU>(a, p.act.kind, grid, s, kid);
    case ROLE_FC2_DGRAD: return launch_glu_family<EPI_DGLU>(a, p.act.kind, grid, s, kid);
    case ROLE_FC2_FPROP:
    case ROLE_FC1_DGRAD:
      return launch_mx<EPI_STORE, 0, false, 64, false, true>(a, grid, s, kid);
    default: {
      // experts with few rows: the weight-gradient tiles are short and their stores dominate,
      // so they go out through shared memory and TMA stores
      if (!kMxPairs && p.rows_per_expert <= 256) {
        uint64_t dims[3] = {(uint64_t)a.N, (uint64_t)a.M, (uint64_t)p.E};
        uint64_t strides[2] = {(uint64_t)a.N * 2, (uint64_t)a.M * a.N * 2};
        uint32_t box[3] = {64, 32, 1};
        if (!make_tmap(&a.tmOut, a.out, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
          return cudaErrorInvalidValue;
        const int64_t tiles = (int64_t)p.E * ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
        grid = (int)std::min<int64_t>(grid, tiles);
        return launch_mx<EPI_STORE, 0, true, 64, true, true, false, true>(a, grid, s, kid);
      }
      constexpr int TMr = kMxPairs ? 2 * BM : BM;
      const int64_t tiles = (int64_t)p.E * ((a.M + TMr - 1) / TMr) * ((a.N + BN - 1) / BN);
      grid = (int)std::min<int64_t>(grid, kMxPairs ? 2 * tiles : tiles);
      return launch_mx<EPI_STORE, 0, true, 64, true, true>(a, grid, s, kid);
    }
  }
}

}  // namespace moe
