// MXFP8 quantiser ([TE-MoE] Challenge 2 and Figure 3: E4M3 elements, one E8M0 scale per 32
// contiguous values). Scale exponent e = clamp(floor(log2 amax) - 8, -127, 127) (-127 for an
// all-zero block), element = E4M3(v * 2^-e) rounded to nearest even with saturation.
//
// Both outputs keep the input's row-major layout: the row-wise copy has blocks of 32 along a
// row, the column-wise copy blocks of 32 rows of one column. Per 128 x 128 tile (staged in
// shared memory by cp.async, three tiles in flight per CTA):
//   phase 1  one thread per (column pair, 32-row block): packed bf16x2 |max| gives the two
//            column-block exponents, kept in shared memory as E8M0 bytes and as 2^-e floats;
//   phase 2  one thread per (row, 32-column block), two blocks each: the 32 values are
//            quantised with their own row scale and with the 32 column scales, and each copy
//            leaves as one 32-byte run (a whole L2 sector, one 256-bit store when aligned);
//   flush    the tile's 128 x 4 row and 128 x 4 column scale bytes leave as 32-bit words; in
//            the MMA slab layout each set is 512 contiguous bytes.
// Index arithmetic is done once per tile; no per-element division.
//
// Rows may be grouped: input row g*G + i (i < G) becomes output row g*Gp + i, and rows
// g*Gp + G .. g*Gp + Gp - 1 are written as zeros (per-expert padding of the operands of the
// block-scaled grouped GEMM). Scales are written either in the logical layout
// ([rows, cols/32], [cols, rows/32]) or in the MMA-ready slab layout of sf_mma_offset.
#include "kernels.cuh"

namespace moe {

struct MxQuantArgs {
  const uint16_t* in;
  int64_t M, N;     // input [M, N] bf16
  int64_t G, Gp;    // row groups of G input rows, output group stride Gp (>= G)
  int rowwise, colwise;
  uint8_t* q_row;   // [Mv, N]       Mv = (M / G) * Gp, blocks along N
  uint8_t* s_row;
  uint8_t* q_col;   // [Mv, N]       blocks along Mv
  uint8_t* s_col;
  int sf_mma;       // 0: logical scale layout, 1: MMA slab layout
  int64_t srow_pad; // MMA layout: padded row count of the row-wise scales (multiple of 128)
  int64_t scol_pad; // MMA layout: padded row count of the column-wise scales
  int wide;         // q_row and q_col are 32-byte aligned: 256-bit stores
};

constexpr int QT_ROWS = 128;
constexpr int QT_COLS = 128;
constexpr int QT_LD = QT_COLS + 8;  // bf16 per smem row (272 B): conflict-free rows and columns
constexpr int QT_BUFS = 3;          // tiles in flight per CTA: the current one and two ahead
constexpr int QT_TILE_BYTES = QT_ROWS * QT_LD * 2;
constexpr int QT_INV_OFF = QT_BUFS * QT_TILE_BYTES;       // float [4][128]: column 2^-e
constexpr int QT_CEXP_OFF = QT_INV_OFF + 4 * QT_COLS * 4;  // uint8 [128 cols][4 row blocks]
constexpr int QT_REXP_OFF = QT_CEXP_OFF + QT_COLS * 4;     // uint8 [128 rows][4 col blocks]
constexpr int QT_SMEM = QT_REXP_OFF + QT_ROWS * 4;
constexpr int QT_THREADS = 256;

// Where one tile sits: virtual rows r0 .. r0+127 (vrows of them < Mv), of which the first
// srows come from input rows src0 .. (the rest are group padding), columns c0 .. c0+127.
struct QTile {
  int64_t r0, src0;
  int c0, vrows, srows;
};

MOE_DEVICE QTile quant_tile(const MxQuantArgs& a, int64_t Mv, uint32_t t, uint32_t tiles_n) {
  QTile q;
  const uint32_t tm = t / tiles_n;
  q.c0 = (int)(t - tm * tiles_n) * QT_COLS;
  q.r0 = (int64_t)tm * QT_ROWS;
  // a tile never straddles two groups: either one group (G == Gp) or Gp % 128 == 0
  const uint32_t g = (uint32_t)q.r0 / (uint32_t)a.Gp;
  const int64_t k0 = q.r0 - (int64_t)g * a.Gp;
  q.src0 = (int64_t)g * a.G + k0;
  q.srows = (int)max((int64_t)0, min((int64_t)QT_ROWS, a.G - k0));
  q.vrows = (int)min((int64_t)QT_ROWS, Mv - q.r0);
  return q;
}

MOE_DEVICE void quant_tile_issue(const MxQuantArgs& a, const QTile& q, int tid,
                                 uint16_t (*buf)[QT_LD]) {
#pragma unroll
  for (int j = 0; j < QT_ROWS * QT_COLS / 8 / QT_THREADS; ++j) {
    const int i = tid + QT_THREADS * j;
    const int rr = i >> 4, cc = (i & 15) * 8;
    const bool ok = rr < q.srows && q.c0 + cc < a.N;  // N % 32 == 0: whole 16-byte chunks
    const uint16_t* src = ok ? a.in + (q.src0 + rr) * a.N + q.c0 + cc : a.in;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(&buf[rr][cc])),
                 "l"(src), "r"(ok ? 16 : 0)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

MOE_DEVICE uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// One 32-byte run: a single 256-bit store when the destination is 32-byte aligned.
MOE_DEVICE void store_run32(uint8_t* dst, const uint32_t (&q)[8], bool wide) {
  if (wide) {
    st_global_v8(dst, q);
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
    d[0] = make_uint4(q[0], q[1], q[2], q[3]);
    d[1] = make_uint4(q[4], q[5], q[6], q[7]);
  }
}

__global__ void __launch_bounds__(QT_THREADS, 2) mxfp8_quantize_kernel(const MxQuantArgs a) {
  MOE_GRIDDEP_ENTRY();
  extern __shared__ __align__(16) uint8_t qsmem[];
  auto tiles = reinterpret_cast<uint16_t (*)[QT_ROWS][QT_LD]>(qsmem);
  float* cinv = reinterpret_cast<float*>(qsmem + QT_INV_OFF);
  uint8_t* cexp = qsmem + QT_CEXP_OFF;
  uint8_t* rexp = qsmem + QT_REXP_OFF;
  const int64_t Mv = (a.M / a.G) * a.Gp;
  const uint32_t tiles_n = (uint32_t)((a.N + QT_COLS - 1) / QT_COLS);
  const uint32_t ntiles = (uint32_t)((Mv + QT_ROWS - 1) / QT_ROWS) * tiles_n;
  const int tid = threadIdx.x;
  // one commit group per tile slot (possibly empty), so "wait until QT_BUFS-1 groups remain"
  // always means "the current tile has landed"
  for (int j = 0; j < QT_BUFS - 1; ++j) {
    const uint32_t tj = blockIdx.x + (uint32_t)j * gridDim.x;
    if (tj < ntiles) quant_tile_issue(a, quant_tile(a, Mv, tj, tiles_n), tid, tiles[j]);
    else asm volatile("cp.async.commit_group;" ::: "memory");
  }
  int it = 0;
  for (uint32_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
    const QTile q = quant_tile(a, Mv, t, tiles_n);
    uint16_t (*tile)[QT_LD] = tiles[it % QT_BUFS];
    const uint32_t tn = t + (uint32_t)(QT_BUFS - 1) * gridDim.x;
    if (tn < ntiles)
      quant_tile_issue(a, quant_tile(a, Mv, tn, tiles_n), tid, tiles[(it + QT_BUFS - 1) % QT_BUFS]);
    else asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group %0;" ::"n"(QT_BUFS - 1) : "memory");
    __syncthreads();
    // ---- phase 1: exponents of (column pair, 32-row block); padding reads as zeros
    if (a.colwise) {
      const int cp = tid & 63, rb = tid >> 6;
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        m = bf16x2_max(m, *reinterpret_cast<const uint32_t*>(&tile[rb * 32 + i][2 * cp]) &
                              0x7FFF7FFFu);
      const int e0 = mx_block_exponent(bf16_lo(m)), e1 = mx_block_exponent(bf16_hi(m));
      *reinterpret_cast<float2*>(cinv + rb * QT_COLS + 2 * cp) =
          make_float2(mx_inv_scale(e0), mx_inv_scale(e1));
      cexp[(2 * cp) * 4 + rb] = (uint8_t)(e0 + 127);
      cexp[(2 * cp + 1) * 4 + rb] = (uint8_t)(e1 + 127);
    }
    __syncthreads();
    // ---- phase 2: (row, 32-column block); a warp spans 32 consecutive rows
    {
      const int rr = tid & 127, half = tid >> 7;
      const int64_t row = q.r0 + rr;
#pragma unroll 1
      for (int b = 0; b < 2; ++b) {
        const int blk = 2 * half + b, cl = 32 * blk;
        const bool ok = rr < q.vrows && q.c0 + cl < a.N;
        uint32_t sbyte = 0;  // scale byte of blocks that are not written
        if (ok) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 w = *reinterpret_cast<const uint4*>(&tile[rr][cl + 8 * i]);
            v[8 * i + 0] = bf16_lo(w.x); v[8 * i + 1] = bf16_hi(w.x);
            v[8 * i + 2] = bf16_lo(w.y); v[8 * i + 3] = bf16_hi(w.y);
            v[8 * i + 4] = bf16_lo(w.z); v[8 * i + 5] = bf16_hi(w.z);
            v[8 * i + 6] = bf16_lo(w.w); v[8 * i + 7] = bf16_hi(w.w);
          }
          const int64_t off = row * a.N + q.c0 + cl;
          uint32_t qw[8];
          if (a.rowwise) {
            sbyte = mx_quant_block(v, qw);
            store_run32(a.q_row + off, qw, a.wide);
          }
          if (a.colwise) {
            const float* iv = cinv + (rr >> 5) * QT_COLS + cl;  // same address across a warp
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 s4 = *reinterpret_cast<const float4*>(iv + 4 * i);
              const uint32_t lo = cvt_e4m3x2(v[4 * i] * s4.x, v[4 * i + 1] * s4.y);
              const uint32_t hi = cvt_e4m3x2(v[4 * i + 2] * s4.z, v[4 * i + 3] * s4.w);
              qw[i] = lo | (hi << 16);
            }
            store_run32(a.q_col + off, qw, a.wide);
          }
        }
        if (a.rowwise) rexp[rr * 4 + blk] = (uint8_t)sbyte;
      }
    }
    __syncthreads();
    // ---- flush the tile's scale bytes (rexp / cexp are rewritten only after the next
    // iteration's first barrier)
    if (a.sf_mma) {
      // slab position p holds row (p & 3) * 32 + (p >> 2) of the 128-row slab
      const int p = tid & 127, lr = (p & 3) * 32 + (p >> 2);
      if (tid < 128) {
        if (a.rowwise)
          *reinterpret_cast<uint32_t*>(a.s_row + ((q.c0 / 128) * a.srow_pad + q.r0 + p) * 4) =
              *reinterpret_cast<const uint32_t*>(rexp + lr * 4);
      } else if (a.colwise) {
        *reinterpret_cast<uint32_t*>(a.s_col + ((q.r0 / 128) * a.scol_pad + q.c0 + p) * 4) =
            *reinterpret_cast<const uint32_t*>(cexp + lr * 4);
      }
    } else {
      if (tid < 128) {
        if (a.rowwise && tid < q.vrows) {
          for (int blk = 0; blk < 4; ++blk)
            if (q.c0 + 32 * blk < a.N)
              a.s_row[(q.r0 + tid) * (a.N / 32) + q.c0 / 32 + blk] = rexp[tid * 4 + blk];
        }
      } else if (a.colwise) {
        const int cl = tid - 128;
        if (q.c0 + cl < a.N) {
          for (int rb = 0; rb < 4; ++rb)
            if (32 * rb < q.vrows)
              a.s_col[(q.c0 + cl) * (Mv / 32) + q.r0 / 32 + rb] = cexp[cl * 4 + rb];
        }
      }
    }
  }
}

static bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

static void launch(MxQuantArgs a, int num_sms, cudaStream_t s) {
  const int64_t Mv = (a.M / a.G) * a.Gp;
  const int64_t tiles = ((Mv + QT_ROWS - 1) / QT_ROWS) * ((a.N + QT_COLS - 1) / QT_COLS);
  if (tiles == 0) return;
  a.wide = (!a.rowwise || aligned32(a.q_row)) && (!a.colwise || aligned32(a.q_col)) &&
           a.N % 32 == 0;
  // on failure the launch below fails too and the caller reports the CUDA error
  ensure_smem_attr(reinterpret_cast<const void*>(mxfp8_quantize_kernel), QT_SMEM);
  const int grid = (int)std::min<int64_t>(tiles, (int64_t)num_sms * 2);
  launch_kernel(mxfp8_quantize_kernel, grid, QT_THREADS, QT_SMEM, s, nullptr, 0, a);
  count_launch(s, MOE_K_MXFP8_QUANTIZE);
}

// Column-wise MXFP8 with blocks that restart at each group's first row (group offsets in
// device memory, any alignment): group g holds rows [off[g], off[g+1]); its i-th block is rows
// off[g] + 32 i .. min(off[g] + 32 i + 32, off[g+1]) (a short last block is quantised as if
// padded with zeros, which leave the block's amax unchanged). The scale of (column c,
// block (g, i)) sits at s[c * nb + off[g] / 32 + g + i]: the start index off[g] / 32 + g grows
// by at least the previous group's block count, so blocks never share an entry; entries no
// block owns are written 0. nb (a multiple of 4) >= ceil(M / 32) + G.
//
// Work item: four consecutive scale entries b0 .. b0+3 (one 32-bit scale word per column)
// over 256 columns; a thread owns a column pair. Offsets are clamped into [0, M] as they are
// read, so invalid offsets cannot take an access outside the buffers.
constexpr int QG_THREADS = 128;
__global__ void __launch_bounds__(QG_THREADS) mxfp8_colwise_grouped_kernel(
    const uint16_t* __restrict__ in, int64_t M, int64_t N, const int32_t* __restrict__ off,
    int G, int64_t nb, uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
  MOE_GRIDDEP_ENTRY();
  __shared__ int64_t s_rb[4], s_re[4];
  const int64_t col_items = (N + 2 * QG_THREADS - 1) / (2 * QG_THREADS);
  const int64_t items = (nb / 4) * col_items;
  auto o = [&](int g) -> int64_t {
    const int64_t v = off[g];
    return v < 0 ? 0 : (v > M ? M : v);
  };
  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    const int64_t b0 = (it / col_items) * 4;
    const int64_t c = (it % col_items) * (2 * QG_THREADS) + 2 * threadIdx.x;
    __syncthreads();  // the previous item's block bounds have been read
    if (threadIdx.x < 4) {
      // the block of scale entry b: the last group whose start index is <= b
      const int64_t b = b0 + threadIdx.x;
      int lo = 0, hi = G;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (o(mid) / 32 + mid <= b) lo = mid; else hi = mid;
      }
      const int64_t i = b - (o(lo) / 32 + lo);
      int64_t rb = o(lo) + 32 * i, re = o(lo + 1);
      if (i < 0 || rb >= re) rb = re = 0;  // no block owns this entry
      s_rb[threadIdx.x] = rb;
      s_re[threadIdx.x] = rb + 32 < re ? rb + 32 : re;
    }
    __syncthreads();
    if (c >= N) continue;
    uint32_t sc0 = 0, sc1 = 0;  // scale words of columns c and c + 1 (byte j: entry b0 + j)
#pragma unroll 1
    for (int j = 0; j < 4; ++j) {
      const int64_t rb = s_rb[j], n = s_re[j] - rb;
      if (n <= 0) continue;
      uint32_t w[32];
      uint32_t m = 0;
#pragma unroll
      for (int r = 0; r < 32; ++r) {
        w[r] = r < n ? *reinterpret_cast<const uint32_t*>(in + (rb + r) * N + c) : 0u;
        m = bf16x2_max(m, w[r] & 0x7FFF7FFFu);
      }
      const int e0 = mx_block_exponent(bf16_lo(m)), e1 = mx_block_exponent(bf16_hi(m));
      const float i0 = mx_inv_scale(e0), i1 = mx_inv_scale(e1);
#pragma unroll
      for (int r = 0; r < 32; ++r)
        if (r < n)
          *reinterpret_cast<uint16_t*>(q + (rb + r) * N + c) =
              (uint16_t)cvt_e4m3x2(bf16_lo(w[r]) * i0, bf16_hi(w[r]) * i1);
      sc0 |= (uint32_t)(e0 + 127) << (8 * j);
      sc1 |= (uint32_t)(e1 + 127) << (8 * j);
    }
    *reinterpret_cast<uint32_t*>(s + c * nb + b0) = sc0;
    *reinterpret_cast<uint32_t*>(s + (c + 1) * nb + b0) = sc1;
  }
}

int64_t mxfp8_grouped_scale_cols(int64_t M, int G) { return ((M + 31) / 32 + G + 3) / 4 * 4; }

void launch_mxfp8_colwise_grouped(const void* in, int64_t M, int64_t N, const int32_t* offsets,
                                  int G, uint8_t* q_col, uint8_t* s_col, int num_sms,
                                  cudaStream_t s) {
  const int64_t nb = mxfp8_grouped_scale_cols(M, G);
  const int64_t items = (nb / 4) * ((N + 2 * QG_THREADS - 1) / (2 * QG_THREADS));
  if (items == 0) return;
  const int grid = (int)std::min<int64_t>(items, (int64_t)num_sms * 8);
  launch_kernel(mxfp8_colwise_grouped_kernel, grid, QG_THREADS, 0, s, nullptr, 0, 
      static_cast<const uint16_t*>(in), M, N, offsets, G, nb, q_col, s_col);
  count_launch(s, MOE_K_MXFP8_QUANTIZE);
}

bool mxfp8_quantize_size_ok(int64_t M, int64_t N) {
  const int64_t tm = (M + QT_ROWS - 1) / QT_ROWS, tn = (N + QT_COLS - 1) / QT_COLS;
  return M <= (int64_t)INT32_MAX - QT_ROWS && N <= (int64_t)INT32_MAX &&
         tm * tn <= (int64_t)INT32_MAX;
}

void launch_mxfp8_quantize(const void* in, int64_t M, int64_t N, int rowwise, int colwise,
                           uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                           int num_sms, cudaStream_t s) {
  // one group spanning all rows
  MxQuantArgs a{static_cast<const uint16_t*>(in), M, N, M, M, rowwise, colwise,
                q_row, s_row, q_col, s_col, 0, 0, 0, 0};
  launch(a, num_sms, s);
}

void launch_mxfp8_quantize_mma(const void* in, int64_t M, int64_t N, int64_t G, int64_t Gp,
                               uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                               int num_sms, cudaStream_t s) {
  if (G == Gp) G = Gp = M;  // ungrouped: one group, so tiles need not align to Gp
  const int64_t Mv = (M / G) * Gp;
  MxQuantArgs a{static_cast<const uint16_t*>(in), M, N, G, Gp, q_row != nullptr,
                q_col != nullptr, q_row, s_row, q_col, s_col, 1, (Mv + 127) / 128 * 128,
                (N + 127) / 128 * 128, 0};
  launch(a, num_sms, s);
}

}  // namespace moe
