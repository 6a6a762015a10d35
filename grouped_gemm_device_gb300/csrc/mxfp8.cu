// MXFP8 quantiser ([TE-MoE] Challenge 2 and Figure 3: E4M3 elements, one E8M0 scale per 32
// contiguous values). Scale exponent e = clamp(floor(log2 amax) - 8, -127, 127) (-127 for an
// all-zero block), element = E4M3(v * 2^-e) rounded to nearest even with saturation.
//
// Both outputs keep the input's row-major layout: the row-wise copy has blocks of 32 along a
// row, the column-wise copy blocks of 32 rows of one column. Per 128-row x 64-column tile
// (staged in shared memory): phase 1, one thread per (column, 32-row block) finds the column
// block's exponent; phase 2, one thread per (row, 32-column block) quantises its 32 values
// twice - with its own row scale and with the 32 column scales - and stores two 32-byte runs.
// Every global store is therefore a contiguous row segment.
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
};

// Tile: 128 (virtual) rows x 64 columns, buffered in shared memory and filled with cp.async
// (16-byte asynchronous copies, zero-fill for padding rows and tails), so later tiles are in
// flight while the current one is quantised and no registers hold in-flight data.
constexpr int QT_ROWS = 128;
constexpr int QT_COLS = 64;
constexpr int QT_LD = QT_COLS + 8;  // padded row (bf16 elements): conflict-free column reads
constexpr int QT_BUFS = 3;          // tiles in flight per CTA: the current one and two ahead
constexpr int QT_TILE_BYTES = QT_ROWS * QT_LD * 2;
constexpr int QT_EXP_BYTES = (QT_ROWS / 32) * QT_COLS * 4;
constexpr int QT_SMEM = QT_BUFS * QT_TILE_BYTES + QT_EXP_BYTES;

MOE_DEVICE void quant_tile_issue(const MxQuantArgs& a, int64_t Mv, int64_t tiles_n, int64_t t,
                                 int tid, uint16_t (*buf)[QT_LD]) {
  const int64_t r0 = (t / tiles_n) * QT_ROWS, c0 = (t % tiles_n) * QT_COLS;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = tid + 256 * j;
    const int rr = i >> 3, cc = (i & 7) * 8;
    const int64_t v = r0 + rr;
    const uint16_t* src = a.in;  // any valid address when nothing is copied
    uint32_t bytes = 0;
    if (v < Mv && c0 + cc < a.N) {
      const int64_t g = v / a.Gp, k = v - g * a.Gp;
      if (k < a.G) {
        src = a.in + (g * a.G + k) * a.N + c0 + cc;
        bytes = 16;
      }
    }
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(&buf[rr][cc])),
                 "l"(src), "r"(bytes)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

__global__ void __launch_bounds__(256) mxfp8_quantize_kernel(const MxQuantArgs a) {
  extern __shared__ __align__(16) uint8_t qsmem[];
  auto tiles = reinterpret_cast<uint16_t (*)[QT_ROWS][QT_LD]>(qsmem);
  int* cexp = reinterpret_cast<int*>(qsmem + QT_BUFS * QT_TILE_BYTES);  // [4][64]
  const int64_t Mv = (a.M / a.G) * a.Gp;
  const int64_t tiles_m = (Mv + QT_ROWS - 1) / QT_ROWS, tiles_n = (a.N + QT_COLS - 1) / QT_COLS;
  const int64_t ntiles = tiles_m * tiles_n;
  const int tid = threadIdx.x;
  // one commit group per tile slot (possibly empty), so "wait until 2 groups remain" always
  // means "the current tile has landed"
  for (int j = 0; j < QT_BUFS - 1; ++j) {
    const int64_t tj = blockIdx.x + (int64_t)j * gridDim.x;
    if (tj < ntiles) quant_tile_issue(a, Mv, tiles_n, tj, tid, tiles[j]);
    else asm volatile("cp.async.commit_group;" ::: "memory");
  }
  int it = 0;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
    const int64_t r0 = (t / tiles_n) * QT_ROWS, c0 = (t % tiles_n) * QT_COLS;
    uint16_t (*tile)[QT_LD] = tiles[it % QT_BUFS];
    const int64_t tn = t + (int64_t)(QT_BUFS - 1) * gridDim.x;
    if (tn < ntiles) quant_tile_issue(a, Mv, tiles_n, tn, tid, tiles[(it + QT_BUFS - 1) % QT_BUFS]);
    else asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group %0;" ::"n"(QT_BUFS - 1) : "memory");
    __syncthreads();
    // ---- phase 1: exponent of each (column, 32-row block)
    if (a.colwise) {
      const int cc = tid & 63, rb = tid >> 6;
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        amax = fmaxf(amax, fabsf(__uint_as_float((uint32_t)tile[rb * 32 + i][cc] << 16)));
      const int e = mx_block_exponent(amax);
      cexp[rb * 64 + cc] = e;
      const int64_t col = c0 + cc, row = r0 + rb * 32;
      if (col < a.N && row < Mv) {
        const int64_t so = a.sf_mma ? sf_mma_offset(col, row / 32, a.scol_pad)
                                    : col * (Mv / 32) + row / 32;
        a.s_col[so] = (uint8_t)(e + 127);
      }
    }
    __syncthreads();
    // ---- phase 2: one (row, 32-column block) per thread; a warp spans 32 consecutive rows
    {
      const int rr = tid & 127, blk = tid >> 7;
      const int64_t row = r0 + rr, col = c0 + blk * 32;
      if (row < Mv && col < a.N) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 w = *reinterpret_cast<const uint4*>(&tile[rr][blk * 32 + 8 * i]);
          v[8 * i + 0] = bf16_lo(w.x); v[8 * i + 1] = bf16_hi(w.x);
          v[8 * i + 2] = bf16_lo(w.y); v[8 * i + 3] = bf16_hi(w.y);
          v[8 * i + 4] = bf16_lo(w.z); v[8 * i + 5] = bf16_hi(w.z);
          v[8 * i + 6] = bf16_lo(w.w); v[8 * i + 7] = bf16_hi(w.w);
        }
        uint32_t q[8];
        if (a.rowwise) {
          const uint32_t s = mx_quant_block(v, q);
          uint4* dst = reinterpret_cast<uint4*>(a.q_row + row * a.N + col);
          dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
          dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
          const int64_t so = a.sf_mma ? sf_mma_offset(row, col / 32, a.srow_pad)
                                      : row * (a.N / 32) + col / 32;
          a.s_row[so] = (uint8_t)s;
        }
        if (a.colwise) {
          const int* ce = cexp + (rr >> 5) * 64 + blk * 32;  // same address across the warp
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int4 e4 = *reinterpret_cast<const int4*>(ce + 4 * i);
            const uint32_t lo = cvt_e4m3x2(v[4 * i] * mx_inv_scale(e4.x),
                                           v[4 * i + 1] * mx_inv_scale(e4.y));
            const uint32_t hi = cvt_e4m3x2(v[4 * i + 2] * mx_inv_scale(e4.z),
                                           v[4 * i + 3] * mx_inv_scale(e4.w));
            q[i] = lo | (hi << 16);
          }
          uint4* dst = reinterpret_cast<uint4*>(a.q_col + row * a.N + col);
          dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
          dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
        }
      }
    }
    __syncthreads();  // this buffer (and cexp) are reused by the next iteration
  }
}

static void launch(const MxQuantArgs& a, int num_sms, cudaStream_t s) {
  const int64_t Mv = (a.M / a.G) * a.Gp;
  const int64_t tiles = ((Mv + QT_ROWS - 1) / QT_ROWS) * ((a.N + QT_COLS - 1) / QT_COLS);
  if (tiles == 0) return;
  static bool configured = false;
  if (!configured) {
    // on failure the launch below fails too and the caller reports the CUDA error
    configured = cudaFuncSetAttribute(mxfp8_quantize_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      QT_SMEM) == cudaSuccess;
  }
  const int grid = (int)std::min<int64_t>(tiles, (int64_t)num_sms * 4);
  mxfp8_quantize_kernel<<<grid, 256, QT_SMEM, s>>>(a);
  count_launch(s, MOE_K_MXFP8_QUANTIZE);
}

void launch_mxfp8_quantize(const void* in, int64_t M, int64_t N, int rowwise, int colwise,
                           uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                           int num_sms, cudaStream_t s) {
  MxQuantArgs a{static_cast<const uint16_t*>(in), M, N, M, M, rowwise, colwise,
                q_row, s_row, q_col, s_col, 0, 0, 0};
  launch(a, num_sms, s);
}

void launch_mxfp8_quantize_mma(const void* in, int64_t M, int64_t N, int64_t G, int64_t Gp,
                               uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                               int num_sms, cudaStream_t s) {
  const int64_t Mv = (M / G) * Gp;
  MxQuantArgs a{static_cast<const uint16_t*>(in), M, N, G, Gp, q_row != nullptr,
                q_col != nullptr, q_row, s_row, q_col, s_col, 1, (Mv + 127) / 128 * 128,
                (N + 127) / 128 * 128};
  launch(a, num_sms, s);
}

}  // namespace moe
