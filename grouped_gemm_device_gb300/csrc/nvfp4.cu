// NVFP4 quantiser and per-tensor amax kernels (scaling rule and layouts in nvfp4.cuh).
//
// [NV-blog] section "fused MXFP8 and NVFP4 quantisation": the quantisation of an NVFP4 GEMM
// operand needs the tensor's amax before any block can be encoded, so it is a second pass over
// a BF16 tensor whose amax is already known: for the FC1 output a_s and for dZ the GEMM
// epilogues provide it; for the routed input, dY and the weights the amax kernels below do.
//
// Quantiser: a CTA of 128 threads walks 128-row x 64-column tiles of a bf16 matrix, staged in
// shared memory (144-byte rows, so that both the row reads and the column reads are free of
// bank conflicts). Thread t then quantises
//   row-wise    row t's 64 values (four 16-blocks along the row, the reduction dimension of
//               the row-grouped GEMMs) into one 32-byte run and one 32-bit word of scales;
//   transposed  columns 2 (t % 32), 2 (t % 32) + 1 over rows 32 (t / 32) .. + 31 (two 16-blocks
//               along the rows per column, optionally Hadamard-rotated first) into a 16-byte
//               run and a 16-bit scale pair per column of the transposed copy [N, M / 2]: the
//               K-major operand of the weight-gradient GEMMs.
// Input rows are grouped (G rows per group in the input, Gp in the output, zero padding rows)
// and optionally cut at a device-side row count (rows at or beyond it read as zero).
#include "kernels.cuh"
#include "nvfp4.cuh"

namespace moe {

namespace {

constexpr int QT_ROWS = 128;
constexpr int QT_COLS = 64;
constexpr int QT_LD = 144;  // bytes per staged row: 128 + 16
constexpr int QT_THREADS = 128;

// Stage one tile: 128 rows x 8 pieces of 16 bytes, 8 consecutive threads a row's 128 bytes;
// a zero row (group padding or past the row limit) copies nothing and reads no global memory.
MOE_DEVICE void stage_tile(const Nvfp4QuantArgs& p, const uint16_t* in, int64_t tile_i,
                           int64_t ntc, int64_t limit, uint32_t dst, int t) {
  const int64_t r0 = (tile_i / ntc) * QT_ROWS;
  const int64_t c0 = (tile_i % ntc) * QT_COLS;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int v = t + QT_THREADS * i;
    const int r = v >> 3, piece = v & 7;
    const int64_t orow = r0 + r;
    const int64_t g = orow / p.Gp, gi = orow - g * p.Gp;
    const bool live = gi < p.G && orow < limit;
    const uint16_t* src = live ? in + (g * p.G + gi) * p.N + c0 + piece * 8 : in;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst + r * QT_LD +
                                                                          piece * 16),
                 "l"(src), "r"(live ? 16 : 0)
                 : "memory");
  }
}

__global__ void __launch_bounds__(QT_THREADS, 6) nvfp4_quantize_kernel(const Nvfp4QuantArgs p) {
  MOE_GRIDDEP_ENTRY();
  // two tile buffers: the next tile streams in while this one is quantised
  __shared__ __align__(16) uint8_t tiles[2][QT_ROWS * QT_LD];
  __shared__ float enc_row[128], enc_col[128];
  const int t = threadIdx.x;
  const int64_t ntr = p.M / QT_ROWS, ntc = p.N / QT_COLS;
  const int64_t ntiles = ntr * ntc;
  const int64_t limit = p.row_limit ? (int64_t)*p.row_limit : p.M;
  const float s_row = p.q_row ? nvfp4_encode_scale(*p.amax_row) : 0.f;
  const float s_col = p.q_col ? nvfp4_encode_scale(*p.amax_col) : 0.f;
  nvfp4_fill_enc_table(enc_row, s_row, t, QT_THREADS);
  nvfp4_fill_enc_table(enc_col, s_col, t, QT_THREADS);  // visible after the first barrier
  const uint16_t* in = static_cast<const uint16_t*>(p.in);
  if ((int64_t)blockIdx.x < ntiles)
    stage_tile(p, in, blockIdx.x, ntc, limit, smem_u32(tiles[0]), t);
  asm volatile("cp.async.commit_group;" ::: "memory");
  int k = 0;
  for (int64_t tile_i = blockIdx.x; tile_i < ntiles; tile_i += gridDim.x, ++k) {
    const int64_t next = tile_i + gridDim.x;
    if (next < ntiles) stage_tile(p, in, next, ntc, limit, smem_u32(tiles[(k + 1) & 1]), t);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    const int64_t r0 = (tile_i / ntc) * QT_ROWS;
    const int64_t c0 = (tile_i % ntc) * QT_COLS;
    const uint8_t* tile = tiles[k & 1];
    __syncthreads();
    if (p.q_row) {
      const uint8_t* src = tile + t * QT_LD;
      uint32_t codes[8], scales = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint4 w0 = *reinterpret_cast<const uint4*>(src + 32 * b);
        const uint4 w1 = *reinterpret_cast<const uint4*>(src + 32 * b + 16);
        const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        uint32_t q[2];
        scales |= nvfp4_quant16_bf16(w, s_row, enc_row, q) << (8 * b);
        codes[2 * b] = q[0];
        codes[2 * b + 1] = q[1];
      }
      const int64_t row = r0 + t;
      st_global_v8(p.q_row + row * (p.N / 2) + c0 / 2, codes);
      *reinterpret_cast<uint32_t*>(p.s_row + sf_mma_offset(row, c0 / 16, p.s_row_pad)) = scales;
    }
    if (p.q_col) {
      // thread t: columns 2 (t % 32) and 2 (t % 32) + 1, rows 32 (t / 32) .. + 31 (two blocks
      // of 16 per column, the two columns as fp32 pairs); a warp's 32-bit reads of one staged
      // row are 128 contiguous bytes
      const int cp = t & 31, h = t >> 5;
      const uint8_t* src = tile + (h * 32) * QT_LD + 4 * cp;
      uint32_t codes[2][4], scales[2] = {0, 0};
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        uint64_t x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(src + (16 * b + i) * QT_LD);
          x[i] = pack_f32x2(bf16_lo(w), bf16_hi(w));
        }
        if (p.rht) rht16_pair(x, p.rht_mask);
        uint32_t qa[2], qb[2];
        const uint32_t sc = nvfp4_quant16_pair(x, s_col, enc_col, qa, qb);
        scales[0] |= (sc & 0xFFu) << (8 * b);
        scales[1] |= (sc >> 8) << (8 * b);
        codes[0][2 * b] = qa[0];
        codes[0][2 * b + 1] = qa[1];
        codes[1][2 * b] = qb[0];
        codes[1][2 * b + 1] = qb[1];
      }
      const int64_t rr = r0 + h * 32;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int64_t col = c0 + 2 * cp + k;
        *reinterpret_cast<uint4*>(p.q_col + col * (p.M / 2) + rr / 2) =
            make_uint4(codes[k][0], codes[k][1], codes[k][2], codes[k][3]);
        *reinterpret_cast<uint16_t*>(p.s_col + sf_mma_offset(col, rr / 16, p.s_col_pad)) =
            (uint16_t)scales[k];
      }
    }
    // every thread is done with this buffer before the next iteration refills it
    __syncthreads();
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Plain amax of n bf16 values (n a multiple of 8, 16-byte aligned).
__global__ void __launch_bounds__(256) nvfp4_amax_kernel(const uint4* in, int64_t n8, float* out) {
  MOE_GRIDDEP_ENTRY();
  float m = 0.f;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 w = in[i];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(ws[j])), fabsf(bf16_hi(ws[j]))));
  }
  amax_flush_warp(m, out);
}

// amax and amax of the 16-row-block rotation along the rows of a bf16 [M, N] matrix (M a
// multiple of 16, N of 64, N / 128 < 65536). A CTA of 8 warps covers 128 rows (grid x) x 128
// columns (grid y): lane l of warp w takes columns 4l .. 4l+3 of rows 16w .. 16w+15 (8-byte
// loads, 256 contiguous bytes a warp and row).
__global__ void __launch_bounds__(256) nvfp4_rht_amax_kernel(const uint16_t* in, int64_t M,
                                                             int64_t N, uint32_t mask,
                                                             float* out, float* out_rht) {
  MOE_GRIDDEP_ENTRY();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t c = blockIdx.y * 128 + 4 * lane;
  const int64_t r0 = blockIdx.x * 128 + w * 16;
  float m = 0.f, mr = 0.f;
  if (r0 < M && c < N) {
    uint2 raw[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) raw[i] = *reinterpret_cast<const uint2*>(in + (r0 + i) * N + c);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t word = (k < 2) ? raw[i].x : raw[i].y;
        v[i] = (k & 1) ? bf16_hi(word) : bf16_lo(word);
        m = fmaxf(m, fabsf(v[i]));
      }
      rht16_regs(v, mask);
#pragma unroll
      for (int i = 0; i < 16; ++i) mr = fmaxf(mr, fabsf(v[i]));
    }
  }
  amax_flush_warp(m, out);
  amax_flush_warp(mr, out_rht);
}

// Gather for an NVFP4 layer: x_perm[r] = x[token(r)] (zero for padding rows), as the plain
// gather, plus the amax of x_perm and of its 16-row-block rotation, so that no separate pass
// reads x_perm for them. A CTA takes 16 consecutive rows (one rotation block; R_cap is a
// multiple of 128); thread t copies the 16-byte column pieces t, t + 256, ... of the 16 rows
// and rotates its 8 columns as four fp32 pairs.
__global__ void __launch_bounds__(256) gather_rows_amax_kernel(const uint4* __restrict__ x,
                                                               const int32_t* __restrict__ src_of,
                                                               const int32_t* __restrict__ offsets,
                                                               int E, int k, int H8, int64_t R_cap,
                                                               uint32_t mask,
                                                               uint4* __restrict__ out,
                                                               float* amax, float* amax_rht) {
  MOE_GRIDDEP_ENTRY();
  __shared__ int64_t src_row[16];
  const int used = offsets[E];
  float m = 0.f, mr = 0.f;
  for (int64_t r0 = (int64_t)blockIdx.x * 16; r0 < R_cap; r0 += (int64_t)gridDim.x * 16) {
    __syncthreads();  // the previous block's rows are no longer read
    if (threadIdx.x < 16) {
      const int64_t r = r0 + threadIdx.x;
      const int src = r < used ? src_of[r] : -1;
      src_row[threadIdx.x] = src >= 0 ? (int64_t)(src / k) : -1;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < H8; i += blockDim.x) {
      uint4 v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int64_t sr = src_row[j];
        v[j] = sr >= 0 ? x[sr * H8 + i] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) out[(r0 + j) * H8 + i] = v[j];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint64_t col[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t word = w == 0 ? v[j].x : w == 1 ? v[j].y : w == 2 ? v[j].z : v[j].w;
          const float lo = bf16_lo(word), hi = bf16_hi(word);
          m = fmaxf(m, fmaxf(fabsf(lo), fabsf(hi)));
          col[j] = pack_f32x2(lo, hi);
        }
        rht16_pair(col, mask);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          mr = fmaxf(mr, fmaxf(fabsf(f32x2_lo(col[j])), fabsf(f32x2_hi(col[j]))));
      }
    }
  }
  amax_flush_warp(m, amax);
  amax_flush_warp(mr, amax_rht);
}

}  // namespace

void launch_gather_rows_amax(const void* x, const int32_t* src_of, const int32_t* offsets, int E,
                             int k, int H, int64_t R_cap, uint32_t mask, void* out, float* amax,
                             float* amax_rht, int num_sms, int kid, cudaStream_t s) {
  const int64_t blocks = R_cap / 16;
  if (blocks <= 0) return;
  const int grid = (int)std::min<int64_t>(blocks, (int64_t)std::max(num_sms, 1) * 8);
  launch_kernel(gather_rows_amax_kernel, grid, 256, 0, s, nullptr, 0, static_cast<const uint4*>(x), src_of, offsets, E,
                                               k, H / 8, R_cap, mask, static_cast<uint4*>(out),
                                               amax, amax_rht);
  count_launch(s, kid);
}

bool nvfp4_quantize_shape_ok(int64_t M, int64_t N) {
  return M > 0 && N > 0 && M % QT_ROWS == 0 && N % QT_COLS == 0;
}

int64_t nvfp4_sf_bytes(int64_t rows, int64_t cols) {
  // slabs of 64 elements, plus four: a 256-element k-block fetches four slabs from the one it
  // starts in, and may start in the last; plus 1 KB for a 256-row B fetch past the end
  const int64_t slabs = (cols + 63) / 64 + 4;
  return slabs * ((rows + 127) / 128 * 128) * 4 + 1024;
}

void launch_nvfp4_quantize(const Nvfp4QuantArgs& a, int num_sms, cudaStream_t s) {
  const int64_t tiles = (a.M / QT_ROWS) * (a.N / QT_COLS);
  if (tiles <= 0) return;
  // 36 KB of tile buffers a CTA: six CTAs per SM
  const int grid = (int)std::min<int64_t>(tiles, (int64_t)std::max(num_sms, 1) * 6);
  launch_kernel(nvfp4_quantize_kernel, grid, QT_THREADS, 0, s, nullptr, 0, a);
  count_launch(s, MOE_K_NVFP4_QUANTIZE);
}

void launch_nvfp4_amax(const void* in, int64_t n, float* out, int num_sms, cudaStream_t s) {
  const int64_t n8 = n / 8;
  if (n8 <= 0) return;
  const int grid = (int)std::min<int64_t>((n8 + 255) / 256, (int64_t)std::max(num_sms, 1) * 8);
  launch_kernel(nvfp4_amax_kernel, grid, 256, 0, s, nullptr, 0, static_cast<const uint4*>(in), n8, out);
  count_launch(s, MOE_K_NVFP4_AMAX);
}

void launch_nvfp4_rht_amax(const void* in, int64_t M, int64_t N, uint32_t mask, float* out,
                           float* out_rht, cudaStream_t s) {
  if (M <= 0 || N <= 0) return;
  const dim3 grid((unsigned)((M + 127) / 128), (unsigned)((N + 127) / 128));
  launch_kernel(nvfp4_rht_amax_kernel, grid, 256, 0, s, nullptr, 0, static_cast<const uint16_t*>(in), M, N, mask, out,
                                             out_rht);
  count_launch(s, MOE_K_NVFP4_AMAX);
}

}  // namespace moe
