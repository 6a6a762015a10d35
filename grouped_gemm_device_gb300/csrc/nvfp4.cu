// NVFP4 quantiser and per-tensor amax kernels (scaling rule and layouts in nvfp4.cuh).
//
// [NV-blog] section "fused MXFP8 and NVFP4 quantisation": the quantisation of an NVFP4 GEMM
// operand needs the tensor's amax before any block can be encoded, so it is a second pass over
// a BF16 tensor whose amax is already known: for the FC1 output a_s and for dZ the GEMM
// epilogues provide it; for the routed input, dY and the weights the amax kernels below do.
//
// Quantiser: a persistent CTA of 128 threads walks 128-row x 64-column tiles of a bf16 matrix.
// Tiles arrive by TMA (one 3-D box {64, 128, 1} over [groups][G][N], 128-byte swizzle) into a
// ring of shared-memory stages (two per CTA, three or five CTAs per SM); group padding rows are the box's out-of-bounds rows (zero
// filled) and rows at or beyond the device-side row count are zeroed in shared memory, so no
// global memory is read for them. Thread t then quantises
//   row-wise    row t's 64 values (four 16-blocks along the row, the reduction dimension of
//               the row-grouped GEMMs) into one 32-byte run and one 32-bit word of scales;
//   transposed  columns 2 (t % 32), 2 (t % 32) + 1 over rows 32 (t / 32) .. + 31 (two 16-blocks
//               along the rows per column, optionally Hadamard-rotated first) for the transposed
//               copy [N, M / 2], the K-major operand of the weight-gradient GEMMs. Its codes and
//               scales go through a shared-memory buffer so that each column leaves as whole
//               32-byte runs and each scale as a whole 32-bit word.
// Input rows are grouped (G rows per group in the input, Gp in the output, Gp a multiple of
// 128) and optionally cut at a device-side row count (rows at or beyond it read as zero).
#include "gemm_common.cuh"
#include "nvfp4.cuh"

namespace moe {

namespace {

constexpr int QT_ROWS = 128;
constexpr int QT_COLS = 64;
constexpr int QT_THREADS = 128;
constexpr int QT_TILE_BYTES = QT_ROWS * QT_COLS * 2;  // 16 KB: 128 rows of 128 bytes

template <int STAGES>
struct QtSmem {
  uint8_t tile[STAGES][QT_TILE_BYTES];  // 1024-byte aligned (the swizzle atom)
  // transposed codes of a tile, two buffers: row j holds columns 2j and 2j + 1 (64 bytes
  // each), its 16-byte pieces XOR-swizzled by (j mod 8)
  uint8_t colq[2][32 * 128];
  uint16_t cols[2][2][64][2];  // transposed scales: [buffer][slab][column][half word]
  float enc_row[128], enc_col[128];
  uint64_t full[STAGES];
  int abort;
};
template <int STAGES>
constexpr int qt_smem_bytes() { return (int)sizeof(QtSmem<STAGES>) + 1024; }

struct QtArgs {
  Nvfp4QuantArgs a;
  CUtensorMap tm;  // input as [groups][G][N] bf16, box {64, 128, 1}, 128-byte swizzle
};

// 16 butterflies of the Hadamard rotation on column pairs whose signs are already applied;
// the same fp32 operations as rht16_pair after its sign step.
MOE_DEVICE void rht16_pair_signed(uint64_t (&x)[16]) {
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

template <int STAGES>
__global__ void __launch_bounds__(QT_THREADS) nvfp4_quantize_kernel(const __grid_constant__ QtArgs q) {
  MOE_GRIDDEP_ENTRY();
  const Nvfp4QuantArgs& p = q.a;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  QtSmem<STAGES>& sm =
      *reinterpret_cast<QtSmem<STAGES>*>(smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr));
  const int t = threadIdx.x;
  const int64_t ntc = p.N / QT_COLS;
  const int64_t ntiles = (p.M / QT_ROWS) * ntc;
  const int64_t limit = p.row_limit ? (int64_t)*p.row_limit : p.M;
  const float s_row = p.q_row ? nvfp4_encode_scale(*p.amax_row) : 0.f;
  const float s_col = p.q_col ? nvfp4_encode_scale(*p.amax_col) : 0.f;
  nvfp4_fill_enc_table(sm.enc_row, s_row, t, QT_THREADS);
  nvfp4_fill_enc_table(sm.enc_col, s_col, t, QT_THREADS);
  if (t == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&sm.full[s], 1);
    sm.abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&q.tm);
  }
  __syncthreads();
  // thread 0: bring tile `ti` into stage s (a tile wholly at or beyond the row count is only
  // marked arrived: its stage is zeroed instead)
  auto issue = [&](int64_t ti, int s) {
    const int64_t r0 = (ti / ntc) * QT_ROWS, c0 = (ti % ntc) * QT_COLS;
    if (r0 >= limit) {
      mbar_arrive(&sm.full[s]);
      return;
    }
    mbar_arrive_expect_tx(&sm.full[s], QT_TILE_BYTES);
    tma_load_3d(sm.tile[s], &q.tm, &sm.full[s], (int)c0, (int)(r0 % p.Gp), (int)(r0 / p.Gp));
  };
  if (t == 0)
    for (int s = 0; s < STAGES; ++s) {
      const int64_t ti = blockIdx.x + (int64_t)s * gridDim.x;
      if (ti < ntiles) issue(ti, s);
    }
  const uint32_t sign_mask = p.rht ? p.rht_mask : 0u;
  volatile int* abort = &sm.abort;
  int k = 0;
  for (int64_t tile_i = blockIdx.x; tile_i < ntiles; tile_i += gridDim.x, ++k) {
    const int s = k % STAGES;
    const int64_t r0 = (tile_i / ntc) * QT_ROWS;
    const int64_t c0 = (tile_i % ntc) * QT_COLS;
    uint8_t* tile = sm.tile[s];
    const bool ok = mbar_wait(&sm.full[s], (uint32_t)(k / STAGES) & 1u, abort, p.err);
    if (r0 + QT_ROWS > limit) {  // CTA-uniform: rows at or beyond the row count read as zero
      if (t >= limit - r0) {
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(tile + t * 128 + c * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
    }
    if (__syncthreads_or(!ok)) {
      // give up: wait (bounded) for the loads still in flight, then leave
      if (t == 0) {
        int own_abort = 0;
        for (int j = k; j < k + STAGES; ++j) {
          const int64_t ti = blockIdx.x + (int64_t)j * gridDim.x;
          if (ti < ntiles)
            mbar_wait(&sm.full[j % STAGES], (uint32_t)(j / STAGES) & 1u, &own_abort,
                      nullptr);
        }
      }
      return;
    }
    if (p.q_row) {
      const uint8_t* src = tile + t * 128;
      uint32_t codes[8], scales = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint4 w0 = *reinterpret_cast<const uint4*>(src + (((2 * b) ^ (t & 7)) << 4));
        const uint4 w1 = *reinterpret_cast<const uint4*>(src + (((2 * b + 1) ^ (t & 7)) << 4));
        const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        uint32_t qq[2];
        scales |= nvfp4_quant16_bf16(w, s_row, sm.enc_row, qq) << (8 * b);
        codes[2 * b] = qq[0];
        codes[2 * b + 1] = qq[1];
      }
      const int64_t row = r0 + t;
      st_global_v8(p.q_row + row * (p.N / 2) + c0 / 2, codes);
      *reinterpret_cast<uint32_t*>(p.s_row + sf_mma_offset(row, c0 / 16, p.s_row_pad)) = scales;
    }
    uint8_t* cq = sm.colq[k & 1];
    if (p.q_col) {
      // thread t: columns 2 cp, 2 cp + 1 (a 32-bit word of each staged row) over rows
      // 32 h .. 32 h + 31; a warp's reads of one row cover its 128 bytes once
      const int cp = t & 31, h = t >> 5;
      uint32_t codes[2][4], scales[2] = {0, 0};
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        uint64_t x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = h * 32 + 16 * b + i;  // r mod 8 == i mod 8
          uint32_t w = *reinterpret_cast<const uint32_t*>(
              tile + r * 128 + ((((cp >> 2) ^ (i & 7)) << 4) | ((cp & 3) << 2)));
          // the rotation's sign d_i flips both bf16 values (exactly the fp32 negation)
          w ^= (0u - ((sign_mask >> i) & 1u)) & 0x80008000u;
          x[i] = pack_f32x2(bf16_lo(w), bf16_hi(w));
        }
        if (p.rht) rht16_pair_signed(x);
        uint32_t qa[2], qb[2];
        const uint32_t sc = nvfp4_quant16_pair(x, s_col, sm.enc_col, qa, qb);
        scales[0] |= (sc & 0xFFu) << (8 * b);
        scales[1] |= (sc >> 8) << (8 * b);
        codes[0][2 * b] = qa[0];
        codes[0][2 * b + 1] = qa[1];
        codes[1][2 * b] = qb[0];
        codes[1][2 * b + 1] = qb[1];
      }
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        *reinterpret_cast<uint4*>(cq + cp * 128 + (((kk * 4 + h) ^ (cp & 7)) << 4)) =
            make_uint4(codes[kk][0], codes[kk][1], codes[kk][2], codes[kk][3]);
        sm.cols[k & 1][h >> 1][2 * cp + kk][h & 1] = (uint16_t)scales[kk];
      }
    }
    // stage s is consumed and the transposed buffer complete
    __syncthreads();
    if (t == 0) {
      const int64_t next = tile_i + (int64_t)STAGES * gridDim.x;
      if (next < ntiles) issue(next, s);
    }
    if (p.q_col) {
      // thread t: column c0 + j (j = t / 2), rows r0 + 64 (t % 2) .. + 63 as one 32-byte run
      const int j = t >> 1, half = t & 1, rho = j >> 1, kk = j & 1;
      const uint8_t* rowp = cq + rho * 128;
      const uint4 a = *reinterpret_cast<const uint4*>(rowp + (((kk * 4 + 2 * half) ^ (rho & 7)) << 4));
      const uint4 b =
          *reinterpret_cast<const uint4*>(rowp + (((kk * 4 + 2 * half + 1) ^ (rho & 7)) << 4));
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      st_global_v8(p.q_col + (c0 + j) * (p.M / 2) + r0 / 2 + half * 32, w);
      // thread t: the 32-bit scale word of column c0 + (t % 64) in slab r0 / 64 + t / 64
      const int slab = t >> 6, jj = t & 63;
      const uint32_t wd = (uint32_t)sm.cols[k & 1][slab][jj][0] |
                          ((uint32_t)sm.cols[k & 1][slab][jj][1] << 16);
      *reinterpret_cast<uint32_t*>(
          p.s_col + sf_mma_offset(c0 + jj, r0 / 16 + 4 * slab, p.s_col_pad)) = wd;
    }
  }
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

// STAGES tiles in flight per CTA, CTAS CTAs per SM
template <int STAGES, int CTAS>
bool launch_nvfp4_quantize_cfg(const Nvfp4QuantArgs& a, int num_sms, cudaStream_t s) {
  const int64_t tiles = (a.M / QT_ROWS) * (a.N / QT_COLS);
  if (tiles <= 0) return true;
  if (a.Gp <= 0 || a.Gp % QT_ROWS || a.M % a.Gp || a.G <= 0 || a.G > a.Gp) return false;
  QtArgs q;
  q.a = a;
  const uint64_t dims[3] = {(uint64_t)a.N, (uint64_t)a.G, (uint64_t)(a.M / a.Gp)};
  const uint64_t strides[2] = {(uint64_t)a.N * 2, (uint64_t)a.G * a.N * 2};
  const uint32_t box[3] = {QT_COLS, QT_ROWS, 1};
  if (!make_tmap(&q.tm, a.in, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
    return false;
  constexpr int smem = qt_smem_bytes<STAGES>();
  if (ensure_smem_attr(reinterpret_cast<const void*>(nvfp4_quantize_kernel<STAGES>), smem) !=
      cudaSuccess)
    return false;
  const int grid = (int)std::min<int64_t>(tiles, (int64_t)std::max(num_sms, 1) * CTAS);
  launch_kernel(nvfp4_quantize_kernel<STAGES>, grid, QT_THREADS, smem, s, nullptr, 0, q);
  count_launch(s, MOE_K_NVFP4_QUANTIZE);
  return true;
}

bool launch_nvfp4_quantize(const Nvfp4QuantArgs& a, int num_sms, cudaStream_t s) {
  // two stages a CTA; five CTAs (20 warps) per SM for the rotated copy, whose butterflies
  // make it issue-bound, three without the rotation (measured on GB300: 4.7 against 4.1 TB/s
  // for three CTAs of three stages on a rotated 33792 x 4096 tensor; 5.8-6.0 TB/s on the
  // unrotated Mixtral and GPT-OSS weights, where four CTAs lost up to 22% on the latter)
  return a.rht && a.q_col ? launch_nvfp4_quantize_cfg<2, 5>(a, num_sms, s)
                          : launch_nvfp4_quantize_cfg<2, 3>(a, num_sms, s);
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
