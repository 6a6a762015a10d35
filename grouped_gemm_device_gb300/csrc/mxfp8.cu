// MXFP8 quantiser ([TE-MoE] Challenge 2 and Figure 3: E4M3 elements, one E8M0 scale per 32
// contiguous values). Scale exponent e = clamp(floor(log2 amax) - 8, -127, 127) (-127 for an
// all-zero block), element = E4M3(v * 2^-e) rounded to nearest even with saturation.
//
// One CTA quantises 64x64 tiles (grid-stride): the tile is staged in shared memory, threads
// 0..127 produce the row-wise blocks (64 rows x 2 blocks) and threads 128..255 the
// column-wise blocks (64 columns x 2 blocks) written transposed, so each output block is one
// contiguous 32-byte run in global memory.
#include "kernels.cuh"

namespace moe {

// Quantise 32 fp32 values (one block) into 32 E4M3 bytes (as 8 words) and return the scale
// byte.
MOE_DEVICE uint32_t mx_quant_block(const float (&v)[32], uint32_t (&q)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int e = mx_block_exponent(amax);
  const float inv = mx_inv_scale(e);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t lo = cvt_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv);
    uint32_t hi = cvt_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv);
    q[i] = lo | (hi << 16);
  }
  return (uint32_t)(e + 127);
}

__global__ void __launch_bounds__(256) mxfp8_quantize_kernel(
    const uint16_t* __restrict__ in, int64_t M, int64_t N, int rowwise, int colwise,
    uint8_t* __restrict__ q_row, uint8_t* __restrict__ s_row, uint8_t* __restrict__ q_col,
    uint8_t* __restrict__ s_col) {
  __shared__ __align__(16) uint16_t tile[64][64 + 8];
  const int64_t tiles_m = (M + 63) / 64, tiles_n = (N + 63) / 64;
  const int tid = threadIdx.x;
  for (int64_t t = blockIdx.x; t < tiles_m * tiles_n; t += gridDim.x) {
    const int64_t r0 = (t / tiles_n) * 64, c0 = (t % tiles_n) * 64;
    __syncthreads();
    // stage: 64 rows x 8 uint4 (8 bf16 each); out-of-range parts are zero
    for (int i = tid; i < 64 * 8; i += 256) {
      const int rr = i >> 3, cc = (i & 7) * 8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r0 + rr < M && c0 + cc < N)
        v = *reinterpret_cast<const uint4*>(in + (r0 + rr) * N + c0 + cc);
      *reinterpret_cast<uint4*>(&tile[rr][cc]) = v;
    }
    __syncthreads();
    float v[32];
    uint32_t q[8];
    if (tid < 128) {
      const int rr = tid >> 1, blk = tid & 1;
      const int64_t row = r0 + rr, col = c0 + blk * 32;
      if (rowwise && row < M && col < N) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          v[i] = __uint_as_float((uint32_t)tile[rr][blk * 32 + i] << 16);
        uint32_t s = mx_quant_block(v, q);
        uint4* dst = reinterpret_cast<uint4*>(q_row + row * N + col);
        dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
        dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
        s_row[row * (N / 32) + col / 32] = (uint8_t)s;
      }
    } else {
      const int cc = (tid - 128) & 63, rb = (tid - 128) >> 6;
      const int64_t col = c0 + cc, row = r0 + rb * 32;
      if (colwise && col < N && row < M) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          v[i] = __uint_as_float((uint32_t)tile[rb * 32 + i][cc] << 16);
        uint32_t s = mx_quant_block(v, q);
        uint4* dst = reinterpret_cast<uint4*>(q_col + col * M + row);
        dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
        dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
        s_col[col * (M / 32) + row / 32] = (uint8_t)s;
      }
    }
  }
}

void launch_mxfp8_quantize(const void* in, int64_t M, int64_t N, int rowwise, int colwise,
                           uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                           int num_sms, cudaStream_t s) {
  const int64_t tiles = ((M + 63) / 64) * ((N + 63) / 64);
  if (tiles == 0) return;
  int grid = (int)std::min<int64_t>(tiles, (int64_t)num_sms * 8);
  mxfp8_quantize_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(in), M, N, rowwise,
                                             colwise, q_row, s_row, q_col, s_col);
  count_launch(s, MOE_K_MXFP8_QUANTIZE);
}

}  // namespace moe
