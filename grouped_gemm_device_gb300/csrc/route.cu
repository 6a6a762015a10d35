// Routing and data-movement kernels of the expert layer (all HBM- or latency-bound):
//   route_topk_kernel      top-k over fp32 logits, softmax over the chosen k, expert histogram
//   assign_rows_kernel     padded offsets (exclusive scan) and the stable (expert, token) order
//   gather_rows_kernel     x_perm[r] = x[token(r)] (zero for padding rows)
//   combine_rows_kernel    out[t] = sum_j in[row_of[t, j]] in fp32, j ascending
//   dprob_reduce_kernel    d_probs[t, j] = sum over column tiles of the partial d_prob
//   pack_fc1_kernel        GLU weight repacking ([NV-blog] GLU-epilogue section, Figure 2)
//   group_colsum_kernel    per-expert sums of the dGLU epilogue's per-32-row column sums
//                          (the FC1 bias and feature-scale gradients)
// Sources: [TE-MoE] Figure 1 (top-2 router, weighted sum) and Challenge 1 (per-expert loop
// with index_add: the row order here is the order torch.where visits tokens); [NV-blog]
// host-sync section (per-group token counts kept in device memory).
#include "kernels.cuh"

namespace moe {

// One warp per token. Each lane keeps E/32 logits; k rounds of a warp arg-max pick the
// experts (larger logit first, ties to the lower index). Probabilities are the softmax over
// the chosen logits. Expert counts are accumulated in a block histogram, then globally.
// Non-finite logits: a NaN is read as -inf, so every round picks an untaken expert in [0, E)
// (its arg-max starts from -inf, which any untaken expert equals or beats); a chosen logit
// equal to the chosen maximum gets weight 1 (exp(0) for finite ones), which is the limit of
// the softmax when the maximum is +inf (shared among the +inf ones) or -inf (uniform).
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T,
                                                         int E, int k, int32_t* __restrict__ ids,
                                                         float* __restrict__ probs,
                                                         int32_t* __restrict__ counts) {
  MOE_GRIDDEP_ENTRY();
  __shared__ int hist[256];
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warps_per_block = blockDim.x >> 5;
  const int per_lane = (E + 31) >> 5;  // <= 8
  for (int t = blockIdx.x * warps_per_block + (threadIdx.x >> 5); t < T;
       t += gridDim.x * warps_per_block) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int e = i * 32 + lane;
      const float lv = (i < per_lane && e < E) ? logits[(size_t)t * E + e] : -INFINITY;
      v[i] = lv == lv ? lv : -INFINITY;
    }
    bool taken[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) taken[i] = !(i < per_lane && i * 32 + lane < E);
    float sel_v[8];
    int sel_e[8];
    for (int j = 0; j < k; ++j) {
      // lane-local best
      float bv = -INFINITY;
      int be = 0x7FFFFFFF;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        int e = i * 32 + lane;
        if (!taken[i] && (v[i] > bv || (v[i] == bv && e < be))) {
          bv = v[i];
          be = e;
        }
      }
      // warp arg-max with index tie-break
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
        int oe = __shfl_xor_sync(0xFFFFFFFFu, be, off);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      sel_v[j] = bv;
      sel_e[j] = be;
      if ((be & 31) == lane) taken[be >> 5] = true;
    }
    if (lane == 0) {
      float m = sel_v[0];
      float w[8];
      float s = 0.f;
      for (int j = 0; j < k; ++j) {
        w[j] = sel_v[j] == m ? 1.0f : expf(sel_v[j] - m);
        s += w[j];
      }
      const float inv = 1.0f / s;
      for (int j = 0; j < k; ++j) {
        ids[(size_t)t * k + j] = sel_e[j];
        probs[(size_t)t * k + j] = w[j] * inv;
        atomicAdd(&hist[sel_e[j]], 1);
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x)
    if (hist[i]) atomicAdd(&counts[i], hist[i]);
}

// One block per expert e. Every block recomputes the padded exclusive scan of the counts
// (E <= 256) so no extra launch or grid sync is needed; block 0 publishes offsets[]. The
// block then walks all (token, slot) pairs in token order and gives the pairs routed to e
// consecutive rows (token ascending) by a block-wide prefix sum.
__global__ void __launch_bounds__(1024) assign_rows_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ probs,
    const int32_t* __restrict__ counts, int T, int E, int k, int align, int64_t R_cap,
    int32_t* __restrict__ offsets, int32_t* __restrict__ row_of, int32_t* __restrict__ src_of,
    float* __restrict__ row_prob, int* err) {
  MOE_GRIDDEP_ENTRY();
  __shared__ int s_off[257];
  __shared__ int s_warp[32];
  __shared__ int s_base;
  const int e = blockIdx.x;
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int i = 0; i < E; ++i) {
      s_off[i] = acc;
      int c = counts[i];
      acc += (c + align - 1) / align * align;
    }
    s_off[E] = acc;
    if (acc > R_cap) set_error(err, MOE_DEVERR_CAPACITY);
    s_base = 0;
  }
  __syncthreads();
  if (s_off[E] > R_cap) return;
  if (e == 0)
    for (int i = threadIdx.x; i <= E; i += blockDim.x) offsets[i] = s_off[i];
  const int off_e = s_off[e];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  // tokens per thread per chunk
  constexpr int TPT = 4;
  const int chunk = blockDim.x * TPT;
  for (int t0 = 0; t0 < T; t0 += chunk) {
    int my_slot[TPT];
    int my_cnt = 0;
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
      int t = t0 + threadIdx.x * TPT + i;
      my_slot[i] = -1;
      if (t < T) {
        for (int j = 0; j < k; ++j)
          if (ids[(size_t)t * k + j] == e) my_slot[i] = j;
        my_cnt += my_slot[i] >= 0;
      }
    }
    // block exclusive scan of my_cnt
    int incl = my_cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      int w = lane < nw ? s_warp[lane] : 0;
      int wi = w;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xFFFFFFFFu, wi, off);
        if (lane >= off) wi += o;
      }
      if (lane < nw) s_warp[lane] = wi - w;  // exclusive warp prefix
    }
    __syncthreads();
    int rank = s_base + s_warp[wid] + incl - my_cnt;
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
      if (my_slot[i] >= 0) {
        int t = t0 + threadIdx.x * TPT + i;
        int src = t * k + my_slot[i];
        int row = off_e + rank;
        row_of[src] = row;
        src_of[row] = src;
        row_prob[row] = probs[src];
        ++rank;
      }
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) s_base = rank;
    __syncthreads();
  }
  // padding rows of this expert's segment
  const int cnt = counts[e];
  const int end = s_off[e + 1];
  for (int r = off_e + cnt + threadIdx.x; r < end; r += blockDim.x) {
    src_of[r] = -1;
    row_prob[r] = 0.f;
  }
}

// Copies of the routing maps into caller buffers (any destination may be null).
__global__ void __launch_bounds__(256) route_export_kernel(
    const int32_t* __restrict__ off_ws, int n_off, const int32_t* __restrict__ row_of_ws,
    int64_t n_row_of, const int32_t* __restrict__ src_of_ws, const float* __restrict__ prob_ws,
    int64_t n_rows, int64_t n_total, int32_t* off, int32_t* row_of, int32_t* src_of,
    float* row_prob) {
  MOE_GRIDDEP_ENTRY();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_total; i += stride) {
    if (off && i < n_off) off[i] = off_ws[i];
    if (row_of && i < n_row_of) row_of[i] = row_of_ws[i];
    if (src_of && i < n_rows) src_of[i] = src_of_ws[i];
    if (row_prob && i < n_rows) row_prob[i] = prob_ws[i];
  }
}

// x_perm[r, :] = x[src_of[r] / k, :] for rows in use, zero for padding rows and for rows at
// or beyond offsets[E]. One block per row; 16-byte vectors.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ src_of,
                                                          const int32_t* __restrict__ offsets,
                                                          int E, int k, int H8, int64_t R_cap,
                                                          uint4* __restrict__ out) {
  MOE_GRIDDEP_ENTRY();
  const int used = offsets[E];
  for (int64_t r = blockIdx.x; r < R_cap; r += gridDim.x) {
    int src = r < used ? src_of[r] : -1;
    uint4* o = out + r * H8;
    if (src >= 0) {
      const uint4* in = x + (int64_t)(src / k) * H8;
      for (int i = threadIdx.x; i < H8; i += blockDim.x) o[i] = in[i];
    } else {
      for (int i = threadIdx.x; i < H8; i += blockDim.x) o[i] = make_uint4(0, 0, 0, 0);
    }
  }
}

// out[t, :] = sum_{j<k} in[row_of[t*k+j], :], fp32 accumulation in slot order, bf16 result.
__global__ void __launch_bounds__(256) combine_rows_kernel(const uint4* __restrict__ in,
                                                           const int32_t* __restrict__ row_of,
                                                           int T, int k, int H8,
                                                           uint4* __restrict__ out) {
  MOE_GRIDDEP_ENTRY();
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    int rows[8];
    for (int j = 0; j < k; ++j) rows[j] = row_of[(size_t)t * k + j];
    for (int i = threadIdx.x; i < H8; i += blockDim.x) {
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.f;
      for (int j = 0; j < k; ++j) {
        uint4 v = in[(int64_t)rows[j] * H8 + i];
        acc[0] += bf16_lo(v.x); acc[1] += bf16_hi(v.x);
        acc[2] += bf16_lo(v.y); acc[3] += bf16_hi(v.y);
        acc[4] += bf16_lo(v.z); acc[5] += bf16_hi(v.z);
        acc[6] += bf16_lo(v.w); acc[7] += bf16_hi(v.w);
      }
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      out[(int64_t)t * H8 + i] = o;
    }
  }
}

// d_probs[t*k+j] = sum_i part[row_of[t*k+j], i] (column tiles in order).
__global__ void dprob_reduce_kernel(const float* __restrict__ part, int nparts,
                                    const int32_t* __restrict__ row_of, int n,
                                    float* __restrict__ d_probs) {
  MOE_GRIDDEP_ENTRY();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const float* p = part + (int64_t)row_of[i] * nparts;
    float s = 0.f;
    for (int q = 0; q < nparts; ++q) s += p[q];
    d_probs[i] = s;
  }
}

// Packed row p of expert e <-> logical column c(p) of [H, N1]:
//   gated: block b = p / ilv; c = (b & 1) * F + (b >> 1) * ilv + p % ilv;  sReLU: c = p.
// forward: dst[e][p][h] = src[e][h][c(p)];  inverse: dst[e][h][c(p)] = src[e][p][h].
// 32x32 tiles through shared memory so both sides are read/written along rows.
__global__ void __launch_bounds__(256) pack_fc1_kernel(const uint16_t* __restrict__ src,
                                                       uint16_t* __restrict__ dst, int E, int H,
                                                       int F, int N1, int gated, int ilv,
                                                       int inverse) {
  MOE_GRIDDEP_ENTRY();
  __shared__ uint16_t tile[32][33];
  const int tiles_p = N1 / 32, tiles_h = H / 32;
  const int64_t per_e = (int64_t)tiles_p * tiles_h;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int64_t tix = blockIdx.x; tix < per_e * E; tix += gridDim.x) {
    const int e = (int)(tix / per_e);
    const int64_t rem = tix % per_e;
    const int p0 = (int)(rem / tiles_h) * 32, h0 = (int)(rem % tiles_h) * 32;
    // logical columns of packed rows p0..p0+31 are contiguous (ilv is a multiple of 32)
    int c0 = p0;
    if (gated) {
      int b = p0 / ilv;
      c0 = (b & 1) * F + (b >> 1) * ilv + p0 % ilv;
    }
    const uint16_t* s = src + (int64_t)e * H * N1;
    uint16_t* d = dst + (int64_t)e * H * N1;
    __syncthreads();
    if (!inverse) {
      for (int i = ty; i < 32; i += 8) tile[i][tx] = s[(int64_t)(h0 + i) * N1 + c0 + tx];
      __syncthreads();
      for (int i = ty; i < 32; i += 8) d[(int64_t)(p0 + i) * H + h0 + tx] = tile[tx][i];
    } else {
      for (int i = ty; i < 32; i += 8) tile[i][tx] = s[(int64_t)(p0 + i) * H + h0 + tx];
      __syncthreads();
      for (int i = ty; i < 32; i += 8) d[(int64_t)(h0 + i) * N1 + c0 + tx] = tile[tx][i];
    }
  }
}

}  // namespace moe

namespace moe {

// out[e][c] = sum over the 32-row groups g of expert e (g in [off[e]/32, off[e+1]/32); the
// segments are 32-row aligned) of part[g][col0 + c], for c < ncols. One thread per (column,
// expert), groups in ascending order: deterministic.
__global__ void __launch_bounds__(256) group_colsum_kernel(const float* __restrict__ part,
                                                           int ld, int col0, int ncols,
                                                           const int32_t* __restrict__ offsets,
                                                           float* __restrict__ out) {
  MOE_GRIDDEP_ENTRY();
  const int e = blockIdx.y;
  const int c = blockIdx.x * 256 + threadIdx.x;
  if (c >= ncols) return;
  const int g0 = offsets[e] >> 5, g1 = offsets[e + 1] >> 5;
  float acc = 0.f;
  for (int g = g0; g < g1; ++g) acc += part[(int64_t)g * ld + col0 + c];
  out[(int64_t)e * ncols + c] = acc;
}

}  // namespace moe
