// Declarations shared between the translation units of the library.
#pragma once

#include <algorithm>
#include <utility>

#include "common.cuh"

namespace moe {

// launch accounting and the optional event timeline (api.cu); kid is a moe_kernel_id_t
void count_launch(cudaStream_t s, int kid);

// Whether the kernels the current entry-point call enqueues are launched with programmatic
// stream serialization (desc->pdl; thread-local, set for the duration of the call by api.cu).
bool pdl_enabled();
// Launch `k` like <<<grid, block, smem, s>>>, with programmatic stream serialization when the
// current call asked for it (extra_attrs: further launch attributes, e.g. a cluster shape).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          const cudaLaunchAttribute* extra_attrs, int n_extra, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attrs[4];
  int n = 0;
  for (int i = 0; i < n_extra && n < 3; ++i) attrs[n++] = extra_attrs[i];
  if (pdl_enabled()) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}
// set the message returned by moe_last_error_string for this thread (api.cu)
void set_last_error(const char* msg);

// route.cu
__global__ void route_topk_kernel(const float* logits, int T, int E, int k, int32_t* ids,
                                  float* probs, int32_t* counts);
__global__ void assign_rows_kernel(const int32_t* ids, const float* probs, const int32_t* counts,
                                   int T, int E, int k, int align, int64_t R_cap,
                                   int32_t* offsets, int32_t* row_of, int32_t* src_of,
                                   float* row_prob, int* err);
__global__ void gather_rows_kernel(const uint4* x, const int32_t* src_of, const int32_t* offsets,
                                   int E, int k, int H8, int64_t R_cap, uint4* out);
__global__ void route_export_kernel(const int32_t* off_ws, int n_off, const int32_t* row_of_ws,
                                    int64_t n_row_of, const int32_t* src_of_ws,
                                    const float* prob_ws, int64_t n_rows, int64_t n_total,
                                    int32_t* off, int32_t* row_of, int32_t* src_of,
                                    float* row_prob);
__global__ void combine_rows_kernel(const uint4* in, const int32_t* row_of, int T, int k, int H8,
                                    uint4* out);
__global__ void dprob_reduce_kernel(const float* part, int nparts, const int32_t* row_of, int n,
                                    float* d_probs);
__global__ void pack_fc1_kernel(const uint16_t* src, uint16_t* dst, int E, int H, int F, int N1,
                                int gated, int ilv, int inverse);

__global__ void group_colsum_kernel(const float* part, int ld, int col0, int ncols,
                                    const int32_t* offsets, float* out);

// Sets a kernel's dynamic shared-memory limit once per (kernel, device); thread-safe. The
// attribute belongs to the device's context, so a process driving several GPUs sets it on each.
cudaError_t ensure_smem_attr(const void* kernel, int bytes);
// clusters of two CTAs of `kernel` (launched with `cfg`) that fit on the device at once, cached
// per (kernel, device); 0 when the query fails
int max_resident_pairs(const void* kernel, const cudaLaunchConfig_t* cfg);

// mxfp8.cu
// Sizes the quantiser's 32-bit tile indexing covers (M rows < 2^31, tile count < 2^31).
bool mxfp8_quantize_size_ok(int64_t M, int64_t N);
// column-wise blocks restarting at device-resident group offsets; s_col [N, scale_cols]
int64_t mxfp8_grouped_scale_cols(int64_t M, int G);
void launch_mxfp8_colwise_grouped(const void* in, int64_t M, int64_t N, const int32_t* offsets,
                                  int G, uint8_t* q_col, uint8_t* s_col, int num_sms,
                                  cudaStream_t s);
void launch_mxfp8_quantize(const void* in, int64_t M, int64_t N, int rowwise, int colwise,
                           uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                           int num_sms, cudaStream_t s);
// Operand quantisation for the block-scaled GEMM: input rows grouped by G (output stride Gp,
// padding rows zero), scales in the MMA slab layout (rows padded to 128). A NULL q_row or
// q_col skips that direction.
void launch_mxfp8_quantize_mma(const void* in, int64_t M, int64_t N, int64_t G, int64_t Gp,
                               uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                               int num_sms, cudaStream_t s);

// gemm.cu --------------------------------------------------------------------------------
struct ActDev {
  int kind;  // moe_activation_t
  float beta, gate_max, lin_lo, lin_hi, lin_offset;
};

enum GemmRole {
  ROLE_FC1_FPROP = 0,   // Z = X W1 (+ GLU epilogue -> z, a_s)
  ROLE_FC2_FPROP = 1,   // Y = a_s W2
  ROLE_FC2_DGRAD = 2,   // dA_s = dY W2^T (+ dGLU epilogue -> dz, partial d_prob)
  ROLE_FC2_WGRAD = 3,   // dW2_e = a_s^T dY
  ROLE_FC1_DGRAD = 4,   // dX = dZ W1^T
  ROLE_FC1_WGRAD = 5    // dW1_e = dZ^T X (stored [N1, H])
};

struct GemmProblem {
  int role;
  int E, H, F, N1;
  int64_t R_cap;
  const int32_t* offsets;  // [E+1] device
  // operands (bf16)
  const void* x_perm;      // [R_cap, H]
  const void* w1p;         // [E, N1, H]
  const void* w2;          // [E, F, H]
  const void* a_s;         // [R_cap, F]
  const void* dy_perm;     // [R_cap, H]
  const void* dz;          // [R_cap, N1]
  const void* z;           // [R_cap, N1] (saved, dGLU epilogue input)
  const float* row_prob;   // [R_cap]
  // outputs
  void* out;               // role output (z, y_perm, dz, dW2, dx_perm, dW1)
  void* out2;              // FC1: a_s
  float* dprob_part;       // FC2 dgrad: [R_cap, nparts]
  // epilogue extras (BF16 gated; NULL when absent): FC1 bias [E, N1] logical order, feature
  // scale [E, F]; FC2 dgrad writes per-32-row column sums into ext_part [R_cap/32, N1 + F]
  const float* fc1_bias;
  const float* fscale;
  float* ext_part;
  int gated, ilv;
  ActDev act;
  int* err;
  int num_ctas;            // persistent grid size (SMs - margin)
  int64_t rows_per_expert; // T_max * k / E: the routed rows an expert averages at capacity
  // failure-detection self-test only: the TMA producer issues no loads (stall_loads = 1), so
  // every consumer wait runs out, after wait_ns (0: the default limit)
  int stall_loads;
  uint64_t wait_ns;
};

int gemm_bn(int role);
// gemm_rc.cu: FC2 dgrad + dGLU with the FC1 output recomputed in the same kernel (BF16)
int dprob_parts_recompute(int F);
cudaError_t launch_fc2_dgrad_recompute(const GemmProblem& p, cudaStream_t s);
int dprob_parts(int F);  // partial d_prob columns per row written by the FC2 dgrad epilogue
cudaError_t launch_grouped_gemm(const GemmProblem& p, cudaStream_t s);

// gemm_mx.cu ------------------------------------------------------------------------------
// One MXFP8 GEMM operand: E4M3 codes [rows, cols] (cols = the reduction dimension) and its
// scales in the MMA slab layout with rows padded to s_pad (a multiple of 128).
struct MxOperand {
  uint8_t* q;
  uint8_t* s;
  int64_t rows, cols, s_pad;
};

struct MxProblem {
  int role;  // GemmRole
  int E, H, F, N1, N1p, Fp;  // N1p, Fp: per-expert weight rows padded to 128
  int64_t R_cap;             // rows of every permuted buffer (multiple of 128)
  const int32_t* offsets;    // [E+1], segments 128-row aligned
  // row-wise (K = last dim, read K-major) and column-wise (source layout, read MN-major)
  // copies of each GEMM input
  MxOperand x, xt, a, at, dy, dyt, dz, dzt, w1, w1t, w2, w2t;
  const float* row_prob;
  const void* z;             // bf16 [R_cap, N1] saved FC1 output
  void* out;                 // bf16 role output (z for FC1, y_perm, dx_perm, dW2, dW1)
  float* dprob_part;
  // epilogue extras (gated layers; NULL when absent): FC1 bias [E, N1] in logical [gate |
  // linear] order and feature scale [E, F], fp32; per-32-row column sums of dZ and of
  // p * dA_s * a written by the dGLU epilogue into ext_part [R_cap / 32, N1 + F]
  const float* fc1_bias;
  const float* fscale;
  float* ext_part;
  int gated, ilv;
  ActDev act;
  int* err;
  int num_ctas;
  int64_t rows_per_expert;   // T_max * k / E: the routed rows an expert averages at capacity
};

int dprob_parts_mx(int F);
cudaError_t launch_grouped_gemm_mx(const MxProblem& p, cudaStream_t s);
// FC2 dgrad that recomputes the FC1 output next to dA_s (MXFP8 operands, gated activations)
int dprob_parts_mx_recompute(int F);
cudaError_t launch_fc2_dgrad_recompute_mx(const MxProblem& p, cudaStream_t s);

// nvfp4.cu --------------------------------------------------------------------------------
// NVFP4 quantiser arguments: in bf16 [G-row groups of the input, N]; output rows M = groups *
// Gp (padding rows zero), rows at or beyond *row_limit (when given) zero. Row-wise copy
// q_row [M, N/2] + s_row (slab layout, rows padded to s_row_pad); transposed copy q_col
// [N, M/2] + s_col (rows N padded to s_col_pad), rotated along M when rht. NULL q_row / q_col
// skips that copy. amax_* are device pointers to the per-tensor amax of each copy.
struct Nvfp4QuantArgs {
  const void* in;
  int64_t M, N, G, Gp;
  const int32_t* row_limit;
  const float* amax_row;
  const float* amax_col;
  uint8_t* q_row;
  uint8_t* s_row;
  int64_t s_row_pad;
  uint8_t* q_col;
  uint8_t* s_col;
  int64_t s_col_pad;
  int rht;
  uint32_t rht_mask;
  int* err;  // device error word for a load that never lands (may be null)
};
bool nvfp4_quantize_shape_ok(int64_t M, int64_t N);  // M % 128 == 0, N % 64 == 0
// scale bytes of an NVFP4 GEMM operand [rows, cols] in the slab layout, with the slack the
// 256-element k-blocks and 256-row B fetches of the FP4 GEMM read past the end
int64_t nvfp4_sf_bytes(int64_t rows, int64_t cols);
// false (nothing launched) unless Gp % 128 == 0, M % Gp == 0 and 0 < G <= Gp, or when the
// tensor map or the shared-memory limit cannot be set
bool launch_nvfp4_quantize(const Nvfp4QuantArgs& a, int num_sms, cudaStream_t s);
// amax of n bf16 values (n % 8 == 0) max-merged into *out (caller zeroes it)
void launch_nvfp4_amax(const void* in, int64_t n, float* out, int num_sms, cudaStream_t s);
// NVFP4 layers: the gather of route / backward (x_perm[r] = x[token(r)], padding rows zero)
// fused with the amax and the 16-row rotated amax of its output, max-merged into *amax and
// *amax_rht (R_cap a multiple of 16, H of 8); kid is the launch's moe_kernel_id_t
void launch_gather_rows_amax(const void* x, const int32_t* src_of, const int32_t* offsets, int E,
                             int k, int H, int64_t R_cap, uint32_t mask, void* out, float* amax,
                             float* amax_rht, int num_sms, int kid, cudaStream_t s);
// amax and amax of the 16-row Hadamard rotation along the rows of [M, N] (M % 16 == 0,
// N % 64 == 0), max-merged into *out and *out_rht
void launch_nvfp4_rht_amax(const void* in, int64_t M, int64_t N, uint32_t mask, float* out,
                           float* out_rht, cudaStream_t s);

// gemm_fp4.cu -----------------------------------------------------------------------------
// Per-tensor amax slots of an NVFP4 layer (workspace nv_amax), in the public order.
enum Nvfp4AmaxSlot {
  AM_X = 0, AM_XT = 1, AM_W1 = 2, AM_W2 = 3, AM_A = 4, AM_AT = 5, AM_DY = 6, AM_DYT = 7,
  AM_DZ = 8, AM_DZT = 9, AM_COUNT = 10
};

// An NVFP4 GEMM operand reuses MxOperand: q = packed E2M1 codes [rows, cols/2] (the reduction
// dimension cols innermost, read K-major), s = E4M3 scales in the slab layout (16-element
// blocks), rows padded to s_pad.
struct Fp4Problem {
  int role;  // GemmRole
  int E, H, F, N1, N1p, Fp;
  int64_t R_cap;
  const int32_t* offsets;
  // row-wise copies (K = the row) and transposed copies (rows = features, K = tokens or the
  // weight's other dimension); every copy is K-major
  MxOperand x, xt, a, at, dy, dyt, dz, dzt, w1, w1t, w2, w2t;
  float* amax;               // [AM_COUNT] per-tensor amax slots
  const float* row_prob;
  const void* z;             // bf16 [R_cap, N1] saved FC1 output (dGLU input)
  void* out;                 // bf16 role output (z for FC1, y_perm, dz, dx_perm, dW2, dW1)
  void* out2;                // FC1: bf16 a_s [R_cap, F]
  float* dprob_part;
  int gated, ilv;
  uint32_t rht_mask;
  ActDev act;
  int* err;
  int num_ctas;
  // epilogue extras (gated; NULL when absent): FC1 bias [E, N1] logical order, feature scale
  // [E, F]; FC2 dgrad writes per-32-row column sums into ext_part [R_cap/32, N1 + F]
  const float* fc1_bias;
  const float* fscale;
  float* ext_part;
};
int dprob_parts_fp4(int F);
cudaError_t launch_grouped_gemm_fp4(const Fp4Problem& p, cudaStream_t s);
// FC2 dgrad + dActivation with the FC1 output recomputed from the NVFP4 copies of X and W1
// (activation recomputation); dZ, its amaxes and the d_prob partials as the saved-Z kernel
int dprob_parts_fp4_recompute(int F);
cudaError_t launch_fc2_dgrad_recompute_fp4(const Fp4Problem& p, cudaStream_t s);

}  // namespace moe
