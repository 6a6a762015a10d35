/*
 * moegmm.h - C ABI of the GB300 (sm_103a) fused grouped expert MLP of a Mixture-of-Experts
 * layer: routing + permutation, fused FC1 -> GLU -> probability scale -> FC2 forward, the
 * matching backward (BF16, MXFP8 or NVFP4 GEMM operands), and the standalone MXFP8 and NVFP4
 * quantisers.
 *
 * Sources (by page title and section):
 *   [NV-blog] NVIDIA technical blog "Boosting MoE Training Throughput with Advanced Fusion
 *             Kernels" (zh-cn 借助高级融合内核提高 MoE 训练吞吐量): the three fused kernel
 *             families (GroupGemm + quantise; GroupGemm + activation + quantise/transpose;
 *             GroupGemm + dActivation + quantise/transpose), the SwiGLU equation and GLU weight
 *             repacking (GLU-epilogue section, Figure 2), device-resident per-group token
 *             counts (host-sync section), fused MXFP8 quantisation, dynamic scheduling and the
 *             configurable SM margin (kernel-to-pretraining section).
 *   [TE-MoE]  "NVIDIA Transformer Engine 优化 MoE 生物基础模型训练" (Transformer Engine MoE
 *             article): GroupedLinear with per-expert token counts, the per-expert loop with
 *             index_add (Challenge 1), MXFP8 format (Challenge 2, Figure 3), ScaledSwiGLU and
 *             the fused GroupedLinear -> ScaledSwiGLU -> GroupedLinear op (Challenge 3, Fig. 4).
 *   NVFP4 is named by [NV-blog] ("fused MXFP8 and NVFP4 quantisation": the forward kernel
 *   emits BF16 output plus a per-tensor amax, the backward kernel the amax of the
 *   Hadamard-rotated transposed output) but not defined there; the published format is used:
 *   E2M1 values, one unsigned E4M3 scale per 16 values, one fp32 scale per tensor (below).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers unless a name says host. Layouts are row-major.
 *     bf16 is passed as void* (2-byte IEEE bfloat16), e4m3 and e8m0 as uint8_t.
 *   - The caller owns every buffer, including the workspace `ws` (size from
 *     moe_workspace_size). No entry point allocates device memory or synchronises the host;
 *     all work is enqueued on `stream` (NULL = legacy default stream), so whole layer steps can
 *     be captured in a CUDA graph. Token counts and offsets never leave the device.
 *   - Host-side argument checks run before any launch and return MOE_ERR_INVALID_ARG or
 *     MOE_ERR_UNSUPPORTED with nothing enqueued. A CUDA launch error returns MOE_ERR_CUDA.
 *     Conditions only the device can see (routing capacity overflow, a bounded wait that timed
 *     out inside a kernel) set a sticky error word in the workspace, read by moe_get_error.
 *     No kernel traps, asserts or spins without a bound.
 *   - moe_last_error_string() describes the most recent host-side failure of this thread.
 */
#ifndef MOEGMM_H_
#define MOEGMM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers (same underlying type). */
typedef struct CUstream_st *moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer, k > E, ... */
  MOE_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. H not a multiple of 64)   */
  MOE_ERR_WORKSPACE = 3,    /* ws_bytes smaller than moe_workspace_size                  */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed                       */
  MOE_ERR_DEVICE = 5        /* moe_get_error found a device-side error code               */
} moe_status_t;

/* Device error word codes (sticky until moe_clear_error). */
#define MOE_DEVERR_NONE 0
#define MOE_DEVERR_CAPACITY 1   /* routed rows exceeded the static capacity R_cap        */
#define MOE_DEVERR_TIMEOUT 2    /* a bounded barrier wait in a GEMM kernel gave up       */
#define MOE_DEVERR_BAD_ID 3     /* an expert id outside [0, E)                            */

/* GEMM operand precision. BF16: bf16 operands. MXFP8: E4M3 with one E8M0 scale per 32 values
 * (see mxfp8_quantize). NVFP4: E2M1 with one E4M3 scale per 16 values and one fp32 scale per
 * tensor (see nvfp4_quantize); the weight-gradient operands are Hadamard-rotated along the
 * tokens first (desc.rht_mask). Outputs and the saved FC1 output are bf16 in every case. */
typedef enum { MOE_PREC_BF16 = 0, MOE_PREC_MXFP8 = 1, MOE_PREC_NVFP4 = 2 } moe_precision_t;

/* Activations of [NV-blog] (SwiGLU, GeGLU, sReLU, "with clamp and scale options"):
 *   SWIGLU          a = lin * g * sigmoid(beta*g)                  (SwiGLU equation, b=c=0)
 *   CLAMPED_SWIGLU  g' = min(g, gate_max), l' = clamp(lin, lin_lo, lin_hi),
 *                   a = (l' + lin_offset) * g' * sigmoid(beta*g')
 *   GEGLU           a = lin * g * Phi(g)                           (exact erf GELU)
 *   SRELU           a = max(z, 0)^2, non-gated: FC1 has F (not 2F) output columns
 * The gradient passes a clamp at equality (the clamp is active strictly beyond a limit). */
typedef enum {
  MOE_ACT_SWIGLU = 0,
  MOE_ACT_CLAMPED_SWIGLU = 1,
  MOE_ACT_GEGLU = 2,
  MOE_ACT_SRELU = 3
} moe_activation_t;

/* Static description of one layer. Capacities are fixed here so that every call has the
 * same launch shapes (graph-capturable); the per-call token count T must be <= T_max. */
typedef struct {
  int32_t E;          /* experts (1..256)                                                */
  int32_t k;          /* experts per token (1..min(E,8))                                 */
  int32_t H;          /* hidden size, multiple of 64                                     */
  int32_t F;          /* expert FFN width, multiple of 64                                */
  int32_t T_max;      /* token capacity                                                  */
  int32_t precision;  /* moe_precision_t                                                 */
  int32_t activation; /* moe_activation_t                                                */
  float beta;         /* Swish beta (1.0 SwiGLU, 1.702 clamped GPT-OSS form)             */
  float gate_max;     /* clamped SwiGLU: upper clamp of the gate                         */
  float lin_lo;       /* clamped SwiGLU: lower clamp of the linear half                  */
  float lin_hi;       /* clamped SwiGLU: upper clamp of the linear half                  */
  float lin_offset;   /* clamped SwiGLU: added to the clamped linear half                */
  int32_t sm_margin;  /* SMs left free for concurrent kernels ([NV-blog] cluster margin) */
  int32_t ilv;        /* gate/linear interleave block of the packed W1 (32, 64 or 128)   */
  int32_t align;      /* expert segment alignment in rows: 32, 64 or 128 (BF16); 128
                         (MXFP8, NVFP4: segments start on 128-row scale slabs)            */
  int32_t recompute;  /* 1: keep no FC1 output between forward and backward; the FC2-dgrad
                         kernel recomputes it ([NV-blog] "What's next": activation
                         recomputation). Any precision and activation; 0 otherwise      */
  int32_t extras;     /* epilogue extras ([NV-blog] GLU-epilogue section: bias-vector addition
                         and feature scaling): bit 0 FC1 bias, bit 1 per-feature scale of the
                         activation output; used through the _ex entry points. Any
                         precision with a gated activation, without recompute; 0 otherwise */
  uint32_t rht_mask;  /* NVFP4: signs of the 16-point random Hadamard rotation applied along
                         the tokens to the weight-gradient operands (bit j set: the j-th row
                         of each 16-row block is negated before H16 / 4); drawn once by the
                         caller. Ignored by the other precisions                             */
  int32_t reuse_weights; /* MXFP8 / NVFP4: 1 = the forward does not quantise W1 and W2 again
                         but uses the block-scaled weight copies (and, NVFP4, their per-tensor
                         amaxes) that an earlier forward on the same workspace made from the
                         same BF16 master weights - the micro-batches of one gradient
                         accumulation step share them ([TE-MoE] Challenge 2: BF16 master
                         weights quantised before the low-precision GEMMs). The caller
                         guarantees the weights did not change since. 0 = quantise (always
                         correct). Ignored by BF16 layers                                    */
  int32_t pdl;        /* 1: every kernel the call enqueues is launched with programmatic stream
                         serialization (programmatic dependent launch), so that a kernel's CTAs
                         are scheduled while the previous kernel's last CTAs finish and only its
                         data reads wait for that kernel; 0: ordinary stream order. Results
                         are the same either way                                              */
} moe_layer_desc_t;

/* Byte offsets (from ws) of the intermediates that live in the workspace, for inspection
 * and tests. Offsets that do not apply to the layer's precision are SIZE_MAX. R_cap =
 * T_max*k + E*(align-1) rows. All row-indexed buffers use the permuted row order:
 * expert ascending, token ascending within an expert, each expert's segment starting at a
 * multiple of `align`; padding rows are zero and have probability 0. */
typedef struct {
  size_t total;          /* == moe_workspace_size                                        */
  int64_t R_cap;         /* row capacity                                                 */
  size_t err;            /* int32 device error word                                      */
  size_t offsets;        /* int32 [E+1] padded segment starts; offsets[E] = rows in use  */
  size_t row_of;         /* int32 [T_max*k] row of (token t, slot j) at t*k+j            */
  size_t src_of;         /* int32 [R_cap] t*k+j of a row, -1 for padding                 */
  size_t row_prob;       /* fp32 [R_cap] routing probability of a row, 0 for padding     */
  size_t x_perm;         /* bf16 [R_cap, H] gathered tokens                              */
  size_t z;              /* bf16 [R_cap, N1] FC1 output saved for backward (packed cols);
                            SIZE_MAX when the layer recomputes it                        */
  size_t a_s;            /* bf16 [R_cap, F] p * act(z), the FC2 input                    */
  size_t y_perm;         /* bf16 [R_cap, H] FC2 output before combine (shared with dx_perm) */
  size_t dy_perm;        /* bf16 [R_cap, H] gathered upstream gradient                   */
  size_t dz;             /* bf16 [R_cap, N1] gradient of z (packed cols)                 */
  size_t dx_perm;        /* bf16 [R_cap, H] FC1 dgrad output before combine              */
  size_t dprob_part;     /* fp32 [R_cap, ceil(F/128)] per-column-tile partial d_prob     */
  size_t ext_part;       /* fp32 [R_cap/32, N1 + F] per-32-row column sums of dZ and of
                            p * dA_s * a (extras only; SIZE_MAX otherwise)                 */
  size_t mx_base;        /* start of the MXFP8 operand copies (MXFP8 layers only)        */
  size_t nv_amax;        /* NVFP4 only: fp32 [16] per-tensor amax of each NVFP4 copy, in the
                            order x, x^T (rotated), W1, W2, a_s, a_s^T (rotated), dY, dY^T
                            (rotated), dZ, dZ^T (rotated); SIZE_MAX otherwise               */
  size_t nv_base;        /* start of the NVFP4 operand copies (NVFP4 layers only)        */
} moe_ws_layout_t;

/* Workspace bytes for a layer (0 if the description is invalid). */
size_t moe_workspace_size(const moe_layer_desc_t *desc);
/* Fill *out with the workspace layout. */
moe_status_t moe_workspace_layout(const moe_layer_desc_t *desc, moe_ws_layout_t *out);

/* Route + permute ([TE-MoE] Figure 1 top-k router; [NV-blog] host-sync section: per-group
 * token counts stay in device memory).
 *   logits     fp32 [T, E]   router logits
 *   x          bf16 [T, H]   tokens
 *   topk_ids   int32 [T, k]  out: experts by descending logit, ties to the lower index
 *   topk_probs fp32 [T, k]   out: softmax over the k chosen logits
 *   counts     int32 [E]     out: tokens routed to each expert
 * Writes offsets, row_of, src_of, row_prob and x_perm (and, for MXFP8 layers, the MXFP8
 * row-wise and column-wise copies of x_perm; for NVFP4 layers the amax and rotated amax of
 * x_perm, taken during the gather, and its row-wise and rotated transposed NVFP4 copies) into
 * ws. T in [0, T_max]. */
moe_status_t moe_route_permute(const moe_layer_desc_t *desc, int32_t T, const float *logits,
                               const void *x, int32_t *topk_ids, float *topk_probs,
                               int32_t *counts, void *ws, size_t ws_bytes, moe_stream_t stream);

/* The routing maps of the last moe_route_permute on ws, copied into caller buffers (device
 * memory; [NV-blog] host-sync section: the per-expert counts and offsets stay on the device):
 *   offsets  int32 [E+1]    padded segment starts; offsets[E] = rows in use
 *   row_of   int32 [T*k]    permuted row of (token t, slot j) at t*k+j
 *   src_of   int32 [R_cap]  t*k+j of a permuted row, -1 for a padding row
 *   row_prob fp32  [R_cap]  routing probability of a permuted row, 0 for a padding row
 * R_cap as in moe_workspace_layout; rows at or beyond offsets[E] carry no routing (their
 * src_of / row_prob entries are left from earlier calls). Any of the four may be NULL (not
 * copied); each one given
 * must be 4-byte aligned. T must be the T of that moe_route_permute call, in [0, T_max]. One
 * kernel on `stream`, no host synchronisation, graph-capturable. Returns MOE_ERR_INVALID_ARG
 * for a bad description, workspace, T or pointer. */
moe_status_t moe_route_export(const moe_layer_desc_t *desc, const void *ws, size_t ws_bytes,
                              int32_t T, int32_t *offsets, int32_t *row_of, int32_t *src_of,
                              float *row_prob, moe_stream_t stream);

/* Fused grouped MLP forward ([NV-blog] kernel families 1 and 2, Figure 1; [TE-MoE]
 * GroupedLinear -> ScaledSwiGLU -> GroupedLinear):
 *   Z = X_e W1_e (FC1, grouped over experts from the device offsets), a = act(Z),
 *   a_s = p * a, Y_e = a_s W2_e (FC2), y[t] = sum_j Y[row_of[t,j]].
 *   w1_packed bf16 [E, N1, H]  FC1 weight, N1 = 2F (gated) or F (sReLU), rows in the packed
 *                              order of moe_pack_fc1_weight (gate/linear blocks interleaved)
 *   w2        bf16 [E, F, H]   FC2 weight (logical [F, H] per expert)
 *   y         bf16 [T, H]      out
 * Requires a preceding moe_route_permute on the same ws. Saves z and a_s in ws for the
 * backward. MXFP8 layers also quantise both weights (both directions) into ws first. NVFP4
 * layers take the weights' amax and NVFP4 copies (both directions) first; their FC1 kernel
 * also writes the amax and the rotated amax of a_s into ws (nv_amax), from which a_s's NVFP4
 * copies are made for FC2 and for the FC2 weight gradient. */
moe_status_t moe_grouped_mlp_fwd(const moe_layer_desc_t *desc, int32_t T, const void *w1_packed,
                                 const void *w2, void *y, void *ws, size_t ws_bytes,
                                 moe_stream_t stream);

/* Fused grouped MLP backward ([NV-blog] kernel family 3: FC2 dgrad + dActivation +
 * quantise/transpose; unfused weight-gradient GEMMs, Figure 1):
 *   dA_s = dY W2^T;  d_prob = sum_f dA_s * a;  dA = p * dA_s;  dZ = dact(Z, dA);
 *   dW2_e = a_s^T dY_e;  dW1_e = X_e^T dZ_e;  dX = dZ W1^T;  dx[t] = sum_j dX[row_of[t,j]].
 *   dy         bf16 [T, H]       upstream gradient of y
 *   dx         bf16 [T, H]       out
 *   dw1_packed bf16 [E, N1, H]   out, same packed row order as w1_packed (an expert with no
 *                                tokens gets exact zeros)
 *   dw2        bf16 [E, F, H]    out
 *   d_probs    fp32 [T, k]       out, gradient of topk_probs
 * Requires the forward's ws contents. NVFP4 layers gather dY together with its amax and
 * rotated amax, and their FC2-dgrad kernel writes dZ with its amax and rotated amax; every
 * GEMM then reads NVFP4 copies, the weight-gradient operands rotated along the tokens. */
moe_status_t moe_grouped_mlp_bwd(const moe_layer_desc_t *desc, int32_t T, const void *dy,
                                 const void *w1_packed, const void *w2, void *dx,
                                 void *dw1_packed, void *dw2, float *d_probs, void *ws,
                                 size_t ws_bytes, moe_stream_t stream);

/* Forward and backward with the epilogue extras (desc->extras; [NV-blog] GLU-epilogue
 * section: bias-vector addition and feature scaling; the SwiGLU equation's b and c):
 *   Z = X_e W1_e + b1_e (the bias in logical [gate | linear] column order, saved with Z),
 *   a_s = p * s_e * act(Z)  (s the per-feature scale of the activation output);
 *   backward: dA = p * s * dA_s, d_prob = sum_f dA_s * s * a,
 *             d_fc1_bias_e = sum over the expert's rows of dZ,
 *             d_feat_scale_e = sum over the expert's rows of p * dA_s * a.
 *   fc1_bias     fp32 [E, N1] logical order (bit 0 of extras; NULL otherwise)
 *   feat_scale   fp32 [E, F]  (bit 1; NULL otherwise)
 *   d_fc1_bias   fp32 [E, N1] out (bit 0; NULL otherwise)
 *   d_feat_scale fp32 [E, F]  out (bit 1; NULL otherwise)
 * Other arguments as moe_grouped_mlp_fwd / moe_grouped_mlp_bwd, which return
 * MOE_ERR_UNSUPPORTED for a layer with extras. The backward needs no bias (Z includes it).
 * Layers with a gated activation (BF16, MXFP8, NVFP4); in MXFP8 the scaled activation is
 * what the FC1 epilogue quantises, in NVFP4 what it emits in BF16 (with its amaxes), and the
 * dGLU epilogue takes the two column sums from the fp32 values, before dZ is rounded. */
moe_status_t moe_grouped_mlp_fwd_ex(const moe_layer_desc_t *desc, int32_t T,
                                    const void *w1_packed, const void *w2,
                                    const float *fc1_bias, const float *feat_scale, void *y,
                                    void *ws, size_t ws_bytes, moe_stream_t stream);
moe_status_t moe_grouped_mlp_bwd_ex(const moe_layer_desc_t *desc, int32_t T, const void *dy,
                                    const void *w1_packed, const void *w2,
                                    const float *feat_scale, void *dx, void *dw1_packed,
                                    void *dw2, float *d_probs, float *d_fc1_bias,
                                    float *d_feat_scale, void *ws, size_t ws_bytes,
                                    moe_stream_t stream);

/* Route + permute without any device allocation and without a workspace. The pages have no
 * counterpart of this entry point; it exists for callers that cannot call cudaMalloc, such as
 * plugins hosted by a framework that owns the whole device memory pool and forbids
 * allocations of its own, or code that runs where an allocation would stall or is not
 * allowed (for example while a CUDA graph is being recorded).
 * It computes the same results as moe_route_permute (topk_ids, topk_probs, counts, and the
 * gathered tokens) but writes the padded offsets and the gathered tokens to caller buffers:
 *   offsets  int32 [E+1]                  out: padded expert segment starts
 *   x_perm   bf16  [x_perm_rows, H]       out: x_perm_rows >= T_max*k + E*(align-1); same
 *                                          rows as moe_route_permute's workspace x_perm
 * Its scratch (row map, per-row source and probability, an error word) is a fixed
 * file-scope device array of about 1.6 MB inside the library, held by every GPU that loads
 * the library until the process exits. Limit: T_max*k <= 131072 routed (token, expert)
 * pairs, which with E <= 256 and any segment alignment (32, 64, 128) keeps R_cap within the
 * array's 163584 rows; larger descriptions return MOE_ERR_UNSUPPORTED before any launch. Only
 * BF16 layers. The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current, and looks it up again when the device's
 * context has changed since (after cudaDeviceReset, for example); make the first call after
 * such a change before any stream capture. All calls on a device share the array and it keeps
 * the last call's contents: the
 * error word and counts are cleared at the start of every call, and calls whose execution
 * overlaps on the GPU (for example on two streams) race. Capacity errors detected on the
 * device are not reported by this entry point (they cannot occur when T <= T_max). */
moe_status_t moe_route_permute_noalloc(const moe_layer_desc_t *desc, int32_t T,
                                       const float *logits, const void *x, int32_t *topk_ids,
                                       float *topk_probs, int32_t *counts, int32_t *offsets,
                                       void *x_perm, int64_t x_perm_rows, moe_stream_t stream);

/* Standalone MXFP8 quantiser ([TE-MoE] Challenge 2, Figure 3: E4M3 elements with one E8M0
 * scale per 32 contiguous values):
 *   scale exponent e = clamp(floor(log2(amax)) - 8, -127, 127) (e = -127 when amax = 0),
 *   scale byte e + 127, q = E4M3(v / 2^e) rounded to nearest even, saturating at +-448.
 *   in      bf16 [M, N]
 *   rowwise:  q_row  e4m3 [M, N]       blocks of 32 along N; s_row e8m0 [M, N/32]
 *   colwise:  q_col  e4m3 [M, N]       blocks of 32 along M (same layout as in);
 *             s_col  e8m0 [N, M/32]    without groups: blocks start at every 32nd row
 *   group_offsets  int32 [num_groups + 1], DEVICE memory, or NULL: rows [off[g], off[g+1])
 *             form group g (off[0] = 0, non-decreasing, off[num_groups] = M; the per-expert
 *             token counts of a GroupedLinear, [TE-MoE] Challenge 1, need not be multiples
 *             of 32). Column-wise blocks then restart at each group's first row: block i of
 *             group g is rows off[g] + 32i .. min(off[g] + 32i + 32, off[g+1]) (a short last
 *             block is quantised as if padded with zeros), and
 *             s_col e8m0 [N, nb], nb = 4 * ceil((ceil(M/32) + num_groups) / 4): the scale of
 *             column c, block (g, i) is s_col[c * nb + off[g]/32 + g + i] (integer division);
 *             entries no block owns are written 0. The offsets are read on the device only
 *             (no host sync); offsets outside [0, M] are clamped, and offsets that break the
 *             rules above give unspecified (but in-bounds) results. The row-wise copy does not
 *             depend on the groups. num_groups must be in [1, 65536] when group_offsets is set.
 * N must be a multiple of 32; M a multiple of 32 for colwise without groups (any M with
 * groups); in and q_col 16-byte aligned and s_col 4-byte aligned with groups; the pointers of
 * an unused direction may be NULL. Bit-exact: the result does not depend on the launch. */
moe_status_t mxfp8_quantize(const void *in, int64_t M, int64_t N, int32_t rowwise,
                            int32_t colwise, const int32_t *group_offsets, int32_t num_groups,
                            uint8_t *q_row, uint8_t *s_row, uint8_t *q_col, uint8_t *s_col,
                            moe_stream_t stream);

/* NVFP4 per-tensor amax ([NV-blog] "fused MXFP8 and NVFP4 quantisation": the scale of an NVFP4
 * tensor needs its amax first).
 *   in        bf16 [M, N]
 *   amax      fp32 [1] out: max |in|
 *   amax_rht  fp32 [1] out (may be NULL): max |y| over y = (1/4) H16 diag(d) x for every
 *             column and every block of 16 consecutive rows (x the block's 16 values, H16
 *             the Sylvester Hadamard matrix, d_j = -1 where bit j of sign_mask is set)
 * Both outputs are overwritten (the call zeroes them first). N must be a multiple of 64 (and
 * below 64 * 65536); M a multiple of 16 when amax_rht is given. M = 0 gives 0. */
moe_status_t nvfp4_amax(const void *in, int64_t M, int64_t N, uint32_t sign_mask, float *amax,
                        float *amax_rht, moe_stream_t stream);

/* Standalone NVFP4 quantiser. Per tensor S = min(2688 / amax, FLT_MAX) (2688 = 6 * 448); per
 * block of 16 values s_b = E4M3(fp32(amax_b / 6) * S) (round to nearest even, saturating);
 * per value q = E2M1(v * fp32(S / s_b)) (nearest even, saturating at +-6; factor 0 when
 * s_b = 0). Each step is one IEEE fp32 operation. The value represented is E2M1(q) * s_b / S.
 *   in        bf16 [M, N]
 *   amax_row  fp32 [1] device: the amax S is computed from for the row-wise copy
 *   amax_col  fp32 [1] device: the same for the transposed copy (the rotated amax when rht)
 *   row-wise:    q_row  [M, N/2] bytes, two E2M1 codes a byte (even index in the low nibble),
 *                       blocks of 16 along N;
 *                s_row  E4M3 scales in the MMA slab layout: the scale of (row r, block j) at
 *                       byte ((j/4) * M + perm(r)) * 4 + j%4, perm(r) = (r & ~127) |
 *                       ((r & 31) << 2) | ((r >> 5) & 3); (N/64) * M * 4 bytes
 *   transposed:  q_col  [N, M/2] bytes: row n holds column n of in, blocks of 16 along M,
 *                       each block first rotated as in nvfp4_amax when rht != 0;
 *                s_col  slab layout of (row n, block j): (M/64) * round128(N) * 4 bytes
 * M must be a positive multiple of 128 and N of 64; q_row and q_col 32-byte aligned, s_row
 * and s_col 4-byte aligned. q_row/s_row or q_col/s_col may both be NULL to skip that copy (its
 * amax pointer may then be NULL). Bit-exact: the result does not depend on the launch. */
moe_status_t nvfp4_quantize(const void *in, int64_t M, int64_t N, const float *amax_row,
                            const float *amax_col, int32_t rht, uint32_t sign_mask,
                            uint8_t *q_row, uint8_t *s_row, uint8_t *q_col, uint8_t *s_col,
                            moe_stream_t stream);

/* GLU weight repacking ([NV-blog] GLU-epilogue section and Figure 2: the gate and linear
 * columns are repacked so one output tile holds half a tile of each; done once, before
 * training or at checkpoint load).
 *   forward (inverse = 0): w1_logical bf16 [E, H, N1] -> w1_packed bf16 [E, N1, H]
 *   inverse (inverse = 1): w1_packed -> w1_logical
 * Gated (N1 = 2F): packed row p belongs to block b = p / ilv; even blocks are gate columns
 * (b/2)*ilv + p%ilv, odd blocks the linear columns F + (b/2)*ilv + p%ilv. sReLU (N1 = F):
 * packed = transpose. ilv must be a multiple of 32 that divides F. */
moe_status_t moe_pack_fc1_weight(const void *w1_src, void *w1_dst, int32_t E, int32_t H,
                                 int32_t F, int32_t gated, int32_t ilv, int32_t inverse,
                                 moe_stream_t stream);

/* Enqueue a copy of the device error word into *host_code (pinned or pageable host int);
 * the value is valid once the stream has been synchronised. */
moe_status_t moe_get_error(const moe_layer_desc_t *desc, const void *ws, int32_t *host_code,
                           moe_stream_t stream);
/* Enqueue a reset of the device error word to MOE_DEVERR_NONE. */
moe_status_t moe_clear_error(const moe_layer_desc_t *desc, void *ws, moe_stream_t stream);

/* Failure-detection self-test (no counterpart on the pages; it exercises this library's own
 * bounded waits). Enqueues one kernel whose single barrier wait can never complete: the same
 * bounded wait the GEMM kernels use gives up after limit_ns nanoseconds (1 ms .. 10 s) and
 * writes MOE_DEVERR_TIMEOUT into *err (device int32; written only if it holds 0). The kernel
 * then returns normally, so the context stays usable; no fault, trap or endless loop is
 * involved. Returns MOE_ERR_INVALID_ARG for a NULL err or a limit outside the range. */
moe_status_t moe_selftest_wait_timeout(int32_t *err, uint64_t limit_ns, moe_stream_t stream);

/* Failure-detection self-test of a GEMM kernel itself (no counterpart on the pages). For a BF16
 * layer whose moe_route_permute (and forward) ran on ws, enqueues the FC2 forward grouped GEMM
 * (a_s x W2 -> the workspace's permuted output; w2 as for moe_grouped_mlp_fwd) with its TMA
 * producer issuing no loads. Every MMA and epilogue wait of the kernel then runs out after
 * limit_ns nanoseconds (1 ms .. 10 s): the CTA raises its abort flag, MOE_DEVERR_TIMEOUT goes
 * into the workspace error word (moe_get_error; moe_clear_error resets it), every role leaves
 * its loop, TMEM is freed and the kernel returns, so the context stays usable. The permuted
 * output in the workspace is left undefined until the next forward. Returns
 * MOE_ERR_UNSUPPORTED for a non-BF16 layer, MOE_ERR_INVALID_ARG for a bad description,
 * workspace, w2 or limit. */
moe_status_t moe_selftest_gemm_timeout(const moe_layer_desc_t *desc, void *ws, size_t ws_bytes,
                                       const void *w2, uint64_t limit_ns, moe_stream_t stream);

/* Number of SMs the persistent GEMM uses on the current device for this description
 * (device SM count minus sm_margin, at least 1). */
int32_t moe_gemm_ctas(const moe_layer_desc_t *desc);

/* Kernels this library enqueued on any stream since load (a monotonically increasing
 * host-side counter, for launch accounting). */
uint64_t moe_launch_count(void);

/* Kernel identifiers reported by the launch timeline. */
typedef enum {
  MOE_K_ROUTE_TOPK = 0,
  MOE_K_ASSIGN_ROWS = 1,
  MOE_K_GATHER_X = 2,
  MOE_K_GEMM_FC1_FPROP = 3,
  MOE_K_GEMM_FC2_FPROP = 4,
  MOE_K_COMBINE_Y = 5,
  MOE_K_GATHER_DY = 6,
  MOE_K_GEMM_FC2_DGRAD = 7,
  MOE_K_DPROB_REDUCE = 8,
  MOE_K_GEMM_FC2_WGRAD = 9,
  MOE_K_GEMM_FC1_DGRAD = 10,
  MOE_K_COMBINE_DX = 11,
  MOE_K_GEMM_FC1_WGRAD = 12,
  MOE_K_MXFP8_QUANTIZE = 13,
  MOE_K_PACK_FC1 = 14,
  MOE_K_EXTRAS_REDUCE = 15,
  MOE_K_NVFP4_AMAX = 16,
  MOE_K_NVFP4_QUANTIZE = 17,
  MOE_K_ROUTE_EXPORT = 18,
  MOE_K_COUNT = 19
} moe_kernel_id_t;

/* Launch timeline, for measurement. Between moe_timeline_begin and moe_timeline_end the
 * library records events[i] (caller-created cudaEvent_t handles, passed as void*) on the
 * launching stream right after its i-th kernel launch, for i < capacity, and remembers the
 * kernel's moe_kernel_id_t. Kernels of one stream run in order, so the elapsed time between
 * consecutive events is the duration of the later kernel. Process-wide; not thread-safe.
 * moe_timeline_end copies the ids into kernel_ids (capacity entries, may be NULL), stops
 * recording and returns how many events were recorded. */
moe_status_t moe_timeline_begin(void *const *events, int32_t capacity);
int32_t moe_timeline_end(int32_t *kernel_ids);

/* Human-readable message for the last host-side error of the calling thread. */
const char *moe_last_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* MOEGMM_H_ */
