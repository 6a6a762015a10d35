// C ABI of the library (declared in include/moegmm.h): host-side validation, workspace
// layout, and the launch sequences of routing, forward and backward. Nothing here allocates
// device memory or synchronises; everything is enqueued on the caller's stream.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <string>

#include "kernels.cuh"
#include "nvfp4.cuh"

namespace moe {

static std::atomic<uint64_t> g_launches{0};
static cudaEvent_t* g_tl_events = nullptr;
static int g_tl_cap = 0;
static int g_tl_n = 0;
static int g_tl_ids[4096];

// programmatic dependent launch for the kernels of the current entry-point call
static thread_local bool g_pdl = false;
bool pdl_enabled() { return g_pdl; }
namespace {
struct PdlScope {
  bool prev;
  explicit PdlScope(const moe_layer_desc_t* d) : prev(g_pdl) { g_pdl = d && d->pdl == 1; }
  ~PdlScope() { g_pdl = prev; }
};
}  // namespace

void count_launch(cudaStream_t s, int kid) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (g_tl_events && g_tl_n < g_tl_cap) {
    cudaEventRecord(g_tl_events[g_tl_n], s);
    g_tl_ids[g_tl_n++] = kid;
  }
}

static thread_local std::string g_last_error;

static moe_status_t fail(moe_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

void set_last_error(const char* msg) { g_last_error = msg; }

cudaError_t ensure_smem_attr(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kernel, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({kernel, dev});
  return e;
}

int max_resident_pairs(const void* kernel, const cudaLaunchConfig_t* cfg) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find({kernel, dev});
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t c = *cfg;
  c.gridDim = dim3(2, 1, 1);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &c) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of a failed query
    n = 0;
  }
  cache[{kernel, dev}] = n;
  return n;
}

static moe_status_t cuda_fail(cudaError_t e, const char* where) {
  return fail(MOE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

static int device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int64_t r_cap(const moe_layer_desc_t* d) {
  const int64_t r = (int64_t)d->T_max * d->k + (int64_t)d->E * (d->align - 1);
  // MXFP8 / NVFP4: every permuted buffer spans whole 128-row scale slabs
  return d->precision != MOE_PREC_BF16 ? (r + 127) / 128 * 128 : r;
}
static int64_t round128(int64_t v) { return (v + 127) / 128 * 128; }
static int n1_of(const moe_layer_desc_t* d) {
  return d->activation == MOE_ACT_SRELU ? d->F : 2 * d->F;
}

static moe_status_t validate_desc(const moe_layer_desc_t* d) {
  if (!d) return fail(MOE_ERR_INVALID_ARG, "desc is NULL");
  if (d->E < 1 || d->E > 256) return fail(MOE_ERR_INVALID_ARG, "E=%d outside [1,256]", d->E);
  if (d->k < 1 || d->k > 8 || d->k > d->E)
    return fail(MOE_ERR_INVALID_ARG, "k=%d must be in [1, min(E,8)]", d->k);
  if (d->H <= 0 || d->F <= 0 || d->T_max < 0)
    return fail(MOE_ERR_INVALID_ARG, "H, F must be positive and T_max >= 0");
  if (d->H % 64 || d->F % 64)
    return fail(MOE_ERR_UNSUPPORTED, "H=%d and F=%d must be multiples of 64", d->H, d->F);
  if (d->precision == MOE_PREC_BF16 && d->align != 32 && d->align != 64 && d->align != 128)
    return fail(MOE_ERR_UNSUPPORTED, "align must be 32, 64 or 128");
  if (d->precision == MOE_PREC_MXFP8 && d->align != 128)
    return fail(MOE_ERR_UNSUPPORTED, "MXFP8 layers need align = 128 (whole scale slabs)");
  if (d->precision == MOE_PREC_MXFP8 && d->activation != MOE_ACT_SRELU && d->ilv != 32 &&
      d->ilv != 64)
    return fail(MOE_ERR_UNSUPPORTED, "MXFP8 layers need ilv = 32 or 64");
  if (d->precision != MOE_PREC_BF16 && d->precision != MOE_PREC_MXFP8 &&
      d->precision != MOE_PREC_NVFP4)
    return fail(MOE_ERR_INVALID_ARG, "unknown precision %d", d->precision);
  if (d->precision == MOE_PREC_NVFP4 && d->align != 128)
    return fail(MOE_ERR_UNSUPPORTED, "NVFP4 layers need align = 128 (whole scale slabs)");
  if (d->precision == MOE_PREC_NVFP4 && d->activation != MOE_ACT_SRELU && d->ilv != 64)
    return fail(MOE_ERR_UNSUPPORTED, "NVFP4 layers need ilv = 64");
  if (d->activation < MOE_ACT_SWIGLU || d->activation > MOE_ACT_SRELU)
    return fail(MOE_ERR_INVALID_ARG, "unknown activation %d", d->activation);
  if (d->activation != MOE_ACT_SRELU) {
    if (d->ilv != 32 && d->ilv != 64 && d->ilv != 128)
      return fail(MOE_ERR_UNSUPPORTED, "ilv=%d must be 32, 64 or 128", d->ilv);
    if (d->F % d->ilv) return fail(MOE_ERR_UNSUPPORTED, "F must be a multiple of ilv");
  }
  if (d->sm_margin < 0) return fail(MOE_ERR_INVALID_ARG, "sm_margin must be >= 0");
  if (d->recompute != 0 && d->recompute != 1)
    return fail(MOE_ERR_INVALID_ARG, "recompute must be 0 or 1");
  if (d->extras & ~3) return fail(MOE_ERR_INVALID_ARG, "extras has unknown bits");
  if (d->reuse_weights != 0 && d->reuse_weights != 1)
    return fail(MOE_ERR_INVALID_ARG, "reuse_weights must be 0 or 1");
  if (d->pdl != 0 && d->pdl != 1) return fail(MOE_ERR_INVALID_ARG, "pdl must be 0 or 1");
  if (d->extras && (d->activation == MOE_ACT_SRELU || d->recompute))
    return fail(MOE_ERR_UNSUPPORTED,
                "epilogue extras need a gated activation and no recompute");
  if (r_cap(d) > (int64_t)INT32_MAX / 2) return fail(MOE_ERR_UNSUPPORTED, "row capacity too large");
  if (d->precision != MOE_PREC_BF16 &&
      (int64_t)d->E * round128(n1_of(d)) * d->H > (int64_t)INT32_MAX * 8)
    return fail(MOE_ERR_UNSUPPORTED, "block-scaled weight copies too large");
  return MOE_OK;
}

static size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

// The MXFP8 operand copies, in order after mx_base: for each GEMM input the row-wise copy
// (blocks along a row, read K-major) and the column-wise copy (blocks down a column), each
// with its slab-layout scales. rows/cols of a column-wise copy name the MMA view (rows = the
// source's columns, cols = the reduction length); its bytes keep the source's row-major
// layout, which the GEMM reads as an MN-major operand.
struct MxOps {
  MxOperand x, xt, a, at, dy, dyt, dz, dzt, w1, w1t, w2, w2t;
  int N1p, Fp;
};

// Scales of an operand [rows, cols] in the slab layout, plus 1 KB: the B operand's scales
// are fetched 256 rows at a time, so the last tile of the last k-group may read up to 128
// rows past the padded end.
static size_t mx_sf_bytes(int64_t rows, int64_t cols) {
  return (size_t)((cols / 32 + 3) / 4) * (size_t)round128(rows) * 4 + 1024;
}

// Lay the operands out from `base` (an address or 0 for offsets); returns the end offset.
static size_t mx_ops(const moe_layer_desc_t* d, int64_t R, uint8_t* base, size_t o, MxOps& m) {
  const int64_t H = d->H, F = d->F, N1 = n1_of(d), E = d->E;
  m.N1p = (int)round128(N1);
  m.Fp = (int)round128(F);
  auto op = [&](MxOperand& t, int64_t rows, int64_t cols) {
    t.rows = rows;
    t.cols = cols;
    t.s_pad = round128(rows);
    t.q = base + o;
    o = up256(o + (size_t)rows * cols);
    t.s = base + o;
    o = up256(o + mx_sf_bytes(rows, cols));
  };
  op(m.x, R, H);
  op(m.xt, H, R);
  op(m.a, R, F);
  op(m.at, F, R);
  op(m.dy, R, H);
  op(m.dyt, H, R);
  op(m.dz, R, N1);
  op(m.dzt, N1, R);
  op(m.w1, E * m.N1p, H);
  op(m.w1t, H, E * m.N1p);
  op(m.w2, E * m.Fp, H);
  op(m.w2t, H, E * m.Fp);
  return o;
}

// The NVFP4 operand copies, in order after nv_base: the same twelve operands as MXFP8, each
// K-major: packed E2M1 codes [rows, cols / 2] and E4M3 scales in the slab layout (16-value
// blocks), with the transposed copies holding rows = features and cols = the reduction
// (tokens for the weight-gradient operands, the weight's other dimension otherwise).
static size_t nv_ops(const moe_layer_desc_t* d, int64_t R, uint8_t* base, size_t o, MxOps& m) {
  const int64_t H = d->H, F = d->F, N1 = n1_of(d), E = d->E;
  m.N1p = (int)round128(N1);
  m.Fp = (int)round128(F);
  auto op = [&](MxOperand& t, int64_t rows, int64_t cols) {
    t.rows = rows;
    t.cols = cols;
    t.s_pad = round128(rows);
    t.q = base + o;
    o = up256(o + (size_t)(rows * cols / 2));
    t.s = base + o;
    o = up256(o + (size_t)nvfp4_sf_bytes(rows, cols));
  };
  op(m.x, R, H);
  op(m.xt, H, R);
  op(m.a, R, F);
  op(m.at, F, R);
  op(m.dy, R, H);
  op(m.dyt, H, R);
  op(m.dz, R, N1);
  op(m.dzt, N1, R);
  op(m.w1, E * m.N1p, H);
  op(m.w1t, H, E * m.N1p);
  op(m.w2, E * m.Fp, H);
  op(m.w2t, H, E * m.Fp);
  return o;
}

static void compute_layout(const moe_layer_desc_t* d, moe_ws_layout_t* L) {
  const int64_t R = r_cap(d);
  const int64_t H = d->H, F = d->F, N1 = n1_of(d), E = d->E;
  const bool mx = d->precision == MOE_PREC_MXFP8;
  const bool nv = d->precision == MOE_PREC_NVFP4;
  const int64_t nparts = mx ? (d->recompute ? dprob_parts_mx_recompute((int)F)
                                            : dprob_parts_mx((int)F))
                         : nv ? (d->recompute ? dprob_parts_fp4_recompute((int)F)
                                              : dprob_parts_fp4((int)F))
                              : (d->recompute ? dprob_parts_recompute((int)F)
                                              : dprob_parts((int)F));
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = up256(o + bytes);
    return at;
  };
  L->R_cap = R;
  L->err = take(256);
  L->offsets = take((E + 1) * 4);
  L->row_of = take((size_t)d->T_max * d->k * 4);
  L->src_of = take(R * 4);
  L->row_prob = take(R * 4);
  L->x_perm = take(R * H * 2);
  L->z = d->recompute ? SIZE_MAX : take(R * N1 * 2);
  // bf16 a_s and dz exist only in the BF16 path (MXFP8 keeps them as MXFP8 copies)
  L->a_s = mx ? SIZE_MAX : take(R * F * 2);
  L->y_perm = take(R * H * 2);
  L->dx_perm = L->y_perm;  // y_perm is dead once y is combined
  L->dy_perm = take(R * H * 2);
  L->dz = mx ? SIZE_MAX : take(R * N1 * 2);
  L->dprob_part = take(R * nparts * 4);
  L->ext_part = d->extras ? take((R + 31) / 32 * (N1 + F) * 4) : SIZE_MAX;
  L->mx_base = SIZE_MAX;
  if (mx) {
    MxOps m;
    L->mx_base = o;
    o = mx_ops(d, R, nullptr, o, m);
  }
  L->nv_amax = SIZE_MAX;
  L->nv_base = SIZE_MAX;
  if (nv) {
    MxOps m;
    L->nv_amax = take(16 * sizeof(float));
    L->nv_base = o;
    o = nv_ops(d, R, nullptr, o, m);
  }
  L->total = o;
}

struct Ws {
  moe_ws_layout_t L;
  uint8_t* base;
  template <class T>
  T* at(size_t off) const { return reinterpret_cast<T*>(base + off); }
};

static moe_status_t check_ws(const moe_layer_desc_t* d, void* ws, size_t ws_bytes, Ws& w) {
  compute_layout(d, &w.L);
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "ws is NULL");
  if (reinterpret_cast<uintptr_t>(ws) & 255u)
    return fail(MOE_ERR_INVALID_ARG, "ws must be 256-byte aligned");
  if (ws_bytes < w.L.total)
    return fail(MOE_ERR_WORKSPACE, "ws_bytes=%zu < required %zu", ws_bytes, w.L.total);
  w.base = static_cast<uint8_t*>(ws);
  return MOE_OK;
}

static ActDev act_of(const moe_layer_desc_t* d) {
  ActDev a;
  a.kind = d->activation;
  a.beta = d->beta;
  a.gate_max = d->gate_max;
  a.lin_lo = d->lin_lo;
  a.lin_hi = d->lin_hi;
  a.lin_offset = d->lin_offset;
  return a;
}

static int gemm_ctas(const moe_layer_desc_t* d) {
  int n = device_sms() - d->sm_margin;
  return n < 1 ? 1 : n;
}

static GemmProblem base_problem(const moe_layer_desc_t* d, const Ws& w) {
  GemmProblem p;
  memset(&p, 0, sizeof(p));
  p.E = d->E;
  p.H = d->H;
  p.F = d->F;
  p.N1 = n1_of(d);
  p.R_cap = w.L.R_cap;
  p.offsets = w.at<int32_t>(w.L.offsets);
  p.row_prob = w.at<float>(w.L.row_prob);
  p.x_perm = w.at<void>(w.L.x_perm);
  p.a_s = w.L.a_s == SIZE_MAX ? nullptr : w.at<void>(w.L.a_s);
  p.z = w.L.z == SIZE_MAX ? nullptr : w.at<void>(w.L.z);
  p.dz = w.L.dz == SIZE_MAX ? nullptr : w.at<void>(w.L.dz);
  p.dy_perm = w.at<void>(w.L.dy_perm);
  p.gated = d->activation != MOE_ACT_SRELU;
  p.ilv = d->ilv;
  p.act = act_of(d);
  p.err = w.at<int>(w.L.err);
  p.num_ctas = gemm_ctas(d);
  p.rows_per_expert = (int64_t)d->T_max * d->k / d->E;
  return p;
}

static int grid_for(int64_t work, int per_sm) {
  int sms = device_sms();
  if (sms <= 0) sms = 1;
  int64_t g = std::min<int64_t>(work, (int64_t)sms * per_sm);
  return (int)std::max<int64_t>(g, 1);
}

static MxProblem mx_problem(const moe_layer_desc_t* d, const Ws& w) {
  MxProblem p;
  memset(&p, 0, sizeof(p));
  MxOps m;
  mx_ops(d, w.L.R_cap, w.base, w.L.mx_base, m);
  p.E = d->E;
  p.H = d->H;
  p.F = d->F;
  p.N1 = n1_of(d);
  p.N1p = m.N1p;
  p.Fp = m.Fp;
  p.R_cap = w.L.R_cap;
  p.offsets = w.at<int32_t>(w.L.offsets);
  p.x = m.x; p.xt = m.xt; p.a = m.a; p.at = m.at; p.dy = m.dy; p.dyt = m.dyt;
  p.dz = m.dz; p.dzt = m.dzt; p.w1 = m.w1; p.w1t = m.w1t; p.w2 = m.w2; p.w2t = m.w2t;
  p.row_prob = w.at<float>(w.L.row_prob);
  p.z = w.L.z == SIZE_MAX ? nullptr : w.at<void>(w.L.z);
  p.gated = d->activation != MOE_ACT_SRELU;
  p.ilv = d->ilv;
  p.act = act_of(d);
  p.err = w.at<int>(w.L.err);
  p.num_ctas = gemm_ctas(d);
  p.rows_per_expert = (int64_t)d->T_max * d->k / d->E;
  return p;
}

static Fp4Problem fp4_problem(const moe_layer_desc_t* d, const Ws& w) {
  Fp4Problem p;
  memset(&p, 0, sizeof(p));
  MxOps m;
  nv_ops(d, w.L.R_cap, w.base, w.L.nv_base, m);
  p.E = d->E;
  p.H = d->H;
  p.F = d->F;
  p.N1 = n1_of(d);
  p.N1p = m.N1p;
  p.Fp = m.Fp;
  p.R_cap = w.L.R_cap;
  p.offsets = w.at<int32_t>(w.L.offsets);
  p.x = m.x; p.xt = m.xt; p.a = m.a; p.at = m.at; p.dy = m.dy; p.dyt = m.dyt;
  p.dz = m.dz; p.dzt = m.dzt; p.w1 = m.w1; p.w1t = m.w1t; p.w2 = m.w2; p.w2t = m.w2t;
  p.amax = w.at<float>(w.L.nv_amax);
  p.row_prob = w.at<float>(w.L.row_prob);
  p.z = w.at<void>(w.L.z);
  p.gated = d->activation != MOE_ACT_SRELU;
  p.ilv = d->ilv;
  p.rht_mask = d->rht_mask & 0xFFFFu;
  p.act = act_of(d);
  p.err = w.at<int>(w.L.err);
  p.num_ctas = gemm_ctas(d);
  return p;
}

// NVFP4 copies of a bf16 matrix [M, N] (input row groups G stored at stride Gp; rows at or
// beyond *row_limit zero when given): the row-wise copy `row` with the encode scale of
// amax[row_slot] and the transposed copy `col` with that of amax[col_slot], rotated when rht.
static bool nv_quantize(const void* in, int64_t M, int64_t N, int64_t G, int64_t Gp,
                        const int32_t* row_limit, const Fp4Problem& p, int row_slot,
                        int col_slot, const MxOperand& row, const MxOperand& col, int rht,
                        cudaStream_t s) {
  Nvfp4QuantArgs a;
  memset(&a, 0, sizeof(a));
  a.in = in;
  a.M = M;
  a.N = N;
  a.G = G;
  a.Gp = Gp;
  a.row_limit = row_limit;
  a.amax_row = p.amax + row_slot;
  a.amax_col = p.amax + col_slot;
  a.q_row = row.q;
  a.s_row = row.s;
  a.s_row_pad = row.s_pad;
  a.q_col = col.q;
  a.s_col = col.s;
  a.s_col_pad = col.s_pad;
  a.rht = rht;
  a.rht_mask = p.rht_mask;
  a.err = p.err;
  return launch_nvfp4_quantize(a, std::max(device_sms(), 1), s);
}

// Quantise a bf16 matrix [M, N] (row groups G padded to Gp) into the row-wise and the
// column-wise MXFP8 operands of the block-scaled GEMM (both in the source's layout).
static void mx_quantize_operands(const void* in, int64_t M, int64_t N, int64_t G, int64_t Gp,
                                 const MxOperand& row, const MxOperand& col, cudaStream_t s) {
  launch_mxfp8_quantize_mma(in, M, N, G, Gp, row.q, row.s, col.q, col.s,
                            std::max(device_sms(), 1), s);
}

// One thread waits, with the bounded wait every GEMM uses, on an mbarrier that expects one
// arrival nobody makes; the wait gives up after limit_ns, records MOE_DEVERR_TIMEOUT and the
// kernel returns normally.
__global__ void selftest_wait_timeout_kernel(int* err, uint64_t limit_ns) {
  MOE_GRIDDEP_ENTRY();
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    abort_flag = 0;
    mbar_wait(&bar, 0, &abort_flag, err, limit_ns);
  }
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_size(const moe_layer_desc_t* desc) {
  if (validate_desc(desc) != MOE_OK) return 0;
  moe_ws_layout_t L;
  compute_layout(desc, &L);
  return L.total;
}

moe_status_t moe_workspace_layout(const moe_layer_desc_t* desc, moe_ws_layout_t* out) {
  moe_status_t st = validate_desc(desc);
  if (st != MOE_OK) return st;
  if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
  compute_layout(desc, out);
  return MOE_OK;
}

moe_status_t moe_route_permute(const moe_layer_desc_t* d, int32_t T, const float* logits,
                               const void* x, int32_t* topk_ids, float* topk_probs,
                               int32_t* counts, void* ws, size_t ws_bytes, moe_stream_t stream) {
  PdlScope pdl_scope(d);
  moe_status_t st = validate_desc(d);
  if (st != MOE_OK) return st;
  if (T < 0 || T > d->T_max) return fail(MOE_ERR_INVALID_ARG, "T=%d outside [0, T_max]", T);
  if ((T > 0 && (!logits || !x || !topk_ids || !topk_probs)) || !counts)
    return fail(MOE_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(x)) return fail(MOE_ERR_INVALID_ARG, "x must be 16-byte aligned");
  Ws w;
  if ((st = check_ws(d, ws, ws_bytes, w)) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * d->E, s);
  if (e != cudaSuccess) return cuda_fail(e, "memset counts");
  int32_t* offsets = w.at<int32_t>(w.L.offsets);
  int32_t* row_of = w.at<int32_t>(w.L.row_of);
  int32_t* src_of = w.at<int32_t>(w.L.src_of);
  float* row_prob = w.at<float>(w.L.row_prob);
  int* err = w.at<int>(w.L.err);
  if (T > 0) {
    launch_kernel(route_topk_kernel, grid_for((T + 7) / 8, 8), 256, 0, s, nullptr, 0, logits, T, d->E, d->k, topk_ids,
                                                                 topk_probs, counts);
    count_launch(s, MOE_K_ROUTE_TOPK);
  }
  launch_kernel(assign_rows_kernel, d->E, 1024, 0, s, nullptr, 0, topk_ids, topk_probs, counts, T, d->E, d->k, d->align,
                                           w.L.R_cap, offsets, row_of, src_of, row_prob, err);
  count_launch(s, MOE_K_ASSIGN_ROWS);
  if (d->precision == MOE_PREC_NVFP4) {
    // gather fused with X's amax and rotated amax, then its copies: along H for FC1 and
    // transposed, rotated along the expert's rows, for the FC1 weight gradient
    const Fp4Problem p = fp4_problem(d, w);
    e = cudaMemsetAsync(p.amax + AM_X, 0, 2 * sizeof(float), s);
    if (e != cudaSuccess) return cuda_fail(e, "memset amax");
    launch_gather_rows_amax(x, src_of, offsets, d->E, d->k, d->H, w.L.R_cap, p.rht_mask,
                            w.at<void>(w.L.x_perm), p.amax + AM_X, p.amax + AM_XT, device_sms(),
                            MOE_K_GATHER_X, s);
    if (!nv_quantize(w.at<void>(w.L.x_perm), w.L.R_cap, d->H, w.L.R_cap, w.L.R_cap, nullptr, p,
                     AM_X, AM_XT, p.x, p.xt, 1, s))
      return fail(MOE_ERR_CUDA, "NVFP4 quantiser: tensor map or shared-memory limit");
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "route_permute launch");
    return MOE_OK;
  }
  launch_kernel(gather_rows_kernel, grid_for(w.L.R_cap, 8), 256, 0, s, nullptr, 0, 
      static_cast<const uint4*>(x), src_of, offsets, d->E, d->k, d->H / 8, w.L.R_cap,
      w.at<uint4>(w.L.x_perm));
  count_launch(s, MOE_K_GATHER_X);
  if (d->precision == MOE_PREC_MXFP8) {
    // X along H for FC1 and column-wise (along the expert's rows) for the FC1 weight gradient
    const MxProblem m = mx_problem(d, w);
    mx_quantize_operands(w.at<void>(w.L.x_perm), w.L.R_cap, d->H, w.L.R_cap, w.L.R_cap, m.x,
                         m.xt, s);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "route_permute launch");
  return MOE_OK;
}

static moe_status_t fwd_impl(const moe_layer_desc_t* d, int32_t T, const void* w1_packed,
                             const void* w2, const float* fc1_bias, const float* feat_scale,
                             void* y, void* ws, size_t ws_bytes, moe_stream_t stream) {
  PdlScope pdl_scope(d);
  moe_status_t st = validate_desc(d);
  if (st != MOE_OK) return st;
  if (((d->extras & 1) != 0) != (fc1_bias != nullptr) ||
      ((d->extras & 2) != 0) != (feat_scale != nullptr))
    return fail(MOE_ERR_INVALID_ARG, "fc1_bias / feat_scale must match desc->extras");
  if (T < 0 || T > d->T_max) return fail(MOE_ERR_INVALID_ARG, "T=%d outside [0, T_max]", T);
  if (!w1_packed || !w2 || (T > 0 && !y)) return fail(MOE_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(w1_packed) || !aligned16(w2) || !aligned16(y))
    return fail(MOE_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  Ws w;
  if ((st = check_ws(d, ws, ws_bytes, w)) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (d->precision == MOE_PREC_MXFP8) {
    MxProblem m = mx_problem(d, w);
    // BF16 master weights -> MXFP8 along both reduction directions ([TE-MoE] Challenge 3),
    // unless the copies of an earlier forward are reused
    if (!d->reuse_weights) {
      mx_quantize_operands(w1_packed, (int64_t)d->E * m.N1, d->H, m.N1, m.N1p, m.w1, m.w1t, s);
      mx_quantize_operands(w2, (int64_t)d->E * d->F, d->H, d->F, m.Fp, m.w2, m.w2t, s);
    }
    // FC1 + activation + probability scale + MXFP8 quantise/transpose (kernel family 2), with
    // the optional bias and feature scale
    m.role = ROLE_FC1_FPROP;
    m.out = d->recompute ? nullptr : w.at<void>(w.L.z);  // NULL: Z is not kept
    m.fc1_bias = fc1_bias;
    m.fscale = feat_scale;
    if ((e = launch_grouped_gemm_mx(m, s)) != cudaSuccess) return cuda_fail(e, "FC1 MX GEMM");
    m.fc1_bias = m.fscale = nullptr;
    m.role = ROLE_FC2_FPROP;
    m.out = w.at<void>(w.L.y_perm);
    if ((e = launch_grouped_gemm_mx(m, s)) != cudaSuccess) return cuda_fail(e, "FC2 MX GEMM");
    if (T > 0) {
      launch_kernel(combine_rows_kernel, grid_for(T, 8), 256, 0, s, nullptr, 0, w.at<uint4>(w.L.y_perm),
                                                        w.at<int32_t>(w.L.row_of), T, d->k,
                                                        d->H / 8, static_cast<uint4*>(y));
      count_launch(s, MOE_K_COMBINE_Y);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "fwd launch");
    return MOE_OK;
  }
  if (d->precision == MOE_PREC_NVFP4) {
    Fp4Problem m = fp4_problem(d, w);
    const int32_t* live = w.at<int32_t>(w.L.offsets) + d->E;  // rows in use
    // BF16 master weights -> NVFP4 along both reduction directions (per-tensor amax first),
    // unless the copies and amaxes of an earlier forward are reused; the FC1 epilogue's
    // amax slots (a_s and its rotation) start at zero either way
    static_assert(AM_W2 == AM_W1 + 1 && AM_A == AM_W1 + 2 && AM_AT == AM_W1 + 3,
                  "amax slot order");
    if ((e = cudaMemsetAsync(m.amax + (d->reuse_weights ? AM_A : AM_W1), 0,
                             (d->reuse_weights ? 2 : 4) * sizeof(float), s)) != cudaSuccess)
      return cuda_fail(e, "memset amax");
    if (!d->reuse_weights) {
      launch_nvfp4_amax(w1_packed, (int64_t)d->E * m.N1 * d->H, m.amax + AM_W1, device_sms(), s);
      launch_nvfp4_amax(w2, (int64_t)d->E * d->F * d->H, m.amax + AM_W2, device_sms(), s);
      if (!nv_quantize(w1_packed, (int64_t)d->E * m.N1p, d->H, m.N1, m.N1p, nullptr, m, AM_W1,
                       AM_W1, m.w1, m.w1t, 0, s) ||
          !nv_quantize(w2, (int64_t)d->E * m.Fp, d->H, d->F, m.Fp, nullptr, m, AM_W2, AM_W2,
                       m.w2, m.w2t, 0, s))
        return fail(MOE_ERR_CUDA, "NVFP4 quantiser: tensor map or shared-memory limit");
    }
    // FC1 + activation + probability scale, BF16 a_s plus its amax and rotated amax
    m.role = ROLE_FC1_FPROP;
    m.out = d->recompute ? nullptr : w.at<void>(w.L.z);  // NULL: Z is not kept
    m.out2 = w.at<void>(w.L.a_s);
    m.fc1_bias = fc1_bias;
    m.fscale = feat_scale;
    if ((e = launch_grouped_gemm_fp4(m, s)) != cudaSuccess) return cuda_fail(e, "FC1 FP4 GEMM");
    m.fc1_bias = m.fscale = nullptr;
    if (!nv_quantize(w.at<void>(w.L.a_s), w.L.R_cap, d->F, w.L.R_cap, w.L.R_cap, live, m, AM_A,
                     AM_AT, m.a, m.at, 1, s))
      return fail(MOE_ERR_CUDA, "NVFP4 quantiser: tensor map or shared-memory limit");
    m.role = ROLE_FC2_FPROP;
    m.out = w.at<void>(w.L.y_perm);
    m.out2 = nullptr;
    if ((e = launch_grouped_gemm_fp4(m, s)) != cudaSuccess) return cuda_fail(e, "FC2 FP4 GEMM");
    if (T > 0) {
      launch_kernel(combine_rows_kernel, grid_for(T, 8), 256, 0, s, nullptr, 0, w.at<uint4>(w.L.y_perm),
                                                        w.at<int32_t>(w.L.row_of), T, d->k,
                                                        d->H / 8, static_cast<uint4*>(y));
      count_launch(s, MOE_K_COMBINE_Y);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "fwd launch");
    return MOE_OK;
  }
  GemmProblem p = base_problem(d, w);
  p.w1p = w1_packed;
  p.w2 = w2;
  p.fc1_bias = fc1_bias;
  p.fscale = feat_scale;
  // FC1 + activation + probability scale (kernel family 2)
  p.role = ROLE_FC1_FPROP;
  p.out = d->recompute ? nullptr : w.at<void>(w.L.z);  // NULL: Z is not kept
  p.out2 = w.at<void>(w.L.a_s);
  if ((e = launch_grouped_gemm(p, s)) != cudaSuccess) return cuda_fail(e, "FC1 grouped GEMM");
  // FC2 (kernel family 1)
  p.role = ROLE_FC2_FPROP;
  p.out = w.at<void>(w.L.y_perm);
  p.out2 = nullptr;
  p.fc1_bias = p.fscale = nullptr;
  if ((e = launch_grouped_gemm(p, s)) != cudaSuccess) return cuda_fail(e, "FC2 grouped GEMM");
  if (T > 0) {
    launch_kernel(combine_rows_kernel, grid_for(T, 8), 256, 0, s, nullptr, 0, w.at<uint4>(w.L.y_perm),
                                                      w.at<int32_t>(w.L.row_of), T, d->k,
                                                      d->H / 8, static_cast<uint4*>(y));
    count_launch(s, MOE_K_COMBINE_Y);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "fwd launch");
  return MOE_OK;
}

// Per-expert sums of the dGLU epilogue's per-32-row column sums: the FC1 bias gradient (the
// dZ columns, logical order) and the feature-scale gradient.
static cudaError_t launch_extras_reduce(const moe_layer_desc_t* d, const Ws& w, float* d_fc1_bias,
                                        float* d_feat_scale, cudaStream_t s) {
  const int N1 = n1_of(d), ld = N1 + d->F;
  const int32_t* off = w.at<int32_t>(w.L.offsets);
  if (d_fc1_bias) {
    launch_kernel(group_colsum_kernel, dim3((N1 + 255) / 256, d->E), 256, 0, s, nullptr, 0,
                  w.at<float>(w.L.ext_part), ld, 0, N1, off, d_fc1_bias);
    count_launch(s, MOE_K_EXTRAS_REDUCE);
  }
  if (d_feat_scale) {
    launch_kernel(group_colsum_kernel, dim3((d->F + 255) / 256, d->E), 256, 0, s, nullptr, 0,
                  w.at<float>(w.L.ext_part), ld, N1, d->F, off, d_feat_scale);
    count_launch(s, MOE_K_EXTRAS_REDUCE);
  }
  return cudaGetLastError();
}

static moe_status_t bwd_impl(const moe_layer_desc_t* d, int32_t T, const void* dy,
                             const void* w1_packed, const void* w2, const float* feat_scale,
                             void* dx, void* dw1_packed, void* dw2, float* d_probs,
                             float* d_fc1_bias, float* d_feat_scale, void* ws, size_t ws_bytes,
                             moe_stream_t stream) {
  PdlScope pdl_scope(d);
  moe_status_t st = validate_desc(d);
  if (st != MOE_OK) return st;
  if (((d->extras & 1) != 0) != (d_fc1_bias != nullptr) ||
      ((d->extras & 2) != 0) != (feat_scale != nullptr && d_feat_scale != nullptr) ||
      ((d->extras & 2) == 0 && (feat_scale || d_feat_scale)))
    return fail(MOE_ERR_INVALID_ARG, "extras pointers must match desc->extras");
  if (T < 0 || T > d->T_max) return fail(MOE_ERR_INVALID_ARG, "T=%d outside [0, T_max]", T);
  if (!w1_packed || !w2 || !dw1_packed || !dw2 || (T > 0 && (!dy || !dx || !d_probs)))
    return fail(MOE_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(dy) || !aligned16(dx) || !aligned16(w1_packed) || !aligned16(w2) ||
      !aligned16(dw1_packed) || !aligned16(dw2))
    return fail(MOE_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  Ws w;
  if ((st = check_ws(d, ws, ws_bytes, w)) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  GemmProblem p = base_problem(d, w);
  p.w1p = w1_packed;
  p.w2 = w2;
  const int32_t* row_of = w.at<int32_t>(w.L.row_of);
  cudaError_t e;
  // dY gathered into the permuted row order (zero for padding rows); for NVFP4 together with
  // its amax and rotated amax
  if (d->precision == MOE_PREC_NVFP4) {
    float* am = w.at<float>(w.L.nv_amax);
    if ((e = cudaMemsetAsync(am + AM_DY, 0, 4 * sizeof(float), s)) != cudaSuccess)
      return cuda_fail(e, "memset amax");
    launch_gather_rows_amax(dy, w.at<int32_t>(w.L.src_of), w.at<int32_t>(w.L.offsets), d->E,
                            d->k, d->H, w.L.R_cap, d->rht_mask & 0xFFFFu, w.at<void>(w.L.dy_perm),
                            am + AM_DY, am + AM_DYT, device_sms(), MOE_K_GATHER_DY, s);
  } else {
    launch_kernel(gather_rows_kernel, grid_for(w.L.R_cap, 8), 256, 0, s, nullptr, 0, 
        static_cast<const uint4*>(dy), w.at<int32_t>(w.L.src_of), w.at<int32_t>(w.L.offsets),
        d->E, d->k, d->H / 8, w.L.R_cap, w.at<uint4>(w.L.dy_perm));
    count_launch(s, MOE_K_GATHER_DY);
  }
  if (d->precision == MOE_PREC_MXFP8) {
    MxProblem m = mx_problem(d, w);
    mx_quantize_operands(w.at<void>(w.L.dy_perm), w.L.R_cap, d->H, w.L.R_cap, w.L.R_cap, m.dy,
                         m.dyt, s);
    // FC2 dgrad + dActivation + MXFP8 quantise/transpose of dZ (kernel family 3)
    m.role = ROLE_FC2_DGRAD;
    m.dprob_part = w.at<float>(w.L.dprob_part);
    if (d->extras) {
      m.fscale = feat_scale;
      m.ext_part = w.at<float>(w.L.ext_part);
    }
    if (d->recompute) {
      // the same kernel family with Z rebuilt from X and W1 next to dA_s
      if ((e = launch_fc2_dgrad_recompute_mx(m, s)) != cudaSuccess)
        return cuda_fail(e, "FC2 dgrad recompute MX");
    } else if ((e = launch_grouped_gemm_mx(m, s)) != cudaSuccess) {
      return cuda_fail(e, "FC2 dgrad MX");
    }
    m.fscale = nullptr;
    m.ext_part = nullptr;
    if (T > 0) {
      const int n = T * d->k;
      launch_kernel(dprob_reduce_kernel, grid_for((n + 255) / 256, 4), 256, 0, s, nullptr, 0,
                    w.at<float>(w.L.dprob_part),
                    d->recompute ? dprob_parts_mx_recompute(d->F) : dprob_parts_mx(d->F),
                    row_of, n, d_probs);
      count_launch(s, MOE_K_DPROB_REDUCE);
    }
    if (d->extras) {
      if ((e = launch_extras_reduce(d, w, d_fc1_bias, d_feat_scale, s)) != cudaSuccess)
        return cuda_fail(e, "extras reduce");
    }
    m.role = ROLE_FC2_WGRAD;
    m.out = dw2;
    if ((e = launch_grouped_gemm_mx(m, s)) != cudaSuccess) return cuda_fail(e, "FC2 wgrad MX");
    m.role = ROLE_FC1_DGRAD;
    m.out = w.at<void>(w.L.dx_perm);
    if ((e = launch_grouped_gemm_mx(m, s)) != cudaSuccess) return cuda_fail(e, "FC1 dgrad MX");
    if (T > 0) {
      launch_kernel(combine_rows_kernel, grid_for(T, 8), 256, 0, s, nullptr, 0, w.at<uint4>(w.L.dx_perm), row_of, T,
                                                        d->k, d->H / 8, static_cast<uint4*>(dx));
      count_launch(s, MOE_K_COMBINE_DX);
    }
    m.role = ROLE_FC1_WGRAD;
    m.out = dw1_packed;
    if ((e = launch_grouped_gemm_mx(m, s)) != cudaSuccess) return cuda_fail(e, "FC1 wgrad MX");
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "bwd launch");
    return MOE_OK;
  }
  if (d->precision == MOE_PREC_NVFP4) {
    Fp4Problem m = fp4_problem(d, w);
    const int32_t* live = w.at<int32_t>(w.L.offsets) + d->E;
    if (!nv_quantize(w.at<void>(w.L.dy_perm), w.L.R_cap, d->H, w.L.R_cap, w.L.R_cap, nullptr, m,
                     AM_DY, AM_DYT, m.dy, m.dyt, 1, s))
      return fail(MOE_ERR_CUDA, "NVFP4 quantiser: tensor map or shared-memory limit");
    // FC2 dgrad + dActivation: BF16 dZ plus its amax and the amax of its rotated transpose
    m.role = ROLE_FC2_DGRAD;
    m.out = w.at<void>(w.L.dz);
    m.dprob_part = w.at<float>(w.L.dprob_part);
    if (d->extras) {
      m.fscale = feat_scale;
      m.ext_part = w.at<float>(w.L.ext_part);
    }
    if (d->recompute) {  // the FC1 output is rebuilt from the NVFP4 copies of X and W1
      if ((e = launch_fc2_dgrad_recompute_fp4(m, s)) != cudaSuccess)
        return cuda_fail(e, "FC2 dgrad recompute FP4");
    } else if ((e = launch_grouped_gemm_fp4(m, s)) != cudaSuccess) {
      return cuda_fail(e, "FC2 dgrad FP4");
    }
    m.fscale = nullptr;
    m.ext_part = nullptr;
    if (d->extras) {
      if ((e = launch_extras_reduce(d, w, d_fc1_bias, d_feat_scale, s)) != cudaSuccess)
        return cuda_fail(e, "extras reduce");
    }
    if (T > 0) {
      const int n = T * d->k;
      launch_kernel(dprob_reduce_kernel, grid_for((n + 255) / 256, 4), 256, 0, s, nullptr, 0,
          w.at<float>(w.L.dprob_part),
          d->recompute ? dprob_parts_fp4_recompute(d->F) : dprob_parts_fp4(d->F), row_of, n,
          d_probs);
      count_launch(s, MOE_K_DPROB_REDUCE);
    }
    if (!nv_quantize(w.at<void>(w.L.dz), w.L.R_cap, m.N1, w.L.R_cap, w.L.R_cap, live, m, AM_DZ,
                     AM_DZT, m.dz, m.dzt, 1, s))
      return fail(MOE_ERR_CUDA, "NVFP4 quantiser: tensor map or shared-memory limit");
    m.role = ROLE_FC2_WGRAD;
    m.out = dw2;
    if ((e = launch_grouped_gemm_fp4(m, s)) != cudaSuccess) return cuda_fail(e, "FC2 wgrad FP4");
    m.role = ROLE_FC1_DGRAD;
    m.out = w.at<void>(w.L.dx_perm);
    if ((e = launch_grouped_gemm_fp4(m, s)) != cudaSuccess) return cuda_fail(e, "FC1 dgrad FP4");
    if (T > 0) {
      launch_kernel(combine_rows_kernel, grid_for(T, 8), 256, 0, s, nullptr, 0, w.at<uint4>(w.L.dx_perm), row_of, T,
                                                        d->k, d->H / 8, static_cast<uint4*>(dx));
      count_launch(s, MOE_K_COMBINE_DX);
    }
    m.role = ROLE_FC1_WGRAD;
    m.out = dw1_packed;
    if ((e = launch_grouped_gemm_fp4(m, s)) != cudaSuccess) return cuda_fail(e, "FC1 wgrad FP4");
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "bwd launch");
    return MOE_OK;
  }
  // FC2 dgrad + dActivation (kernel family 3); with recomputation the same kernel rebuilds Z
  p.role = ROLE_FC2_DGRAD;
  p.out = w.at<void>(w.L.dz);
  p.dprob_part = w.at<float>(w.L.dprob_part);
  if (d->extras) {
    p.fscale = feat_scale;
    p.ext_part = w.at<float>(w.L.ext_part);
  }
  if (d->recompute) {
    p.w1p = w1_packed;
    if ((e = launch_fc2_dgrad_recompute(p, s)) != cudaSuccess)
      return cuda_fail(e, "FC2 dgrad recompute GEMM");
  } else if ((e = launch_grouped_gemm(p, s)) != cudaSuccess) {
    return cuda_fail(e, "FC2 dgrad GEMM");
  }
  if (T > 0) {
    const int nparts = d->recompute ? dprob_parts_recompute(d->F) : dprob_parts(d->F);
    const int n = T * d->k;
    launch_kernel(dprob_reduce_kernel, grid_for((n + 255) / 256, 4), 256, 0, s, nullptr, 0, 
        w.at<float>(w.L.dprob_part), nparts, row_of, n, d_probs);
    count_launch(s, MOE_K_DPROB_REDUCE);
  }
  if (d->extras) {
    if ((e = launch_extras_reduce(d, w, d_fc1_bias, d_feat_scale, s)) != cudaSuccess)
      return cuda_fail(e, "extras reduce");
    p.fscale = nullptr;
    p.ext_part = nullptr;
  }
  // FC2 wgrad
  p.role = ROLE_FC2_WGRAD;
  p.out = dw2;
  if ((e = launch_grouped_gemm(p, s)) != cudaSuccess) return cuda_fail(e, "FC2 wgrad GEMM");
  // FC1 dgrad (kernel family 1) and combine
  p.role = ROLE_FC1_DGRAD;
  p.out = w.at<void>(w.L.dx_perm);
  if ((e = launch_grouped_gemm(p, s)) != cudaSuccess) return cuda_fail(e, "FC1 dgrad GEMM");
  if (T > 0) {
    launch_kernel(combine_rows_kernel, grid_for(T, 8), 256, 0, s, nullptr, 0, w.at<uint4>(w.L.dx_perm), row_of, T,
                                                      d->k, d->H / 8, static_cast<uint4*>(dx));
    count_launch(s, MOE_K_COMBINE_DX);
  }
  // FC1 wgrad
  p.role = ROLE_FC1_WGRAD;
  p.out = dw1_packed;
  if ((e = launch_grouped_gemm(p, s)) != cudaSuccess) return cuda_fail(e, "FC1 wgrad GEMM");
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "bwd launch");
  return MOE_OK;
}

moe_status_t moe_grouped_mlp_fwd(const moe_layer_desc_t* d, int32_t T, const void* w1_packed,
                                 const void* w2, void* y, void* ws, size_t ws_bytes,
                                 moe_stream_t stream) {
  if (d && d->extras) return fail(MOE_ERR_UNSUPPORTED, "a layer with extras uses moe_grouped_mlp_fwd_ex");
  return fwd_impl(d, T, w1_packed, w2, nullptr, nullptr, y, ws, ws_bytes, stream);
}

moe_status_t moe_grouped_mlp_fwd_ex(const moe_layer_desc_t* d, int32_t T, const void* w1_packed,
                                    const void* w2, const float* fc1_bias,
                                    const float* feat_scale, void* y, void* ws, size_t ws_bytes,
                                    moe_stream_t stream) {
  return fwd_impl(d, T, w1_packed, w2, fc1_bias, feat_scale, y, ws, ws_bytes, stream);
}

moe_status_t moe_grouped_mlp_bwd(const moe_layer_desc_t* d, int32_t T, const void* dy,
                                 const void* w1_packed, const void* w2, void* dx,
                                 void* dw1_packed, void* dw2, float* d_probs, void* ws,
                                 size_t ws_bytes, moe_stream_t stream) {
  if (d && d->extras) return fail(MOE_ERR_UNSUPPORTED, "a layer with extras uses moe_grouped_mlp_bwd_ex");
  return bwd_impl(d, T, dy, w1_packed, w2, nullptr, dx, dw1_packed, dw2, d_probs, nullptr,
                  nullptr, ws, ws_bytes, stream);
}

moe_status_t moe_grouped_mlp_bwd_ex(const moe_layer_desc_t* d, int32_t T, const void* dy,
                                    const void* w1_packed, const void* w2,
                                    const float* feat_scale, void* dx, void* dw1_packed,
                                    void* dw2, float* d_probs, float* d_fc1_bias,
                                    float* d_feat_scale, void* ws, size_t ws_bytes,
                                    moe_stream_t stream) {
  return bwd_impl(d, T, dy, w1_packed, w2, feat_scale, dx, dw1_packed, dw2, d_probs, d_fc1_bias,
                  d_feat_scale, ws, ws_bytes, stream);
}

moe_status_t moe_selftest_wait_timeout(int32_t* err, uint64_t limit_ns, moe_stream_t stream) {
  if (!err) return fail(MOE_ERR_INVALID_ARG, "err is NULL");
  if (limit_ns < 1000000ull || limit_ns > 10000000000ull)
    return fail(MOE_ERR_INVALID_ARG, "limit_ns must be in [1 ms, 10 s]");
  launch_kernel(selftest_wait_timeout_kernel, 1, 32, 0, reinterpret_cast<cudaStream_t>(stream), nullptr, 0, err, limit_ns);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
  return MOE_OK;
}

moe_status_t moe_route_export(const moe_layer_desc_t* d, const void* ws, size_t ws_bytes,
                              int32_t T, int32_t* offsets, int32_t* row_of, int32_t* src_of,
                              float* row_prob, moe_stream_t stream) {
  moe_status_t st = validate_desc(d);
  if (st != MOE_OK) return st;
  if (T < 0 || T > d->T_max) return fail(MOE_ERR_INVALID_ARG, "T=%d outside [0, T_max]", T);
  auto a4 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 3) == 0; };
  if (!a4(offsets) || !a4(row_of) || !a4(src_of) || !a4(row_prob))
    return fail(MOE_ERR_INVALID_ARG, "destinations must be 4-byte aligned");
  Ws w;
  if ((st = check_ws(d, const_cast<void*>(ws), ws_bytes, w)) != MOE_OK) return st;
  if (!offsets && !row_of && !src_of && !row_prob) return MOE_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t n_total =
      std::max<int64_t>(w.L.R_cap, std::max<int64_t>((int64_t)T * d->k, d->E + 1));
  const int grid =
      (int)std::min<int64_t>((n_total + 255) / 256, (int64_t)std::max(device_sms(), 1) * 4);
  launch_kernel(route_export_kernel, grid, 256, 0, s, nullptr, 0, w.at<int32_t>(w.L.offsets),
                d->E + 1, w.at<int32_t>(w.L.row_of), (int64_t)T * d->k, w.at<int32_t>(w.L.src_of),
                w.at<float>(w.L.row_prob), (int64_t)w.L.R_cap, n_total, offsets, row_of, src_of,
                row_prob);
  count_launch(s, MOE_K_ROUTE_EXPORT);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "route export launch");
  return MOE_OK;
}

moe_status_t moe_selftest_gemm_timeout(const moe_layer_desc_t* d, void* ws, size_t ws_bytes,
                                       const void* w2, uint64_t limit_ns, moe_stream_t stream) {
  moe_status_t st = validate_desc(d);
  if (st != MOE_OK) return st;
  if (d->precision != MOE_PREC_BF16) return fail(MOE_ERR_UNSUPPORTED, "needs a BF16 layer");
  if (!w2 || !aligned16(w2)) return fail(MOE_ERR_INVALID_ARG, "w2 must be non-NULL, 16B aligned");
  if (limit_ns < 1000000ull || limit_ns > 10000000000ull)
    return fail(MOE_ERR_INVALID_ARG, "limit_ns must be in [1 ms, 10 s]");
  Ws w;
  if ((st = check_ws(d, ws, ws_bytes, w)) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the FC2 forward GEMM of the routed layer, with a producer that issues no loads: every
  // consumer wait runs out after limit_ns, the kernel records the timeout and returns
  GemmProblem p = base_problem(d, w);
  p.w2 = w2;
  p.role = ROLE_FC2_FPROP;
  p.out = w.at<void>(w.L.y_perm);
  p.stall_loads = 1;
  p.wait_ns = limit_ns;
  cudaError_t e = launch_grouped_gemm(p, s);
  if (e != cudaSuccess) return cuda_fail(e, "self-test GEMM launch");
  return MOE_OK;
}

moe_status_t mxfp8_quantize(const void* in, int64_t M, int64_t N, int32_t rowwise,
                            int32_t colwise, const int32_t* group_offsets, int32_t num_groups,
                            uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                            moe_stream_t stream) {
  if (M < 0 || N < 0) return fail(MOE_ERR_INVALID_ARG, "negative size");
  if (!rowwise && !colwise) return fail(MOE_ERR_INVALID_ARG, "neither rowwise nor colwise");
  const bool grouped = group_offsets != nullptr;
  if (grouped && (num_groups < 1 || num_groups > 65536))
    return fail(MOE_ERR_INVALID_ARG, "num_groups must be in [1, 65536] with group_offsets");
  if (M == 0 || N == 0) return MOE_OK;
  if (!in || !aligned16(in)) return fail(MOE_ERR_INVALID_ARG, "in must be non-NULL, 16B aligned");
  if (N % 32) return fail(MOE_ERR_UNSUPPORTED, "N must be a multiple of 32");
  if (colwise && !grouped && M % 32)
    return fail(MOE_ERR_UNSUPPORTED, "M must be a multiple of 32 (colwise without groups)");
  if (!mxfp8_quantize_size_ok(M, N)) return fail(MOE_ERR_UNSUPPORTED, "M or N too large");
  if (rowwise && (!q_row || !s_row || !aligned16(q_row)))
    return fail(MOE_ERR_INVALID_ARG, "rowwise outputs must be non-NULL (q_row 16B aligned)");
  if (colwise && (!q_col || !s_col || !aligned16(q_col)))
    return fail(MOE_ERR_INVALID_ARG, "colwise outputs must be non-NULL (q_col 16B aligned)");
  if (colwise && grouped && (reinterpret_cast<uintptr_t>(s_col) & 3u))
    return fail(MOE_ERR_INVALID_ARG, "s_col must be 4-byte aligned with group_offsets");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int sms = std::max(device_sms(), 1);
  if (colwise && grouped) {
    if (rowwise)
      launch_mxfp8_quantize(in, M, N, 1, 0, q_row, s_row, nullptr, nullptr, sms, s);
    launch_mxfp8_colwise_grouped(in, M, N, group_offsets, num_groups, q_col, s_col, sms, s);
  } else {
    launch_mxfp8_quantize(in, M, N, rowwise, colwise, q_row, s_row, q_col, s_col, sms, s);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "mxfp8_quantize launch");
  return MOE_OK;
}

moe_status_t nvfp4_amax(const void* in, int64_t M, int64_t N, uint32_t sign_mask, float* amax,
                        float* amax_rht, moe_stream_t stream) {
  if (M < 0 || N < 0) return fail(MOE_ERR_INVALID_ARG, "negative size");
  if (!amax) return fail(MOE_ERR_INVALID_ARG, "amax is NULL");
  if (N % 64) return fail(MOE_ERR_UNSUPPORTED, "N must be a multiple of 64");
  if (amax_rht && M % 16) return fail(MOE_ERR_UNSUPPORTED, "M must be a multiple of 16");
  if (N / 64 > 65535) return fail(MOE_ERR_UNSUPPORTED, "N too large");
  if (M > 0 && N > 0 && (!in || !aligned16(in)))
    return fail(MOE_ERR_INVALID_ARG, "in must be non-NULL, 16B aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), s);
  if (e == cudaSuccess && amax_rht) e = cudaMemsetAsync(amax_rht, 0, sizeof(float), s);
  if (e != cudaSuccess) return cuda_fail(e, "memset amax");
  if (M > 0 && N > 0) {
    if (amax_rht)
      launch_nvfp4_rht_amax(in, M, N, sign_mask & 0xFFFFu, amax, amax_rht, s);
    else
      launch_nvfp4_amax(in, M * N, amax, device_sms(), s);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "nvfp4_amax launch");
  return MOE_OK;
}

moe_status_t nvfp4_quantize(const void* in, int64_t M, int64_t N, const float* amax_row,
                            const float* amax_col, int32_t rht, uint32_t sign_mask,
                            uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                            moe_stream_t stream) {
  const bool row = q_row || s_row, col = q_col || s_col;
  if (!row && !col) return fail(MOE_ERR_INVALID_ARG, "neither copy requested");
  if (!nvfp4_quantize_shape_ok(M, N))
    return fail(MOE_ERR_UNSUPPORTED, "M must be a positive multiple of 128, N of 64");
  if (!in || !aligned16(in)) return fail(MOE_ERR_INVALID_ARG, "in must be non-NULL, 16B aligned");
  auto a32 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; };
  auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (row && (!q_row || !s_row || !amax_row || !a32(q_row) || !a4(s_row)))
    return fail(MOE_ERR_INVALID_ARG,
                "row-wise copy needs q_row (32B aligned), s_row (4B aligned) and amax_row");
  if (col && (!q_col || !s_col || !amax_col || !a32(q_col) || !a4(s_col)))
    return fail(MOE_ERR_INVALID_ARG,
                "transposed copy needs q_col (32B aligned), s_col (4B aligned) and amax_col");
  Nvfp4QuantArgs a;
  memset(&a, 0, sizeof(a));
  a.in = in;
  a.M = M;
  a.N = N;
  a.G = M;
  a.Gp = M;
  a.amax_row = amax_row;
  a.amax_col = amax_col;
  a.q_row = row ? q_row : nullptr;
  a.s_row = s_row;
  a.s_row_pad = M;
  a.q_col = col ? q_col : nullptr;
  a.s_col = s_col;
  a.s_col_pad = round128(N);
  a.rht = rht ? 1 : 0;
  a.rht_mask = sign_mask & 0xFFFFu;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!launch_nvfp4_quantize(a, std::max(device_sms(), 1), s))
    return fail(MOE_ERR_CUDA, "nvfp4_quantize: tensor map or shared-memory limit");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "nvfp4_quantize launch");
  return MOE_OK;
}

moe_status_t moe_pack_fc1_weight(const void* src, void* dst, int32_t E, int32_t H, int32_t F,
                                 int32_t gated, int32_t ilv, int32_t inverse,
                                 moe_stream_t stream) {
  if (!src || !dst) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (src == dst) return fail(MOE_ERR_INVALID_ARG, "in-place repacking is not supported");
  if (E < 1 || H <= 0 || F <= 0) return fail(MOE_ERR_INVALID_ARG, "bad sizes");
  if (H % 32 || F % 32) return fail(MOE_ERR_UNSUPPORTED, "H and F must be multiples of 32");
  if (gated && (ilv <= 0 || ilv % 32 || F % ilv))
    return fail(MOE_ERR_UNSUPPORTED, "ilv must be a multiple of 32 dividing F");
  const int N1 = gated ? 2 * F : F;
  const int64_t tiles = (int64_t)E * (N1 / 32) * (H / 32);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  launch_kernel(pack_fc1_kernel, grid_for(tiles, 16), 256, 0, s, nullptr, 0, static_cast<const uint16_t*>(src),
                                                     static_cast<uint16_t*>(dst), E, H, F, N1,
                                                     gated ? 1 : 0, ilv, inverse ? 1 : 0);
  count_launch(s, MOE_K_PACK_FC1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "pack launch");
  return MOE_OK;
}

moe_status_t moe_get_error(const moe_layer_desc_t* d, const void* ws, int32_t* host_code,
                           moe_stream_t stream) {
  if (!ws || !host_code) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  (void)d;  // the error word is at offset 0 of every layout
  cudaError_t e = cudaMemcpyAsync(host_code, ws, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "moe_get_error copy");
  return MOE_OK;
}

moe_status_t moe_clear_error(const moe_layer_desc_t* d, void* ws, moe_stream_t stream) {
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  (void)d;
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "moe_clear_error memset");
  return MOE_OK;
}

int32_t moe_gemm_ctas(const moe_layer_desc_t* desc) {
  if (!desc) return 0;
  return gemm_ctas(desc);
}

uint64_t moe_launch_count(void) { return g_launches.load(); }

moe_status_t moe_timeline_begin(void* const* events, int32_t capacity) {
  if (!events || capacity <= 0) return fail(MOE_ERR_INVALID_ARG, "timeline needs events");
  if (capacity > 4096) return fail(MOE_ERR_UNSUPPORTED, "timeline capacity above 4096");
  g_tl_events = reinterpret_cast<cudaEvent_t*>(const_cast<void**>(events));
  g_tl_cap = capacity;
  g_tl_n = 0;
  return MOE_OK;
}

int32_t moe_timeline_end(int32_t* kernel_ids) {
  const int n = g_tl_n;
  if (kernel_ids)
    for (int i = 0; i < n; ++i) kernel_ids[i] = g_tl_ids[i];
  g_tl_events = nullptr;
  g_tl_cap = 0;
  g_tl_n = 0;
  return n;
}

const char* moe_last_error_string(void) { return g_last_error.c_str(); }

}  // extern "C"
