// moe_route_permute_noalloc: the route + permute step for callers that cannot allocate device
// memory. Its scratch (the per-pair row map, the per-row source index and probability, and a
// device error word) lives in one file-scope __device__ array below instead of a caller
// workspace; the caller still passes every input and output.
//
// The array is a module global: every GPU that loads this library holds it until the process
// exits, and every call on a device shares it (the contents of the previous call remain), so
// calls whose execution overlaps on the GPU race on it.
#include <mutex>

#include "kernels.cuh"

namespace moe {

// Limits of the static scratch: T_max * k routed pairs, and R_cap = T_max * k + E * (align-1)
// rows for E <= 256 experts and any BF16 segment alignment (32, 64 or 128).
constexpr int64_t kNoallocMaxPairs = 131072;
constexpr int64_t kNoallocMaxRows = kNoallocMaxPairs + 256 * 127;
constexpr size_t kNoallocErrBytes = 256;
constexpr size_t kNoallocBytes =
    kNoallocErrBytes + (size_t)kNoallocMaxPairs * 4 + (size_t)kNoallocMaxRows * 4 * 2;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocBytes];

// Host-side device addresses of g_noalloc_scratch, one per device (the symbol's name in host
// code is only a host stand-in; the device address must come from cudaGetSymbolAddress),
// each with the id of the CUDA context it was looked up in. A context that is destroyed and
// created again (cudaDeviceReset, a primary context reset) loads the module again, possibly
// at another address: a call whose current context has another id looks the address up again.
static std::mutex g_noalloc_mu;
static void* g_noalloc_ptr[128];
static unsigned long long g_noalloc_ctx[128];

// Id of the calling thread's current context (0 when none is current or the driver entry
// points are unavailable), through the runtime's driver entry-point lookup so that the
// library does not link the driver library itself.
typedef int (*ctx_get_current_fn)(void**);
typedef int (*ctx_get_id_fn)(void*, unsigned long long*);
static unsigned long long current_ctx_id() {
  static ctx_get_current_fn get_cur = nullptr;
  static ctx_get_id_fn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void* f0 = nullptr;
    void* f1 = nullptr;
    cudaDriverEntryPointQueryResult q0, q1;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f0, 12000, cudaEnableDefault,
                                         &q0) == cudaSuccess &&
        q0 == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f1, 12000, cudaEnableDefault, &q1) ==
            cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess) {
      get_cur = reinterpret_cast<ctx_get_current_fn>(f0);
      get_id = reinterpret_cast<ctx_get_id_fn>(f1);
    }
    looked_up = true;
  }
  if (!get_cur || !get_id) return 0;
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (get_cur(&ctx) != 0 || ctx == nullptr || get_id(ctx, &id) != 0) return 0;
  return id;
}

static moe_status_t noalloc_scratch(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 128) {
    set_last_error("moe_route_permute_noalloc: no usable current device");
    return MOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  const unsigned long long ctx = current_ctx_id();
  if (!g_noalloc_ptr[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      set_last_error("moe_route_permute_noalloc: cudaGetSymbolAddress failed");
      return MOE_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
    // the look-up made the device's primary context current if none was
    g_noalloc_ctx[dev] = current_ctx_id();
  }
  *out = g_noalloc_ptr[dev];
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_route_permute_noalloc(const moe_layer_desc_t* d, int32_t T,
                                                  const float* logits, const void* x,
                                                  int32_t* topk_ids, float* topk_probs,
                                                  int32_t* counts, int32_t* offsets,
                                                  void* x_perm, int64_t x_perm_rows,
                                                  moe_stream_t stream) {
  if (!d) {
    set_last_error("moe_route_permute_noalloc: desc is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  if (moe_workspace_size(d) == 0) return MOE_ERR_INVALID_ARG;  // message set by validation
  if (d->precision != MOE_PREC_BF16) {
    set_last_error("moe_route_permute_noalloc: only BF16 x_perm is produced");
    return MOE_ERR_UNSUPPORTED;
  }
  const int64_t pairs = (int64_t)d->T_max * d->k;
  const int64_t R_cap = pairs + (int64_t)d->E * (d->align - 1);
  if (pairs > kNoallocMaxPairs) {
    set_last_error("moe_route_permute_noalloc: T_max*k exceeds the static scratch limit of "
                   "131072 routed (token, expert) pairs");
    return MOE_ERR_UNSUPPORTED;
  }
  if (R_cap > kNoallocMaxRows) {
    set_last_error("moe_route_permute_noalloc: T_max*k + E*(align-1) exceeds the static "
                   "scratch limit of 163584 permuted rows");
    return MOE_ERR_UNSUPPORTED;
  }
  if (T < 0 || T > d->T_max) {
    set_last_error("moe_route_permute_noalloc: T outside [0, T_max]");
    return MOE_ERR_INVALID_ARG;
  }
  if ((T > 0 && (!logits || !x || !topk_ids || !topk_probs)) || !counts || !offsets ||
      !x_perm) {
    set_last_error("moe_route_permute_noalloc: NULL tensor pointer");
    return MOE_ERR_INVALID_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(x_perm) & 15u)) {
    set_last_error("moe_route_permute_noalloc: x and x_perm must be 16-byte aligned");
    return MOE_ERR_INVALID_ARG;
  }
  if (x_perm_rows < R_cap) {
    set_last_error("moe_route_permute_noalloc: x_perm needs T_max*k + E*(align-1) rows");
    return MOE_ERR_INVALID_ARG;
  }
  void* base = nullptr;
  moe_status_t st = noalloc_scratch(&base);
  if (st != MOE_OK) return st;
  uint8_t* b = static_cast<uint8_t*>(base);
  int* err = reinterpret_cast<int*>(b);
  int32_t* row_of = reinterpret_cast<int32_t*>(b + kNoallocErrBytes);
  int32_t* src_of = row_of + kNoallocMaxPairs;
  float* row_prob = reinterpret_cast<float*>(src_of + kNoallocMaxRows);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  // the error word and the counts start at zero on every call
  cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * d->E, s);
  if (e != cudaSuccess) {
    set_last_error("moe_route_permute_noalloc: memset failed");
    return MOE_ERR_CUDA;
  }
  if (T > 0) {
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((T + 7) / 8, (int64_t)sms * 8));
    launch_kernel(route_topk_kernel, grid, 256, 0, s, nullptr, 0, logits, T, d->E, d->k, topk_ids, topk_probs, counts);
    count_launch(s, MOE_K_ROUTE_TOPK);
  }
  launch_kernel(assign_rows_kernel, d->E, 1024, 0, s, nullptr, 0, topk_ids, topk_probs, counts, T, d->E, d->k, d->align,
                                           R_cap, offsets, row_of, src_of, row_prob, err);
  count_launch(s, MOE_K_ASSIGN_ROWS);
  const int ggrid = (int)std::max<int64_t>(1, std::min<int64_t>(R_cap, (int64_t)sms * 8));
  launch_kernel(gather_rows_kernel, ggrid, 256, 0, s, nullptr, 0, static_cast<const uint4*>(x), src_of, offsets, d->E,
                                           d->k, d->H / 8, R_cap, static_cast<uint4*>(x_perm));
  count_launch(s, MOE_K_GATHER_X);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_error(cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
