// Shared device helpers for the sm_103a kernels: bf16 helpers, MXFP8 element conversion,
// mbarrier, TMA (cp.async.bulk.tensor) and tcgen05 (TMEM alloc / MMA / commit / ld) wrappers
// written as inline PTX, plus the sticky device error word.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moegmm.h"

#define MOE_DEVICE __device__ __forceinline__

namespace moe {

// ----------------------------------------------------------------------------- PDL
// Programmatic dependent launch: every kernel waits, before it touches memory, until the
// previous kernel of the stream has completed and its memory is visible; the persistent GEMMs
// let the stream's next kernel be scheduled once their tile loops are done (a grid's exiting
// CTAs count as having let it, so the short kernels need no call). Triggering at kernel entry
// instead was measured slower: the next kernel's waiting CTAs then share the SMs with this
// kernel's work. Both are no-ops when the kernel was not launched with programmatic stream
// serialization.
MOE_DEVICE void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
MOE_DEVICE void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
#define MOE_GRIDDEP_ENTRY() griddep_wait()

// ----------------------------------------------------------------------------- error word
MOE_DEVICE void set_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);  // keep the first error
}

// ----------------------------------------------------------------------------- bf16
MOE_DEVICE float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
MOE_DEVICE float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xFFFF0000u); }
// round-to-nearest-even pack of two floats into bf16x2 (lo in the low half)
MOE_DEVICE uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ----------------------------------------------------------------------------- MXFP8
// floor(log2(|a|)) of a finite, non-zero fp32 value, exactly from its bits.
MOE_DEVICE int floor_log2_f32(float a) {
  uint32_t b = __float_as_uint(a) & 0x7FFFFFFFu;
  int ex = (int)(b >> 23);
  if (ex != 0) return ex - 127;
  // subnormal: value = mant * 2^-149
  return 31 - __clz((int)b) - 149;
}
// E8M0 exponent of a block with maximum magnitude amax: clamp(floor(log2 amax) - 8, -127, 127),
// -127 for an all-zero block.
MOE_DEVICE int mx_block_exponent(float amax) {
  if (!(amax > 0.0f)) return -127;
  int e = floor_log2_f32(amax) - 8;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}
// 2^-e as fp32 for e in [-127, 126] (a normal number, so x * it is exact unless x*2^-e is
// itself below the fp32 normal range, where E4M3 rounds to zero anyway).
MOE_DEVICE float mx_inv_scale(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }
// Two fp32 -> two E4M3 codes, round to nearest even, saturating to +-448; the first
// argument lands in the low byte.
MOE_DEVICE uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Quantise 32 fp32 values (one block) into 32 E4M3 bytes (as 8 words) and return the scale
// byte.
MOE_DEVICE float amax32(const float (&v)[32]) {
  // four independent chains (max is exact, so the grouping does not change the result)
  float m0 = 0.f, m1 = 0.f, m2 = 0.f, m3 = 0.f;
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    m0 = fmaxf(m0, fabsf(v[i]));
    m1 = fmaxf(m1, fabsf(v[i + 1]));
    m2 = fmaxf(m2, fabsf(v[i + 2]));
    m3 = fmaxf(m3, fabsf(v[i + 3]));
  }
  return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

MOE_DEVICE uint32_t mx_quant_block(const float (&v)[32], uint32_t (&q)[8]) {
  const int e = mx_block_exponent(amax32(v));
  const float inv = mx_inv_scale(e);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t lo = cvt_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv);
    uint32_t hi = cvt_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv);
    q[i] = lo | (hi << 16);
  }
  return (uint32_t)(e + 127);
}

// ----------------------------------------------------------------------------- 256-bit global
// 32 bytes at a 32-byte aligned global address in one access (sm_100 and later).
MOE_DEVICE void st_global_v8(void* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// ----------------------------------------------------------------------------- smem / timer
MOE_DEVICE uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
MOE_DEVICE uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------------------- mbarrier
MOE_DEVICE void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
MOE_DEVICE void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
MOE_DEVICE void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
MOE_DEVICE void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
MOE_DEVICE bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// A wait on a barrier phase that gives up after `limit_ns`, or as soon as another role of
// the CTA has given up (*abort != 0). On giving up it records MOE_DEVERR_TIMEOUT.
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s
MOE_DEVICE bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* err,
                          uint64_t limit_ns = kWaitLimitNs) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(a, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      set_error(err, MOE_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// ----------------------------------------------------------------------------- TMA
MOE_DEVICE void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
MOE_DEVICE void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
MOE_DEVICE void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1,
                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// TMA store of a shared-memory box to a 3-D tensor (out-of-bounds elements are not written),
// tracked in the issuing thread's bulk-async group.
MOE_DEVICE void tma_store_3d(const CUtensorMap* m, const void* src, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
MOE_DEVICE void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until this thread's bulk stores have read their shared-memory sources (reuse is safe).
MOE_DEVICE void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until this thread's bulk stores have completed.
MOE_DEVICE void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Make this thread's shared-memory writes visible to the async (TMA) proxy.
MOE_DEVICE void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------------------- tcgen05
// Allocation is warp-wide (.sync.aligned); the TMEM base address is written to smem.
MOE_DEVICE void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
MOE_DEVICE void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MOE_DEVICE void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
MOE_DEVICE void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
MOE_DEVICE void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
MOE_DEVICE void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on an mbarrier when all previously issued tcgen05.mma of this thread finish.
MOE_DEVICE void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// 32 lanes x 32 consecutive fp32 columns: thread i of the warp receives lane (base+i).
MOE_DEVICE void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}
MOE_DEVICE void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 lanes x 16 consecutive 32-bit columns, both directions.
MOE_DEVICE void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
MOE_DEVICE void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
// 32 lanes x 8 consecutive 32-bit columns, both directions.
MOE_DEVICE void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
MOE_DEVICE void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                   taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
               "r"(r[7])
               : "memory");
}
MOE_DEVICE void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ----------------------------------------------------------------------------- CTA pairs
// A cluster of two CTAs on neighbouring SMs runs one MMA of M = 256 rows (cta_group::2): the
// even-ranked CTA issues it, each CTA holds its 128 rows of A and half of B in shared memory
// and its 128 rows of the accumulator in its own TMEM.
MOE_DEVICE uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
MOE_DEVICE uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
MOE_DEVICE uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Address in the shared::cluster window of the object at `saddr` in CTA `rank`'s memory.
MOE_DEVICE uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Arrive on an mbarrier that may live in the peer CTA (shared::cluster address).
MOE_DEVICE void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Arrive without release semantics: for signals that order no memory accesses of this thread
// (an accumulator whose TMEM loads have all completed), so the arrive does not wait for the
// thread's outstanding global stores.
MOE_DEVICE void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// The same for a barrier in this CTA.
MOE_DEVICE void mbar_arrive_relaxed(uint64_t* bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// Store a flag into the peer CTA's shared memory.
MOE_DEVICE void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v)
               : "memory");
}
// TMA loads into this CTA's shared memory whose completion is counted on an mbarrier that may
// live in the peer CTA of the pair (shared::cluster address, e.g. from mapa_shared).
MOE_DEVICE void tma_load_2d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int c0,
                                 int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}
MOE_DEVICE void tma_load_3d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int c0,
                                 int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Whole-cluster barrier (every thread of both CTAs).
MOE_DEVICE void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
MOE_DEVICE void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
MOE_DEVICE void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
MOE_DEVICE void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D[tmem, both CTAs] (+)= A[smem, 128 rows per CTA] * B[smem, N/2 columns per CTA]^T.
MOE_DEVICE void mma_bf16_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier at the same shared-memory offset in every CTA of `mask` when
// all pair MMAs this thread issued before have completed.
MOE_DEVICE void mma_commit_pair_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma (SM100 format): start address, leading
// and stride byte offsets (all >> 4), version 1 at bit 46, swizzle mode at bits 61..63
// (2 = 128-byte swizzle).
MOE_DEVICE uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D. a_mn / b_mn select MN-major
// operands. N at bits 17..22 (>>3), M at bits 24..28 (>>4).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                       // D format f32
         | (1u << 7)                     // A format bf16
         | (1u << 10)                    // B format bf16
         | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ----------------------------------------------------------------------------- MXFP8 MMA
// Instruction descriptor, kind::mxf8f6f4 block-scaled: E4M3 A and B (format 0), K-major,
// scale factors E8M0 (bit 23), a_sf_id at bits 29..30 and b_sf_id at bits 4..5 select which
// byte of the 32-bit scale-factor column a K=32 step uses.
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N, int sf_id, bool a_mn = false,
                                                  bool b_mn = false) {
  return ((uint32_t)(sf_id & 3) << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24) |
         ((uint32_t)(sf_id & 3) << 29);
}
// D[tmem] (+)= (A * 2^SFA) (B * 2^SFB)^T, E4M3 inputs with per-32 E8M0 scales in TMEM.
MOE_DEVICE void mma_mxf8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::
          "r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Copy a 32-row x 16-byte shared-memory matrix into TMEM (4 columns), replicated into all
// four 32-lane quadrants.
MOE_DEVICE void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
// Pair forms: issued by the leader CTA; each CTA of the pair copies from its own shared
// memory into its own TMEM (scale factors), and the MMA spans both CTAs (M = 256).
MOE_DEVICE void tmem_cp_32x128b_warpx4_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
MOE_DEVICE void mma_mxf8_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                 uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::
          "r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Shared-memory descriptor without swizzle (8-row x 16-byte core matrices, SBO between
// consecutive 8-row groups).
MOE_DEVICE uint64_t smem_desc_noswizzle(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}
// 1-D bulk copy global -> shared, completion counted on an mbarrier (bytes, 16-aligned).
MOE_DEVICE void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Byte offset of scale factor (row, kb) in the MMA-ready scale layout: slabs of 128 rows x 4
// k-blocks (512 bytes), slab (kb/4, row/128) at ((kb/4) * rows_pad + row/128*128) * 4; inside a
// slab, row r = 32*j + i sits in 16-byte line i at bytes 4*j .. 4*j+3 (one per k-block). This is
// the order in which tcgen05.cp.32x128b.warpx4 hands 128 rows x 4 scale bytes to the MMA.
__host__ __device__ inline int64_t sf_mma_offset(int64_t row, int64_t kb, int64_t rows_pad) {
  const int64_t perm = (row & ~(int64_t)127) | ((row & 31) << 2) | ((row >> 5) & 3);
  return ((kb >> 2) * rows_pad + perm) * 4 + (kb & 3);
}

// ----------------------------------------------------------------------------- math
// 1 / (1 + e^-x) with the approximate reciprocal (about 2 ulp): no IEEE-division slow path.
// For x < -87 the denominator overflows to +inf and the quotient is 0, the correct limit.
MOE_DEVICE float sigmoidf_fast(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

}  // namespace moe
