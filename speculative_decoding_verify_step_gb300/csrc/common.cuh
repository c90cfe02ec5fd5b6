// Shared device helpers: inline PTX for mbarriers, TMA, PDL, ldmatrix/mma, and
// the device status word.  sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify.h"

#ifndef SPEC_DEVICE_INLINE
#define SPEC_DEVICE_INLINE __device__ __forceinline__
#endif

namespace spec {

constexpr int kPage = 64;            // tokens per KV page
constexpr int kMaxWidth = 16;        // rows per sequence per forward
constexpr unsigned long long kWaitBudgetCycles = 4000000000ull;  // ~2 s at 2 GHz

// Compute format of activations, the KV cache and the stored weights: fp16.  The
// bf16 weights are re-encoded exactly as fp16 times a per-row power of two (the
// projection epilogue multiplies the row back by 2^-e), which keeps the weight
// values and their bytes while giving activations 11 significant bits instead
// of 8; accumulation is fp32 throughout.
using act_t = __half;
SPEC_DEVICE_INLINE act_t to_act(float x) { return __float2half_rn(fminf(fmaxf(x, -65504.f), 65504.f)); }
// Four values as four consecutive act_t (8 bytes, for one aligned store).
SPEC_DEVICE_INLINE uint2 pack_act4(float a, float b, float c, float d) {
  __half2 lo = __halves2half2(to_act(a), to_act(b));
  __half2 hi = __halves2half2(to_act(c), to_act(d));
  uint2 r;
  r.x = *reinterpret_cast<uint32_t*>(&lo);
  r.y = *reinterpret_cast<uint32_t*>(&hi);
  return r;
}

// ---------------------------------------------------------------- status word
// First error wins; kernels that hit an error skip the offending accesses.
SPEC_DEVICE_INLINE void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ----------------------------------------------------------- smem addressing
SPEC_DEVICE_INLINE uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
SPEC_DEVICE_INLINE void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

SPEC_DEVICE_INLINE void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

SPEC_DEVICE_INLINE void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

SPEC_DEVICE_INLINE void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

SPEC_DEVICE_INLINE void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

SPEC_DEVICE_INLINE bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: returns false (and records SPEC_ERR_TIMEOUT) if the phase with
// the given parity has not completed within the cycle budget.
SPEC_DEVICE_INLINE bool mbar_wait(uint64_t* bar, uint32_t parity, int* status,
                                  unsigned long long budget = kWaitBudgetCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = clock64();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > budget) {
      set_status(status, SPEC_ERR_TIMEOUT);
      return false;
    }
  }
}

// ----------------------------------------------------------------------- TMA
SPEC_DEVICE_INLINE void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Hint: bring [src, src + bytes) into L2 (bulk copy engine; nothing waits on it).
// src 16-byte aligned, bytes a multiple of 16.
SPEC_DEVICE_INLINE void l2_prefetch_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}

// This CTA's share (by linear block index) of [base, base + bytes) brought into
// L2 in pieces of at most 64 KB; bytes a multiple of 16.
SPEC_DEVICE_INLINE void l2_prefetch_share(const void* base, unsigned long long bytes) {
  if (!base || bytes == 0) return;
  const unsigned long long nblk = (unsigned long long)gridDim.x * gridDim.y * gridDim.z;
  const unsigned long long cta = blockIdx.x + (unsigned long long)gridDim.x * (blockIdx.y + (unsigned long long)gridDim.y * blockIdx.z);
  const unsigned long long units = bytes >> 4;  // 16-byte units
  const unsigned long long u1 = units * (cta + 1) / nblk;
  const char* b = static_cast<const char*>(base);
  for (unsigned long long u = units * cta / nblk; u < u1; u += 4096) {
    const unsigned long long n = u1 - u < 4096 ? u1 - u : 4096;
    l2_prefetch_bulk(b + (u << 4), (uint32_t)(n << 4));
  }
}

// 2-D tiled load (coordinates: c0 innermost, in elements) completing on `bar`.
SPEC_DEVICE_INLINE void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 eviction-priority hint (weights are streamed exactly once).
SPEC_DEVICE_INLINE void tma_load_2d_hint(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// CTA-pair form of the two loads above: the box lands in this CTA's shared memory
// and completes on `bar`, a shared::cluster address that may be the peer CTA's
// barrier (the pair's MMA-issuing CTA counts both CTAs' bytes on its own barrier).
SPEC_DEVICE_INLINE void tma_load_2d_pair(void* dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

SPEC_DEVICE_INLINE void tma_load_2d_pair_hint(void* dst, const CUtensorMap* map, int c0, int c1, uint32_t bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}

SPEC_DEVICE_INLINE uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------ programmatic dependent launch
// No-ops unless the kernel was launched with programmatic stream serialization.
// ------------------------------------------------ thread-block cluster helpers
// Cluster barrier in two halves: arrive (release: this thread's prior shared
// memory writes become visible to the cluster) and wait (acquire).  Every thread
// of every CTA in the cluster takes part, a whole warp at a time.
SPEC_DEVICE_INLINE void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
SPEC_DEVICE_INLINE void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Shared-memory address `a` of this CTA mapped into the shared memory of cluster
// rank `rank` (same offset there).
SPEC_DEVICE_INLINE uint32_t mapa_u32(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

SPEC_DEVICE_INLINE float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

SPEC_DEVICE_INLINE float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// This CTA's rank within its cluster.
SPEC_DEVICE_INLINE uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

SPEC_DEVICE_INLINE uint32_t sm_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}

SPEC_DEVICE_INLINE uint32_t ld_dsmem_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

SPEC_DEVICE_INLINE void st_dsmem_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

SPEC_DEVICE_INLINE void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
SPEC_DEVICE_INLINE void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------ ldmatrix / mma
SPEC_DEVICE_INLINE void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

SPEC_DEVICE_INLINE void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

SPEC_DEVICE_INLINE void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D(16x8 fp32) += A(16x16 f16, row) * B(16x8 f16, col)
SPEC_DEVICE_INLINE void mma_f16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                      uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

SPEC_DEVICE_INLINE uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of element (row, col) in a tile whose rows are 128 bytes (64 halves)
// stored with the TMA 128-byte swizzle: 16-byte chunk j of row r lives at chunk
// j ^ (r % 8).  The tile base must be 1024-byte aligned.
SPEC_DEVICE_INLINE uint32_t swz128(int row, int col_elem) {
  return static_cast<uint32_t>(row * 128 + ((((col_elem >> 3) ^ (row & 7)) & 7) << 4) + ((col_elem & 7) << 1));
}

// ------------------------------------------------------------------- tcgen05
// Tensor memory: allocation is warp-wide; the TMEM address lands in shared memory.
SPEC_DEVICE_INLINE void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
SPEC_DEVICE_INLINE void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
SPEC_DEVICE_INLINE void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
SPEC_DEVICE_INLINE void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
SPEC_DEVICE_INLINE void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// CTA-pair (cta_group::2) forms: one warp of each CTA of the pair takes part in
// the allocation and in the release; both get the same column address.
SPEC_DEVICE_INLINE void tmem_alloc2(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
SPEC_DEVICE_INLINE void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
SPEC_DEVICE_INLINE void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row core
// groups 1024 bytes apart (the layout a TMA 128B-swizzled box of 64 16-bit columns
// produces).  Start address, LBO (unused for this layout), SBO, descriptor
// version 1, swizzle mode 2 (128B).
SPEC_DEVICE_INLINE uint64_t sdesc_k_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// Instruction descriptor of kind::f16 with f16 A and B (format 0), fp32 D (format 1),
// both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
SPEC_DEVICE_INLINE void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}

// Pair MMA, issued by one thread of the pair's even CTA: A = 256 rows (128 from
// each CTA's shared memory at the descriptor's address), B = N rows (N/2 from
// each CTA), D = 128 lanes x N columns in each CTA's tensor memory.
SPEC_DEVICE_INLINE void tc_mma2(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}

// Arrive on the barrier at `bar`'s offset in every CTA of `cta_mask` (cluster
// ranks) when every pair MMA this thread issued so far has completed.
SPEC_DEVICE_INLINE void tc_commit2_mc(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// Arrive on `bar` when every MMA this thread issued so far has completed.
SPEC_DEVICE_INLINE void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 lanes x 16 columns of fp32 from TMEM: thread i gets lane (row) base+i, columns c..c+15.
SPEC_DEVICE_INLINE void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------ block reductions
template <typename T>
SPEC_DEVICE_INLINE T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

SPEC_DEVICE_INLINE float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace spec
