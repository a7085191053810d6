// kvq_device.cuh -- small device helpers shared by the kvq kernels (sm_103a):
// status reporting, a wall-clock bound for every wait, mbarriers, bulk and
// tensor TMA copies, warp-level fp16 tensor-core products and the bit tricks
// that turn stored integer codes into exact fp16 values.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvq.h"

namespace kvq {

// ---------------------------------------------------------------------------
// status
// ---------------------------------------------------------------------------

// First error wins: a later error never overwrites an earlier one.
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// Index checks of the debug build (libkvq_debug.so, compiled with
// KVQ_DEBUG=1): KVQ_IN_RANGE(cond, status) is cond there -- and a false cond
// reports KVQ_ERR_BOUNDS, the caller then skipping the access -- and the
// constant true in the shipped library, so the checks cost nothing there.
// They stand in for a memory checker: a check that fails never faults, it
// only records the first failure in the status word.
__device__ __forceinline__ bool debug_in_range(bool ok, int32_t* status) {
  if (!ok) report(status, KVQ_ERR_BOUNDS);
  return ok;
}
#if defined(KVQ_DEBUG) && KVQ_DEBUG
#define KVQ_IN_RANGE(cond, status) (::kvq::debug_in_range((cond), (status)))
#else
#define KVQ_IN_RANGE(cond, status) (static_cast<void>(sizeof((cond) ? 1 : 0)), true)   // unevaluated
#endif

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Every spin in these kernels gives up after a limit (a kernel parameter,
// 2 s unless the caller's policy says otherwise) and reports a timeout.
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s

// ---------------------------------------------------------------------------
// mbarrier (shared memory, CTA scope)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// A translation unit may set KVQ_TRYWAIT_HINT_NS (before including this
// header) to let a waiting thread sleep up to that long inside try_wait
// instead of the hardware's default, so fewer poll iterations are issued; the
// thread still resumes when the phase completes.
#ifndef KVQ_TRYWAIT_HINT_NS
#define KVQ_TRYWAIT_HINT_NS 0
#endif

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
#if KVQ_TRYWAIT_HINT_NS > 0
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase), "n"(KVQ_TRYWAIT_HINT_NS)
      : "memory");
#else
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
#endif
  return ok != 0;
}

// Bounded wait on an mbarrier phase.  Returns false (and reports
// KVQ_ERR_TIMEOUT) if the phase did not complete within limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t phase, int32_t* status, uint64_t limit_ns) {
  if (mbar_try_wait(bar, phase)) return true;
  const uint64_t t0 = global_ns();
  uint32_t n = 0;
  while (!mbar_try_wait(bar, phase)) {
    if ((++n & 255u) == 0 && global_ns() - t0 > limit_ns) {
      report(status, KVQ_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// atomicAdd with release and acquire semantics at GPU scope: the memory
// operations before it (including those of other threads ordered before it by
// a barrier) become visible to whoever reads its result, and the operations
// after it see everything the earlier adders released.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: no-ops unless the kernel was launched with
// the programmatic stream serialization attribute
// ---------------------------------------------------------------------------

// Wait until the grids this one depends on have completed and their memory
// operations are visible.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next dependent grid in the stream to be scheduled.
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA: 1D bulk copy and 2D tensor copy into shared memory, completing on an
// mbarrier (transaction bytes).
// ---------------------------------------------------------------------------

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_2d_g2s(void* dst, const void* tmap, int32_t x, int32_t y,
                                           uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// L2 policy for data read once per call: its lines are the first to go, so
// the small buffers a call re-reads (lengths, queries, split partials) stay.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_2d_g2s_hint(void* dst, const void* tmap, int32_t x, int32_t y, uint64_t* bar,
                                                uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// L2 prefetches (no data returned to the program, no completion to wait for)
__device__ __forceinline__ void prefetch_l2_tile_2d(const void* tmap, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(tmap), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ---------------------------------------------------------------------------
// warp-level tensor-core product D = A(16x16 fp16) * B(16x8 fp16) + C (fp32)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Same product with a zero accumulator: d = A * B.
__device__ __forceinline__ void mma_16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// ---------------------------------------------------------------------------
// ldmatrix: lane l supplies the shared address of row (l & 7) of matrix (l >> 3);
// thread (g = lane/4, t = lane%4) receives, per matrix, the 16-bit elements
// (row g, cols 2t, 2t+1), or with .trans (rows 2t, 2t+1, col g).
// ---------------------------------------------------------------------------

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(saddr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}

// ---------------------------------------------------------------------------
// codes -> fp16.  An fp16 whose top byte is 0x64 and low byte is c has the
// value 1024 + c exactly (exponent 2^10, ten mantissa bits), for 0 <= c < 1024.
// Subtracting (1024 + z) in fp16 then gives the exact integer c - z.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// bytes 0,1 of w -> half2(1024 + w.b0, 1024 + w.b1)
__device__ __forceinline__ uint32_t bytes01_biased(uint32_t w) { return prmt(w, 0x64646464u, 0x5140u); }
// bytes 2,3 of w -> half2(1024 + w.b2, 1024 + w.b3)
__device__ __forceinline__ uint32_t bytes23_biased(uint32_t w) { return prmt(w, 0x64646464u, 0x7362u); }
// bytes 0,2 of w -> half2(1024 + w.b0, 1024 + w.b2); bytes 1,3 likewise
__device__ __forceinline__ uint32_t bytes02_biased(uint32_t w) { return prmt(w, 0x64646464u, 0x5240u); }
__device__ __forceinline__ uint32_t bytes13_biased(uint32_t w) { return prmt(w, 0x64646464u, 0x5341u); }
// nibbles at bits [0,4) and [16,20) of w -> half2(1024 + lo, 1024 + hi)
__device__ __forceinline__ uint32_t nib_biased(uint32_t w) { return (w & 0x000F000Fu) | 0x64006400u; }

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b), *reinterpret_cast<__half2*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}

// The fp16 pair (1024 + n, 1024 + n') of the nibbles at bits 4-7 and 20-23,
// without a shift: masked in place the word is the pair (1024 + 16 n, ...),
// and x / 16 + 960 = 1024 + n, every step exact (one FMA on the FMA pipe
// instead of a shift on the ALU pipe).  nib_hi_biased(w) == nib_biased(w >> 4).
constexpr uint32_t kHalf2Sixteenth = 0x2C002C00u;   // (1/16, 1/16)
__device__ __forceinline__ uint32_t nib_hi_biased(uint32_t w) {
  return hfma2_u32((w & 0x00F000F0u) | 0x64006400u, kHalf2Sixteenth, 0x63806380u /* (960, 960) */);
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Transpose of an 8x8 matrix of 16-bit elements held one register per lane
// (lane l: row l/4, columns 2(l%4), 2(l%4)+1): afterwards the lane holds
// row l/4, columns 2(l%4), 2(l%4)+1 of the transposed matrix.
__device__ __forceinline__ uint32_t movm_trans(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float half_lo(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}
// (1024 + z) broadcast to both halves, from a scale/zero word (zero in the high half)
__device__ __forceinline__ uint32_t zero_biased2(uint32_t sz) {
  __half z = __ushort_as_half(static_cast<unsigned short>(sz >> 16));
  __half zb = __hadd(z, __ushort_as_half(0x6400));  // exact: z is an integer <= 255
  __half2 r = __halves2half2(zb, zb);
  return *reinterpret_cast<uint32_t*>(&r);
}
// half2(s_a, s_b): the fp16 scales of two scale/zero words
__device__ __forceinline__ uint32_t scale_pair(uint32_t sz_a, uint32_t sz_b) { return prmt(sz_a, sz_b, 0x5410u); }
// half2((1024 + z_a), (1024 + z_b)) from two scale/zero words
__device__ __forceinline__ uint32_t zero_biased_pair(uint32_t sz_a, uint32_t sz_b) {
  uint32_t zz = prmt(sz_a, sz_b, 0x7632u);  // high halves: z_a | z_b << 16
  __half2 r = __hadd2(*reinterpret_cast<__half2*>(&zz), __halves2half2(__ushort_as_half(0x6400),
                                                                      __ushort_as_half(0x6400)));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace kvq
