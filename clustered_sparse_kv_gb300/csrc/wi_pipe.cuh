// wi_pipe.cuh -- shared-memory staging with bulk asynchronous copies and
// mbarriers (sm_90+ PTX), plus the warp transpose-reduction.
#pragma once
#include "wi_common.cuh"

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Arrive once and add `bytes` to the transaction count of the current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed.  The wait is
// bounded: after about 2^31 SM cycles (~1 s) without completion it records
// WI_DEVERR_MBAR_TIMEOUT and returns false, so no kernel can spin forever.
constexpr long long kMbarWaitCycles = 1LL << 31;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0u && clock64() - t0 > kMbarWaitCycles) break;
  }
  atomicOr(err, WI_DEVERR_MBAR_TIMEOUT);
  return false;
}

// Bulk copy global -> this CTA's shared memory, completion counted on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Transpose-reduction across a warp: every lane holds NV partial values
// (NV = 8, 16 or 32) of NV different sums.  Afterwards lane l holds the full
// sum of index (l >> (5 - log2 NV)) in v[0].  Halving exchanges first (each
// lane keeps the half whose index bit matches its lane bit), then plain
// butterfly additions for the remaining lane bits.
template <int NV>
__device__ __forceinline__ float transpose_reduce(float (&v)[NV]) {
  static_assert(NV == 8 || NV == 16 || NV == 32, "NV");
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int half = NV / 2, off = 16; half >= 1; half >>= 1, off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float r = v[0];
  constexpr int rest = NV == 32 ? 0 : NV == 16 ? 1 : 2;  // lane bits not consumed above
#pragma unroll
  for (int b = 0; b < rest; ++b) r += __shfl_xor_sync(0xffffffffu, r, 1 << b);
  return r;
}

// Programmatic dependent launch (kernels launched with the programmatic
// stream-serialization attribute): let the next kernel in the stream be
// scheduled early, and wait for the previous kernel's completion (and the
// visibility of its writes) before touching anything it produces.  Both are
// no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Device-scope acquire-release fetch-and-add (returns the old value).
__device__ __forceinline__ unsigned ticket_acq_rel(unsigned* p) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
  return old;
}
