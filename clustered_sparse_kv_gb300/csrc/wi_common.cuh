// wi_common.cuh -- device helpers shared by the wave-index kernels.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define WI_D 128  // head size

typedef __nv_bfloat16 bf16;

// Device-side invariant violations: kernels OR a bit into the index's error
// word instead of trapping; the host reads it in wi_check_device.
enum {
  WI_DEVERR_UNION_OVERFLOW = 1,
  WI_DEVERR_BAD_CLUSTER = 2,
  WI_DEVERR_BAD_ROW = 4,
  WI_DEVERR_TOPK = 8,
  WI_DEVERR_MBAR_TIMEOUT = 16,
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// 4 consecutive bf16 (8 bytes) -> 4 floats
__device__ __forceinline__ void load_bf16x4(const bf16* p, float (&x)[4]) {
  const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
  x[0] = bf16_lo(w.x);
  x[1] = bf16_hi(w.x);
  x[2] = bf16_lo(w.y);
  x[3] = bf16_hi(w.y);
}

__device__ __forceinline__ uint2 ldg_u2(const void* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }

__device__ __forceinline__ void unpack_bf16x4(uint2 w, float (&x)[4]) {
  x[0] = bf16_lo(w.x);
  x[1] = bf16_hi(w.x);
  x[2] = bf16_lo(w.y);
  x[3] = bf16_hi(w.y);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int warp_isum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Order-preserving map of a float to uint32 (larger float -> larger key).
// Key 0 is never produced by a finite float and marks "not a candidate".
__device__ __forceinline__ uint32_t float_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);  // -0 -> +0: equal scores, equal keys
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inclusive warp scan of ints.
__device__ __forceinline__ int warp_inclusive_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Exclusive block scan of one int per thread; `tmp` holds >= 32 ints of
// shared memory; returns the exclusive prefix and writes the block total.
// All threads of the block must call it.
__device__ __forceinline__ int block_exclusive_scan(int v, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  const int inc = warp_inclusive_scan(v);
  __syncthreads();
  if (lane == 31) tmp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int s = lane < nw ? tmp[lane] : 0;
    s = warp_inclusive_scan(s);
    tmp[lane] = s;
  }
  __syncthreads();
  const int base = warp > 0 ? tmp[warp - 1] : 0;
  const int tot = tmp[nw - 1];
  __syncthreads();  // tmp may be reused by the next call
  if (total) *total = tot;
  return base + inc - v;
}

// Raise a kernel's dynamic shared-memory limit once per size increase and per
// device (not on every launch, so that launches inside a stream capture make
// no attribute calls once warmed up; the attribute belongs to the current
// device's context, so a process that uses several devices sets it on each).
// `cur` is a per-kernel static array indexed by device ordinal.
constexpr int kWiSmemDevices = 64;
template <typename F>
inline cudaError_t wi_ensure_smem(F* func, size_t bytes, int (&cur)[kWiSmemDevices]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kWiSmemDevices;
  if (cached && (int)bytes <= cur[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && cached) cur[dev] = (int)bytes;
  return e;
}
