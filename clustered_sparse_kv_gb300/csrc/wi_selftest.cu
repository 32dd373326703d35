// wi_selftest.cu -- the bounded-wait path, exercised on purpose.
//
// Every mbarrier wait in the library's kernels gives up after about 2^31 SM
// cycles, records WI_DEVERR_MBAR_TIMEOUT in the kernel's error word and
// returns (wi_pipe.cuh).  This entry point runs that same wait on a barrier
// that nothing ever completes, so a test can check that the wait ends, that
// the error is recorded, and that the context stays usable afterwards -- the
// failure path checked without faulting or hanging the device.
#include <cuda_runtime.h>

#include <cstdio>

#include "wave_index.h"
#include "wi_common.cuh"
#include "wi_internal.h"
#include "wi_pipe.cuh"

namespace {

__global__ void k_wait_unfinished_barrier(int* err, int* returned) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected, none made
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool done = mbar_wait(&bar, 0, err);  // bounded: returns false after ~2^31 cycles
    *returned = done ? 2 : 1;
  }
}

}  // namespace

static int st_fail(int code, const char* what, cudaError_t e) {
  char msg[256];
  snprintf(msg, sizeof(msg), "wi_selftest_wait_timeout: %s%s%s", what, e != cudaSuccess ? ": " : "",
           e != cudaSuccess ? cudaGetErrorString(e) : "");
  wi_set_error(msg);
  return code;
}

extern "C" int wi_selftest_wait_timeout(int* device_error, int* wait_returned) {
  if (!device_error || !wait_returned) return st_fail(WI_EINVAL, "null output pointer", cudaSuccess);
  int* d = nullptr;
  cudaError_t e = cudaMalloc(&d, 2 * sizeof(int));
  if (e != cudaSuccess) return st_fail(WI_ENOMEM, "cudaMalloc", e);
  int h[2] = {0, 0};
  if ((e = cudaMemset(d, 0, 2 * sizeof(int))) == cudaSuccess) {
    k_wait_unfinished_barrier<<<1, 32>>>(d, d + 1);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  }
  cudaFree(d);
  if (e != cudaSuccess) return st_fail(WI_ECUDA, "launch or copy", e);
  *device_error = h[0];
  *wait_returned = h[1];
  return WI_OK;
}
