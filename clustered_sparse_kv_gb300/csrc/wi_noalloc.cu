// wi_noalloc.cu -- wi_kmeans_step_noalloc: one spherical k-means round that
// allocates nothing.
//
// Some callers cannot allocate device memory when they run a clustering
// round.  A serving process usually hands almost all of the GPU's memory to
// its KV-cache pool at start-up, so a later cudaMalloc / cudaMallocAsync
// fails or has to evict cache blocks; other hosts route every device
// allocation through their own arena and forbid direct CUDA allocation.
// This entry point gives them the same round as wi_kmeans_step, with the
// scratch in a fixed, file-scope device array instead of cudaMallocAsync.
//
// The array is kWiNoallocScratchBytes (8 MiB) on every GPU that loads this
// library and stays allocated until the process exits.  All calls share it,
// so two calls whose work overlaps on the GPU (different streams, or
// different host threads without ordering) race on it; calls on one stream
// are ordered and safe.  The array keeps the previous call's contents; the
// only part that must start at zero, the device error word, is cleared on
// every call.  Every call looks up the array's device address
// (cudaGetSymbolAddress, which allocates nothing) with the caller's device
// current, so the address stays right after the device's context has been
// torn down and made again (a cudaDeviceReset reloads the module).
#include <cuda_runtime.h>

#include <cstdio>

#include "wave_index.h"
#include "wi_internal.h"

namespace {

constexpr size_t kWiNoallocScratchBytes = (size_t)8 << 20;

__device__ __align__(256) unsigned char g_wi_noalloc_scratch[kWiNoallocScratchBytes];

int nfail(int code, const char* msg, cudaError_t e = cudaSuccess) {
  char buf[512];
  if (e != cudaSuccess) {
    cudaGetLastError();
    snprintf(buf, sizeof(buf), "%s: %s", msg, cudaGetErrorString(e));
  } else {
    snprintf(buf, sizeof(buf), "%s", msg);
  }
  wi_set_error(buf);
  return code;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

extern "C" int wi_kmeans_step_noalloc(const wi_config* cfg, const void* k, const void* centroids, int32_t* assign,
                                      void* new_centroids, void* stream) {
  wi_set_error("");
  WiGeom g;
  char msg[256];
  int rc = wi_geom_from_config(cfg, &g, msg, sizeof(msg));
  if (rc != WI_OK) return nfail(rc, msg);
  if (!k || !centroids || !assign || !new_centroids)
    return nfail(WI_EINVAL, "k, centroids, assign and new_centroids must be non-NULL");
  // scratch layout inside the static array
  const size_t SU = (size_t)g.U * g.nseg;
  const size_t o_err = 0;
  const size_t o_cnt = align256(o_err + 4);
  const size_t o_off = align256(o_cnt + SU * g.Cs * 4);
  const size_t o_slot = align256(o_off + SU * (g.Cs + 1) * 4);
  const size_t o_chat = align256(o_slot + SU * g.S * 4);
  const size_t need = align256(o_chat + SU * g.Cs * 128 * 2);
  if (need > kWiNoallocScratchBytes) {
    snprintf(msg, sizeof(msg),
             "problem needs %zu bytes of scratch; the no-allocation round is limited to %zu bytes "
             "(about 400K tokens at 512 clusters per 8192-token segment): use wi_kmeans_step",
             need, kWiNoallocScratchBytes);
    return nfail(WI_EINVAL, msg);
  }
  // host code may not use the symbol itself as a device pointer: ask for this device's address
  void* sym = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&sym, g_wi_noalloc_scratch);
  if (e != cudaSuccess || !sym) return nfail(WI_ECUDA, "cudaGetSymbolAddress(no-allocation scratch)", e);
  unsigned char* base = static_cast<unsigned char*>(sym);
  int* err = reinterpret_cast<int*>(base + o_err);
  int* seg_counts = reinterpret_cast<int*>(base + o_cnt);
  int* seg_offsets = reinterpret_cast<int*>(base + o_off);
  int* slots = reinterpret_cast<int*>(base + o_slot);
  void* chat = base + o_chat;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t cb = SU * g.Cs * 128 * 2;
  if ((e = cudaMemsetAsync(err, 0, 4, st)) != cudaSuccess) return nfail(WI_ECUDA, "clear error word", e);
  if ((e = cudaMemcpyAsync(chat, centroids, cb, cudaMemcpyDeviceToDevice, st)) != cudaSuccess)
    return nfail(WI_ECUDA, "copy centroids", e);
  if ((e = wi_launch_assign(g, k, chat, assign, err, st)) != cudaSuccess) return nfail(WI_ECUDA, "assign", e);
  if ((e = wi_launch_segment_sort(g, assign, seg_counts, seg_offsets, slots, err, st)) != cudaSuccess)
    return nfail(WI_ECUDA, "segment sort", e);
  if ((e = wi_launch_centroid_update(g, k, seg_counts, seg_offsets, slots, chat, st)) != cudaSuccess)
    return nfail(WI_ECUDA, "centroid update", e);
  if ((e = cudaMemcpyAsync(new_centroids, chat, cb, cudaMemcpyDeviceToDevice, st)) != cudaSuccess)
    return nfail(WI_ECUDA, "copy centroids out", e);
  int herr = 0;
  if ((e = cudaMemcpyAsync(&herr, err, 4, cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess)
    return nfail(WI_ECUDA, "read error word", e);
  if (herr) return nfail(WI_EDEVICE, "device invariant violated");
  return WI_OK;
}
