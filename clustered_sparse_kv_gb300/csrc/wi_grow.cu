// wi_grow.cu -- decode-time index maintenance: one more segment from the
// local window.
//
// Segmented clustering (RetroInfer summaries de/fr/zh 2.A) clusters every
// segment of the context on its own, so a segment can be added to a built
// index without touching the others.  The pages describe the index at
// prefill only; this library extends it to decode: appended tokens join the
// local window, and once an append leaves the window holding local_window +
// seg_len rows, its oldest seg_len rows become one more segment (B1-B5 of
// the build on that segment alone) and the window is back to local_window
// rows.  The grown segment's rows are copied into a library-owned buffer
// (cluster-contiguous after its permutation), its clusters take the next
// free cluster ids (reserved, empty, since the index was made), and the
// budget grows with the cluster count.  All of it is enqueued on the
// decode stream: no allocation, no host synchronisation.
#include <cuda_runtime.h>

#include "wi_common.cuh"
#include "wi_internal.h"

namespace {

__global__ void k_set_int(int* p, int v) { *p = v; }

// Rows [w0 + gi*S, w0 + (gi+1)*S) of every unit (w0 = n - W: the build's window start), from the
// caller's cache below position n and from the append buffer above it, into grown segment gi.
__global__ void k_gather_segment(const bf16* __restrict__ K, const bf16* __restrict__ V,
                                 const bf16* __restrict__ appK, const bf16* __restrict__ appV,
                                 bf16* __restrict__ gK, bf16* __restrict__ gV, int U, long long n, int W, int S,
                                 int gi, int amax) {
  const int lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);  // over U * S rows
  if (r >= (long long)U * S) return;
  const int u = (int)(r / S), i = (int)(r % S);
  const long long p = n - W + (long long)gi * S + i;
  const bf16* ks = p < n ? K + ((size_t)u * n + p) * WI_D : appK + ((size_t)u * amax + (p - n)) * WI_D;
  const bf16* vs = p < n ? V + ((size_t)u * n + p) * WI_D : appV + ((size_t)u * amax + (p - n)) * WI_D;
  const size_t d = (((size_t)gi * U + u) * S + i) * WI_D;
  reinterpret_cast<uint2*>(gK + d)[lane] = ldg_u2(ks + 4 * lane);
  reinterpret_cast<uint2*>(gV + d)[lane] = ldg_u2(vs + 4 * lane);
}

// One warp per (unit, cluster j) of the new segment: its count, first row (rows n + gi*S + slot,
// the grown segments' row space), mean key and value sums move to cluster Cb + gi*Cs + j of the
// index; warp 0 of every unit also writes the segment's perm (original positions) and counts its
// non-empty clusters.
__global__ void k_merge_segment(const int* __restrict__ cnt_t, const int* __restrict__ off_t,
                                const bf16* __restrict__ mu_t, const float* __restrict__ vs_t,
                                const int* __restrict__ perm_t, const int* __restrict__ ne_t, int* __restrict__ cnt,
                                int* __restrict__ off, bf16* __restrict__ mu, float* __restrict__ vs,
                                bf16* __restrict__ vs16, int* __restrict__ perm, int* __restrict__ nonempty, int U,
                                int C, int Cb, int Cs, int S, long long n, int W, int n_idx, int pst, int gi) {
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);  // over U * Cs
  if (w >= (long long)U * Cs) return;
  const int u = (int)(w / Cs), j = (int)(w % Cs);
  const long long c = (long long)u * C + Cb + (long long)gi * Cs + j;
  if (lane == 0) {
    cnt[c] = cnt_t[w];
    off[(long long)u * (C + 1) + Cb + (long long)gi * Cs + j] = (int)(n + (long long)gi * S + off_t[(long long)u * (Cs + 1) + j]);
    if (j == Cs - 1) off[(long long)u * (C + 1) + Cb + (long long)(gi + 1) * Cs] = (int)(n + (long long)(gi + 1) * S);
  }
  reinterpret_cast<uint2*>(mu + c * WI_D)[lane] = ldg_u2(mu_t + w * WI_D + 4 * lane);
  const float4 v = reinterpret_cast<const float4*>(vs_t + w * WI_D)[lane];
  reinterpret_cast<float4*>(vs + c * WI_D)[lane] = v;
  if (vs16) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    reinterpret_cast<uint2*>(vs16 + c * WI_D)[lane] =
        make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  }
  if (j == 0) {
    const long long p0 = n - W + (long long)gi * S;
    for (int t = lane; t < S; t += 32)
      perm[(long long)u * pst + n_idx + (long long)gi * S + t] = (int)(p0 + perm_t[(long long)u * S + t]);
    if (lane == 0) nonempty[u] += ne_t[u];
  }
}

}  // namespace

cudaError_t wi_launch_set_int(int* p, int v, cudaStream_t st) {
  k_set_int<<<1, 1, 0, st>>>(p, v);
  return cudaGetLastError();
}

cudaError_t wi_launch_grow(const WiGeom& g, const WiDecodeBufs& b, const WiGrowBufs& w, void* mu, float* valsum,
                           void* valsum16, int* cnt, int* off, int* perm, int* nonempty, int gi, int k_after,
                           int* err, cudaStream_t st) {
  // the segment alone, as a build geometry: U units of S tokens, one segment, no steady zone
  WiGeom s = g;
  s.nseg = 1;
  s.Cb = s.C = g.Cs;
  s.Gmax = 0;
  s.n = g.S;
  s.n_sink = 0;
  s.W = 0;
  s.n_idx = s.perm_stride = g.S;
  const size_t seg_rows = (size_t)g.U * g.S;
  bf16* gK = const_cast<bf16*>(static_cast<const bf16*>(b.grownK)) + (size_t)gi * seg_rows * WI_D;
  bf16* gV = const_cast<bf16*>(static_cast<const bf16*>(b.grownV)) + (size_t)gi * seg_rows * WI_D;
  const int amax = g.max_append > 0 ? g.max_append : 1;
  cudaError_t e;
  k_gather_segment<<<(unsigned)((seg_rows + 7) / 8), 256, 0, st>>>(
      static_cast<const bf16*>(b.K), static_cast<const bf16*>(b.V), static_cast<const bf16*>(b.appK),
      static_cast<const bf16*>(b.appV), const_cast<bf16*>(static_cast<const bf16*>(b.grownK)),
      const_cast<bf16*>(static_cast<const bf16*>(b.grownV)), g.U, g.n, g.W, g.S, gi, amax);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // B1-B4 on the segment (the build's kernels and rounds), B5 in place in the grown buffer
  if ((e = wi_launch_init_centroids(s, gK, w.chat, st)) != cudaSuccess) return e;
  for (int t = 0; t < g.iters; ++t) {
    if ((e = wi_launch_assign(s, gK, w.chat, w.assign, err, st)) != cudaSuccess) return e;
    if ((e = wi_launch_segment_sort(s, w.assign, w.seg_counts, w.seg_offsets, w.slots, err, st)) != cudaSuccess)
      return e;
    if (t + 1 < g.iters &&
        (e = wi_launch_centroid_update(s, gK, w.seg_counts, w.seg_offsets, w.slots, w.chat, st)) !=
            cudaSuccess)
      return e;
  }
  if ((e = wi_launch_reduce_permute(s, gK, gV, w.seg_counts, w.seg_offsets, w.slots, w.mu, w.valsum, w.cnt, w.off,
                                    w.perm, w.nonempty, w.tK, w.tV, g.U, st)) != cudaSuccess)
    return e;
  const long long warps = (long long)g.U * g.Cs;
  k_merge_segment<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(
      w.cnt, w.off, static_cast<const bf16*>(w.mu), w.valsum, w.perm, w.nonempty, cnt, off, static_cast<bf16*>(mu),
      valsum, static_cast<bf16*>(valsum16), perm, nonempty, g.U, g.C, g.Cb, g.Cs, g.S, g.n, g.W, g.n_idx,
      g.perm_stride, gi);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = wi_launch_set_int(b.grown, gi + 1, st)) != cudaSuccess) return e;
  return wi_launch_set_int(b.kcur, k_after, st);
}
