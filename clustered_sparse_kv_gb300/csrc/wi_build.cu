// wi_build.cu -- index build (prefill): segmented spherical k-means and the
// cluster-contiguous index.
//
// RetroInfer summaries de/fr/zh 2.A: segmented clustering cuts the context
// into segments that are clustered independently; fr 2.A.2 names spherical
// k-means; zh 2.A names the precomputed per-cluster value sum that the
// estimation zone reads.  Kernels here:
//   init_centroids   c_j = bf16(K_p / |K_p|), p = segment start + stride * j
//   assign (SIMT)    a_i = argmax_j K_i . c_j, ties to the lowest j
//   segment_sort     counting sort of a segment's tokens by (cluster, position)
//   centroid_update  c_j = bf16(u_j / |u_j|), u_j = sum of member K_i / |K_i|
//   reduce_gather    counts, row offsets, perm, mu_j = bf16(mean K), valsum_j,
//                    and the members' K / V rows gathered cluster by cluster
//   scatter_back     the gathered rows written back: K and V cluster-contiguous
//   gather_rows      the gather alone, by a given perm (an imported index)
#include <cuda_runtime.h>

#include <algorithm>

#include "wi_common.cuh"
#include "wi_internal.h"
#include "wi_pipe.cuh"

namespace {

__device__ __forceinline__ bool is_steady(long long p, long long n, int n_sink, int W) {
  return p < n_sink || p >= n - W;
}

// Row of the first slot of segment s: n_sink + clustered positions before s.
__device__ __forceinline__ long long seg_slot_base(int s, int S, long long n, int n_sink, int W) {
  const long long a = (long long)s * S;
  const long long steady_before = (a < n_sink ? a : n_sink) + (a > n - W ? a - (n - W) : 0);
  return n_sink + a - steady_before;
}

// Four values per thread (n is a multiple of 128).
__global__ void k_to_bf16(const float4* __restrict__ in, uint2* __restrict__ out, long long n4) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 x = in[i];
  const __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y), hi = __floats2bfloat162_rn(x.z, x.w);
  out[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

__global__ void k_init_centroids(const bf16* __restrict__ K, bf16* __restrict__ chat, int total, int nseg, int S,
                                 int Cs, long long n) {
  const int lane = threadIdx.x & 31;
  const int gid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gid >= total) return;
  const int u = gid / (nseg * Cs), s = (gid / Cs) % nseg, j = gid % Cs;
  const long long row = (long long)u * n + (long long)s * S + (long long)j * (S / Cs);
  float x[4];
  load_bf16x4(K + row * WI_D + 4 * lane, x);
  const float nrm = sqrtf(warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]));
  bf16* o = chat + (size_t)gid * WI_D + 4 * lane;
#pragma unroll
  for (int e = 0; e < 4; ++e) o[e] = __float2bfloat16_rn(nrm > 0.f ? x[e] / nrm : 0.f);
}

// SIMT assignment: a CTA scores 32 tokens of one segment against all of the
// segment's centroids (fp32 FMA over e = 0..127 in order), then takes the
// row argmax.  Shared memory: centroids as 32-bit words in rows padded to 65
// words (conflict-free per-thread row reads), tokens fp32 [32][128], scores
// fp32 [32][Cs].
constexpr int kAsgTok = 32;
constexpr int kAsgRowWords = WI_D / 2 + 1;

__global__ void __launch_bounds__(256) k_assign_simt(const bf16* __restrict__ K, const bf16* __restrict__ chat,
                                                     int32_t* __restrict__ assign, int S, int Cs, int nseg,
                                                     long long n, int n_sink, int W, int* err) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint32_t* cw = reinterpret_cast<uint32_t*>(smem_raw);                  // [Cs][65]
  float* tok = reinterpret_cast<float*>(cw + (size_t)Cs * kAsgRowWords);  // [32][128]
  float* sc = tok + kAsgTok * WI_D;                                       // [32][Cs]
  const int u = blockIdx.z, s = blockIdx.y, tile = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t* cg = reinterpret_cast<const uint32_t*>(chat + ((size_t)u * nseg + s) * Cs * WI_D);
  for (int i = tid; i < Cs * (WI_D / 2); i += blockDim.x) {
    const int j = i / (WI_D / 2), w = i % (WI_D / 2);
    cw[j * kAsgRowWords + w] = __ldg(cg + i);
  }
  const long long p0 = (long long)s * S + (long long)tile * kAsgTok;
  const bf16* kt = K + ((long long)u * n + p0) * WI_D;
  for (int i = tid; i < kAsgTok * WI_D; i += blockDim.x) tok[i] = __bfloat162float(kt[i]);
  __syncthreads();
  for (int j = tid; j < Cs; j += blockDim.x) {
    float acc[kAsgTok];
#pragma unroll
    for (int i = 0; i < kAsgTok; ++i) acc[i] = 0.f;
    const uint32_t* row = cw + j * kAsgRowWords;
    for (int w = 0; w < WI_D / 2; ++w) {
      const uint32_t cv = row[w];
      const float c0 = bf16_lo(cv), c1 = bf16_hi(cv);
#pragma unroll
      for (int i = 0; i < kAsgTok; ++i) {
        const float2 t = *reinterpret_cast<const float2*>(tok + i * WI_D + 2 * w);
        acc[i] = fmaf(t.x, c0, acc[i]);
        acc[i] = fmaf(t.y, c1, acc[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < kAsgTok; ++i) sc[i * Cs + j] = acc[i];
  }
  __syncthreads();
  for (int i = warp; i < kAsgTok; i += (blockDim.x >> 5)) {
    float best = -INFINITY;
    int bj = 0x7fffffff;
    for (int j = lane; j < Cs; j += 32) {
      const float v = sc[i * Cs + j];
      if (v > best) { best = v; bj = j; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
      if (ov > best || (ov == best && oj < bj)) { best = ov; bj = oj; }
    }
    if (lane == 0) {
      const long long p = p0 + i;
      int a = -1;
      if (!is_steady(p, n, n_sink, W)) {
        if (bj < 0 || bj >= Cs) { atomicOr(err, WI_DEVERR_BAD_CLUSTER); bj = 0; }
        a = s * Cs + bj;
      }
      assign[(long long)u * n + p] = a;
    }
  }
}

// Counting sort of one segment's clustered tokens by (cluster, position),
// stable and in O(S): each of the W warps takes a contiguous chunk of the
// segment's positions; pass 1 counts per (warp, cluster) (match_any groups the
// lanes of one cluster, whose leader adds the group's size); a scan turns the
// counts into each warp's first slot per cluster (clusters in order, warps in
// position order inside a cluster); pass 2 walks every chunk again in position
// order and gives each lane its slot = that start + its rank among the lanes
// of its cluster.  Outputs per segment-unit: counts [Cs], offsets [Cs+1]
// (local slots), slots [S] (position relative to the segment start, in slot
// order).  W = 32 when the segment-units fit in one wave (shorter chunks: the
// sort's few CTAs are latency-bound), else 16 (more CTAs resident per SM).
template <int kSortWarps>
__global__ void __launch_bounds__(32 * kSortWarps) k_segment_sort(const int32_t* __restrict__ assign,
                                                                  int* __restrict__ seg_counts,
                                                                  int* __restrict__ seg_offsets,
                                                                  int* __restrict__ slots, int S, int Cs, int nseg,
                                                                  long long n, int* err) {
  extern __shared__ __align__(16) int ss_raw[];
  int* wc = ss_raw;                   // [kSortWarps][Cs] counts, then first slots
  int* cnt = wc + kSortWarps * Cs;    // [Cs]
  int* off = cnt + Cs;                // [Cs + 1]
  int* tmp = off + Cs + 1;            // [32]
  int* sb = tmp + 32;                 // [S] sorted positions
  const int su = blockIdx.x, u = su / nseg, s = su % nseg;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t* a = assign + (long long)u * n + (long long)s * S;
  const int chunk = (S + kSortWarps - 1) / kSortWarps;
  const int p0 = warp * chunk, p1 = min(S, p0 + chunk);
  for (int i = tid; i < kSortWarps * Cs; i += blockDim.x) wc[i] = 0;
  __syncthreads();
  int* my = wc + warp * Cs;
  const unsigned below = (1u << lane) - 1u;
  // local cluster of position i, -1 for steady / outside the chunk
  auto local = [&](int i) -> int {
    if (i >= p1) return -1;
    const int c = __ldg(a + i);
    if (c < 0) return -1;
    const int cl = c - s * Cs;
    if (cl < 0 || cl >= Cs) {
      atomicOr(err, WI_DEVERR_BAD_CLUSTER);
      return -1;
    }
    return cl;
  };
  for (int i0 = p0; i0 < p1; i0 += 32) {
    const int cl = local(i0 + lane);
    const unsigned peers = __match_any_sync(0xffffffffu, cl);
    if (cl >= 0 && (peers & below) == 0u) my[cl] += __popc(peers);
  }
  __syncthreads();
  // counts per cluster, offsets, and every warp's first slot per cluster
  int running = 0;
  for (int base = 0; base < Cs; base += blockDim.x) {
    const int j = base + tid;
    int v = 0;
    if (j < Cs)
      for (int w = 0; w < kSortWarps; ++w) v += wc[w * Cs + j];
    int tot;
    const int ex = block_exclusive_scan(v, tmp, &tot);
    if (j < Cs) {
      cnt[j] = v;
      off[j] = running + ex;
      int r = running + ex;
      for (int w = 0; w < kSortWarps; ++w) {
        const int c = wc[w * Cs + j];
        wc[w * Cs + j] = r;
        r += c;
      }
    }
    running += tot;
  }
  if (tid == 0) off[Cs] = running;
  __syncthreads();
  for (int i0 = p0; i0 < p1; i0 += 32) {
    const int cl = local(i0 + lane);
    const unsigned peers = __match_any_sync(0xffffffffu, cl);
    const int first = cl >= 0 ? my[cl] : 0;
    if (cl >= 0) sb[first + __popc(peers & below)] = i0 + lane;
    __syncwarp();
    if (cl >= 0 && (peers & below) == 0u) my[cl] = first + __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  const int total = off[Cs];
  for (int i = tid; i < total; i += blockDim.x) slots[(long long)su * S + i] = sb[i];
  for (int j = tid; j < Cs; j += blockDim.x) seg_counts[(long long)su * Cs + j] = cnt[j];
  for (int j = tid; j <= Cs; j += blockDim.x) seg_offsets[(long long)su * (Cs + 1) + j] = off[j];
}

// One warp per cluster: c_j = bf16(u_j / |u_j|), u_j = sum over members (in
// position order) of K_i * (1/|K_i|), the norm taken in fp32 from the row
// itself.  Eight member rows in flight per warp.  Empty clusters keep c_j.
// The kernel waits on its dependent slot-then-row loads, so resident warps
// set its speed: 40 registers let six blocks (48 warps) share an SM.
constexpr int kUpdRows = 8;
__global__ void __launch_bounds__(256, 6) k_centroid_update(const bf16* __restrict__ K, const int* __restrict__ seg_counts,
                                                         const int* __restrict__ seg_offsets,
                                                         const int* __restrict__ slots, bf16* __restrict__ chat,
                                                         int total, int S, int Cs, int nseg, long long n) {
  const int lane = threadIdx.x & 31;
  const int gid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gid >= total) return;
  const int su = gid / Cs, cl = gid % Cs, u = su / nseg, s = su % nseg;
  const int m = seg_counts[gid];
  if (m == 0) return;
  const int b = seg_offsets[(long long)su * (Cs + 1) + cl];
  const int* sl = slots + (long long)su * S + b;
  const bf16* Kb = K + ((long long)u * n + (long long)s * S) * WI_D + 4 * lane;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int t0 = 0; t0 < m; t0 += kUpdRows) {
    uint2 w[kUpdRows];
#pragma unroll
    for (int i = 0; i < kUpdRows; ++i)
      w[i] = t0 + i < m ? ldg_u2(Kb + (long long)sl[t0 + i] * WI_D) : make_uint2(0u, 0u);
    // the eight rows' squared norms in one warp transpose-reduction (lanes 4i..4i+3 end with row i's);
    // the rows stay packed across it and are unpacked again for the sums (a few integer operations),
    // so the unpacked values never hold 32 registers and more warps fit on an SM
    float ss[kUpdRows];
#pragma unroll
    for (int i = 0; i < kUpdRows; ++i) {
      float x[4];
      unpack_bf16x4(w[i], x);
      ss[i] = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
    }
    const float sq = transpose_reduce<kUpdRows>(ss);
    const float ivl = sq > 0.f ? 1.0f / sqrtf(sq) : 0.f;
#pragma unroll
    for (int i = 0; i < kUpdRows; ++i) {
      const float iv = __shfl_sync(0xffffffffu, ivl, 4 * i);
      if (t0 + i < m) {  // warp-uniform
        uint32_t lo = w[i].x, hi = w[i].y;
        asm volatile("" : "+r"(lo), "+r"(hi));  // a fresh unpack: the first one is not kept alive
        const float x[4] = {bf16_lo(lo), bf16_hi(lo), bf16_lo(hi), bf16_hi(hi)};
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = fmaf(x[e], iv, acc[e]);
      }
    }
  }
  const float nrm = sqrtf(warp_sum(acc[0] * acc[0] + acc[1] * acc[1] + acc[2] * acc[2] + acc[3] * acc[3]));
  bf16* o = chat + (size_t)gid * WI_D + 4 * lane;
#pragma unroll
  for (int e = 0; e < 4; ++e) o[e] = __float2bfloat16_rn(nrm > 0.f ? acc[e] / nrm : 0.f);
}

// One warp per cluster of the final assignment, for the units [u0, u0 + nu):
// count, row offset, perm, mu = bf16(sum K / count), valsum = sum V (fp32),
// summed in position order, and the member rows copied in that order to the
// cluster's slots in the scratch rows tK / tV of the batch (the gather half
// of the in-place permutation).  The C clusters of each unit land in arrays
// of row stride Cst (offsets Cst + 1), perm in rows of pst slots.
__global__ void __launch_bounds__(256) k_reduce_gather(
    const bf16* __restrict__ K, const bf16* __restrict__ V, const int* __restrict__ seg_counts,
    const int* __restrict__ seg_offsets, const int* __restrict__ slots, bf16* __restrict__ mu,
    float* __restrict__ valsum, int* __restrict__ cnt, int* __restrict__ off, int* __restrict__ perm,
    int* __restrict__ nonempty, bf16* __restrict__ tK, bf16* __restrict__ tV, int u0, int nu, int C, int Cst, int S,
    int Cs, int nseg, long long n, int n_sink, int W, int pst, int n_idx) {
  const int lane = threadIdx.x & 31;
  const long long gid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gid >= (long long)nu * C) return;
  const int ub = (int)(gid / C), u = u0 + ub, c = (int)(gid % C), s = c / Cs, cl = c % Cs;
  const long long dst = (long long)u * Cst + c;
  const long long su = (long long)u * nseg + s;
  const int m = seg_counts[su * Cs + cl];
  const int b = seg_offsets[su * (Cs + 1) + cl];
  const long long slot0 = seg_slot_base(s, S, n, n_sink, W) + b;
  if (lane == 0) {
    off[(long long)u * (Cst + 1) + c] = (int)slot0;
    if (c == C - 1) off[(long long)u * (Cst + 1) + C] = (int)(n - W);
    cnt[dst] = m;
    if (m > 0) atomicAdd(&nonempty[u], 1);
  }
  const int* sl = slots + su * S + b;
  for (int t = lane; t < m; t += 32) perm[(long long)u * pst + (slot0 - n_sink) + t] = s * S + sl[t];
  const long long rowbase = (long long)u * n + (long long)s * S;
  const long long trow = (long long)ub * n_idx + (slot0 - n_sink);  // the cluster's first scratch row
  float ak[4] = {0.f, 0.f, 0.f, 0.f}, av[4] = {0.f, 0.f, 0.f, 0.f};
  constexpr int R = 8;
  for (int t0 = 0; t0 < m; t0 += R) {
    uint2 wk[R], wv[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const long long r = rowbase + (t0 + i < m ? sl[t0 + i] : 0);
      wk[i] = t0 + i < m ? ldg_u2(K + r * WI_D + 4 * lane) : make_uint2(0u, 0u);
      wv[i] = t0 + i < m ? ldg_u2(V + r * WI_D + 4 * lane) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
      if (t0 + i < m) {  // warp-uniform
        reinterpret_cast<uint2*>(tK + (trow + t0 + i) * WI_D)[lane] = wk[i];
        reinterpret_cast<uint2*>(tV + (trow + t0 + i) * WI_D)[lane] = wv[i];
        float xk[4], xv[4];
        unpack_bf16x4(wk[i], xk);
        unpack_bf16x4(wv[i], xv);
#pragma unroll
        for (int e = 0; e < 4; ++e) { ak[e] += xk[e]; av[e] += xv[e]; }
      }
    }
  }
  bf16* mo = mu + dst * WI_D + 4 * lane;
  float4 vo;
  const float fm = (float)m;
#pragma unroll
  for (int e = 0; e < 4; ++e) mo[e] = __float2bfloat16_rn(m > 0 ? ak[e] / fm : 0.f);
  vo.x = av[0]; vo.y = av[1]; vo.z = av[2]; vo.w = av[3];
  *reinterpret_cast<float4*>(valsum + dst * WI_D + 4 * lane) = vo;
}

// Cluster-contiguous reorder, through a scratch copy of units [u0, u0+nu):
// tmp[r] = rows[perm[r]] for every clustered slot r, then copied back.
__global__ void k_gather_rows(const bf16* __restrict__ K, const bf16* __restrict__ V, const int* __restrict__ perm,
                              bf16* __restrict__ tK, bf16* __restrict__ tV, int u0, long long n, int n_idx, int pst) {
  const int lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int u = u0 + blockIdx.y;
  if (r >= n_idx) return;
  const long long src = (long long)u * n + perm[(long long)u * pst + r];
  const long long dst = (long long)blockIdx.y * n_idx + r;
  reinterpret_cast<uint2*>(tK + dst * WI_D)[lane] = ldg_u2(K + src * WI_D + 4 * lane);
  reinterpret_cast<uint2*>(tV + dst * WI_D)[lane] = ldg_u2(V + src * WI_D + 4 * lane);
}

__global__ void k_scatter_back(bf16* __restrict__ K, bf16* __restrict__ V, const bf16* __restrict__ tK,
                               const bf16* __restrict__ tV, int u0, long long n, int n_sink, int n_idx) {
  const long long words = (long long)n_idx * WI_D / 8;  // 16-byte words per unit
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= words) return;
  const int u = u0 + blockIdx.y;
  const uint4* sk = reinterpret_cast<const uint4*>(tK + (long long)blockIdx.y * n_idx * WI_D);
  const uint4* sv = reinterpret_cast<const uint4*>(tV + (long long)blockIdx.y * n_idx * WI_D);
  uint4* dk = reinterpret_cast<uint4*>(K + ((long long)u * n + n_sink) * WI_D);
  uint4* dv = reinterpret_cast<uint4*>(V + ((long long)u * n + n_sink) * WI_D);
  dk[i] = sk[i];
  dv[i] = sv[i];
}

}  // namespace

cudaError_t wi_launch_to_bf16(const float* in, void* out, long long n, cudaStream_t st) {
  const long long n4 = n / 4;
  if (n4 <= 0) return cudaSuccess;
  k_to_bf16<<<(unsigned)((n4 + 255) / 256), 256, 0, st>>>(reinterpret_cast<const float4*>(in),
                                                           static_cast<uint2*>(out), n4);
  return cudaGetLastError();
}

cudaError_t wi_launch_init_centroids(const WiGeom& g, const void* K, void* chat, cudaStream_t st) {
  const int total = g.U * g.nseg * g.Cs;
  k_init_centroids<<<(total + 7) / 8, 256, 0, st>>>(static_cast<const bf16*>(K), static_cast<bf16*>(chat), total,
                                                     g.nseg, g.S, g.Cs, g.n);
  return cudaGetLastError();
}

size_t wi_assign_smem_bytes(const WiGeom& g) {
  return (size_t)g.Cs * kAsgRowWords * 4 + (size_t)kAsgTok * WI_D * 4 + (size_t)kAsgTok * g.Cs * 4;
}

cudaError_t wi_launch_assign(const WiGeom& g, const void* K, const void* chat, int32_t* assign, int* err,
                             cudaStream_t st) {
  if (wi_assign_tc_supported(g)) return wi_launch_assign_tc(g, K, chat, assign, err, st);
  const size_t smem = wi_assign_smem_bytes(g);
  static int smem_set[kWiSmemDevices] = {};
  cudaError_t e = wi_ensure_smem(k_assign_simt, smem, smem_set);
  if (e != cudaSuccess) return e;
  dim3 grid(g.S / kAsgTok, g.nseg, g.U);
  k_assign_simt<<<grid, 256, smem, st>>>(static_cast<const bf16*>(K), static_cast<const bf16*>(chat), assign, g.S,
                                         g.Cs, g.nseg, g.n, g.n_sink, g.W, err);
  return cudaGetLastError();
}

cudaError_t wi_launch_segment_sort(const WiGeom& g, const int32_t* assign, int* seg_counts, int* seg_offsets,
                                   int* slots, int* err, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const bool one_wave = (long long)g.U * g.nseg <= sms;
  const int warps = one_wave ? 32 : 16;
  const size_t smem = sizeof(int) * ((size_t)(warps + 2) * g.Cs + 1 + 32 + (size_t)g.S);
  if (one_wave) {
    static int smem_set[kWiSmemDevices] = {};
    if ((e = wi_ensure_smem(k_segment_sort<32>, smem, smem_set)) != cudaSuccess) return e;
    k_segment_sort<32><<<g.U * g.nseg, 32 * 32, smem, st>>>(assign, seg_counts, seg_offsets, slots, g.S, g.Cs,
                                                            g.nseg, g.n, err);
  } else {
    static int smem_set[kWiSmemDevices] = {};
    if ((e = wi_ensure_smem(k_segment_sort<16>, smem, smem_set)) != cudaSuccess) return e;
    k_segment_sort<16><<<g.U * g.nseg, 32 * 16, smem, st>>>(assign, seg_counts, seg_offsets, slots, g.S, g.Cs,
                                                            g.nseg, g.n, err);
  }
  return cudaGetLastError();
}

cudaError_t wi_launch_centroid_update(const WiGeom& g, const void* K, const int* seg_counts, const int* seg_offsets,
                                      const int* slots, void* chat, cudaStream_t st) {
  const int total = g.U * g.nseg * g.Cs;
  k_centroid_update<<<(total + 7) / 8, 256, 0, st>>>(static_cast<const bf16*>(K), seg_counts, seg_offsets, slots,
                                                      static_cast<bf16*>(chat), total, g.S, g.Cs, g.nseg, g.n);
  return cudaGetLastError();
}

cudaError_t wi_launch_reduce_permute(const WiGeom& g, void* K, void* V, const int* seg_counts, const int* seg_offsets,
                                     const int* slots, void* mu, float* valsum, int* cnt, int* off, int* perm,
                                     int* nonempty, void* tmpK, void* tmpV, int batch_units, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(nonempty, 0, sizeof(int) * g.U, st);
  if (e != cudaSuccess) return e;
  if (batch_units < 1) return cudaErrorInvalidValue;
  for (int u0 = 0; u0 < g.U; u0 += batch_units) {
    const int nu = g.U - u0 < batch_units ? g.U - u0 : batch_units;
    const long long warps = (long long)nu * g.Cb;
    k_reduce_gather<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(
        static_cast<const bf16*>(K), static_cast<const bf16*>(V), seg_counts, seg_offsets, slots,
        static_cast<bf16*>(mu), valsum, cnt, off, perm, nonempty, static_cast<bf16*>(tmpK),
        static_cast<bf16*>(tmpV), u0, nu, g.Cb, g.C, g.S, g.Cs, g.nseg, g.n, g.n_sink, g.W, g.perm_stride, g.n_idx);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (g.n_idx == 0) continue;
    const long long words = (long long)g.n_idx * WI_D / 8;
    dim3 g2((unsigned)((words + 255) / 256), nu);
    k_scatter_back<<<g2, 256, 0, st>>>(static_cast<bf16*>(K), static_cast<bf16*>(V), static_cast<const bf16*>(tmpK),
                                       static_cast<const bf16*>(tmpV), u0, g.n, g.n_sink, g.n_idx);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t wi_launch_permute(const WiGeom& g, void* K, void* V, const int* perm, void* tmpK, void* tmpV, int u0,
                              int nu, cudaStream_t st) {
  if (g.n_idx == 0 || nu == 0) return cudaSuccess;
  dim3 g1((unsigned)((g.n_idx + 7) / 8), nu);
  k_gather_rows<<<g1, 256, 0, st>>>(static_cast<const bf16*>(K), static_cast<const bf16*>(V), perm,
                                    static_cast<bf16*>(tmpK), static_cast<bf16*>(tmpV), u0, g.n, g.n_idx,
                                    g.perm_stride);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long words = (long long)g.n_idx * WI_D / 8;
  dim3 g2((unsigned)((words + 255) / 256), nu);
  k_scatter_back<<<g2, 256, 0, st>>>(static_cast<bf16*>(K), static_cast<bf16*>(V), static_cast<const bf16*>(tmpK),
                                     static_cast<const bf16*>(tmpV), u0, g.n, g.n_sink, g.n_idx);
  return cudaGetLastError();
}
