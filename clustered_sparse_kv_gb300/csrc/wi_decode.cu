// wi_decode.cu -- one decode step of the wave index: tripartite attention.
//
// RetroInfer summaries de/fr/zh 2.A (tripartite attention approximation):
//   steady zone      sinks + local window (+ appended tokens), exact;
//   retrieval zone   the top-k clusters by q . mu_j, their tokens exact;
//   estimation zone  every other non-empty cluster j contributes
//                    n_j exp(q.mu_j/sqrt(d)) to the softmax denominator and
//                    exp(q.mu_j/sqrt(d)) * valsum_j to the numerator
//                    (a Jensen lower bound, zh 2.A);
//   the zones merge into one softmax by log-sum-exp.
// Three kernels per step, each over the whole batch, chained by programmatic
// dependent launch:
//   k_scores          s_hj = q_h . mu_j for every cluster on the tensor cores
//                     (tcgen05, TMA-fed), and each CTA's largest score key;
//   k_select_estimate one launch, two roles: per head, the top-k clusters
//                     (ties to the lowest id, ids ascending), their row runs and
//                     the row-balanced splits of the exact rows; per range of
//                     clusters, the estimation partial (m, Z, N) over ALL
//                     non-empty clusters (streamed value sums);
//   k_exact_merge     per head and row split: flash-decode over the steady rows
//                     and the retrieved clusters' contiguous rows (bulk copies
//                     into shared memory), plus the retrieved clusters' value-sum
//                     terms; the last CTA of a head merges estimate - retrieved
//                     terms + exact partials by LSE.
// Index variants are separate kernel instances (the default ones carry none of
// their code): value sums read as a bf16 copy (the estimation role and the
// exact kernel per value type), and group-shared retrieval (k_scores also keys
// the heads' summed score; one top-k per kv head, written out for each head).
#include <cuda_runtime.h>

#include "wi_common.cuh"
#include "wi_internal.h"
#include "wi_pipe.cuh"
#include "wi_tc.cuh"

namespace {

// ------------------------------------------------------ scores / estimate ----
// Both kernels split a unit's clusters evenly over P CTAs (boundaries on
// multiples of 16 clusters so every bulk copy stays 16-byte aligned) and
// stream them through shared memory in tiles of 128 clusters: one producer
// warp issues cp.async.bulk copies into an mbarrier ring, 16 consumer warps
// take 8 clusters each per tile.
constexpr int kSWarps = 16;
constexpr int kSTile = 8 * kSWarps;
constexpr int kSThreads = 32 * (kSWarps + 1);
constexpr int kTopkBins = 2048;  // histogram bins of the top-k passes

// G query heads per kv head, in blocks of 4 heads (HB blocks); GP = heads per
// block rounded up to a power of two; lane l of a warp handles cluster l >> 2
// and in-block head (l & 3) >> SHIFT.
template <int G>
struct HeadGeo {
  static constexpr int HB = G > 4 ? 2 : 1;
  static constexpr int GP = G > 2 ? 4 : (G > 1 ? 2 : 1);
  static constexpr int SHIFT = GP == 4 ? 0 : (GP == 2 ? 1 : 2);
};

// Inverse of float_key for finite scores.
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ void cluster_range(int C, int p, int P, int* c0, int* c1) {
  *c0 = (int)(((long long)C * p / P) & ~15LL);
  *c1 = p + 1 == P ? C : (int)(((long long)C * (p + 1) / P) & ~15LL);
}

// Never leave with copies in flight: wait for the last round of every used stage.
template <int STAGES>
__device__ void drain_stages(uint64_t* full, int issued, int* err) {
  for (int s = 0; s < STAGES && s < issued; ++s) {
    const int last = ((issued - 1 - s) / STAGES) * STAGES + s;
    mbar_wait(&full[s], (last / STAGES) & 1, err);
  }
}

// ---- k_scores: s_hj = q_h . mu_j for every cluster on the tensor cores.
// Per 128-cluster tile: TMA loads the mean keys (A, 128 x 128 bf16, K-major,
// 128-byte swizzle); one thread issues eight tcgen05.mma (M = 128 clusters,
// N = 16 heads (G used, the rest zero), K = 16) into one of four 16-column TMEM
// accumulators; four epilogue warps read one cluster row each per lane
// (tcgen05.ld 32x32b.x16) and store the G scores.  Warp 0: TMA producer;
// warp 1: TMEM allocation + MMA; warps 2..5 and 6..9: two epilogue groups
// that take alternate tiles (four accumulators, so both can be busy).
constexpr int kScTile = 128;
constexpr int kScEpiWarps = 8;  // two groups of 4 (one TMEM lane quarter each), alternate tiles
constexpr int kScAcc = 4;       // TMEM accumulators (16 columns each): tile it uses it % 4
constexpr int kScThreads = 32 * (2 + kScEpiWarps);
constexpr int kScATile = kScTile * WI_D * 2;  // 32 KB: two 16 KB halves of 64 columns
constexpr int kScN = 16;                        // MMA N: heads padded to 16
constexpr int kScQBytes = kScN * WI_D * 2;      // 4 KB, the B operand

template <int G>
struct ScCfg {
  static constexpr int STAGES = 6;
  static constexpr size_t A_OFF = kScQBytes;
  static constexpr size_t CNT_OFF = A_OFF + (size_t)STAGES * kScATile;
  static constexpr size_t WMAX_OFF = CNT_OFF + sizeof(int) * STAGES * kScTile;
  static constexpr size_t BAR_OFF = WMAX_OFF + sizeof(uint32_t) * kScEpiWarps * 9;
  static constexpr size_t SMEM = BAR_OFF + sizeof(uint64_t) * (2 * STAGES + 2 * kScAcc) + 16;
};

template <int G, bool GRP>
__global__ void __launch_bounds__(kScThreads, 1) k_scores(const __grid_constant__ CUtensorMap map_mu,
                                                         const bf16* __restrict__ q, const int* __restrict__ cnt,
                                                         uint32_t* __restrict__ keys, unsigned* __restrict__ kmaxp,
                                                         int C, int P, int* err) {
  constexpr int GK = G + (GRP ? 1 : 0);  // key rows per unit: the heads (+ their summed score)
  using CF = ScCfg<G>;
  constexpr int STAGES = CF::STAGES;
  extern __shared__ __align__(1024) unsigned char sc_raw[];
  unsigned char* qB = sc_raw;                                              // [k half][16 rows][128 B]
  unsigned char* A = sc_raw + CF::A_OFF;                                   // [stage][k half][128 rows][128 B]
  int* cnts = reinterpret_cast<int*>(sc_raw + CF::CNT_OFF);               // [stage][128]
  uint32_t* wmax = reinterpret_cast<uint32_t*>(sc_raw + CF::WMAX_OFF);    // [epilogue warp][GK]
  uint64_t* full = reinterpret_cast<uint64_t*>(sc_raw + CF::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + kScAcc;
  uint32_t* tbase = reinterpret_cast<uint32_t*>(tempty + kScAcc);
  int* s_abort = reinterpret_cast<int*>(tbase + 1);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (smem_addr(sc_raw) & 1023u) {  // the swizzled tiles need 1024-byte alignment; never run misaligned
    if (tid == 0) atomicOr(err, WI_DEVERR_BAD_ROW);
    return;
  }
  const int u = blockIdx.y, p = blockIdx.x;
  int c0, c1;
  cluster_range(C, p, P, &c0, &c1);
  const int ntile = (c1 - c0 + kScTile - 1) / kScTile;
  pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1 + kScEpiWarps / 2);  // the MMA commit and the 4 warps of the tile's group
    }
    for (int b = 0; b < kScAcc; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kScEpiWarps / 2);
    }
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tbase)),
                 "n"(kScAcc * kScN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tbase;
  // the index (written only by build / import) streams before the dependency wait
  auto issue = [&](int it) {
    const int s = it % STAGES;
    const int j0 = c0 + it * kScTile, nj = min(kScTile, c1 - j0);
    mbar_arrive_expect_tx(&full[s], (uint32_t)(kScATile + nj * 4));
    tma_load_2d(A + (size_t)s * kScATile, &map_mu, 0, u * C + j0, &full[s]);
    tma_load_2d(A + (size_t)s * kScATile + kScATile / 2, &map_mu, 64, u * C + j0, &full[s]);
    bulk_g2s(cnts + s * kScTile, cnt + (size_t)u * C + j0, nj * 4, &full[s]);
  };
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_mu)) : "memory");
    for (int it = 0; it < ntile && it < STAGES; ++it) issue(it);
  }
  // the queries may come from the previous kernel: B operand = q of the G heads, rows >= G zero,
  // written in the 128-byte-swizzled K-major layout (row n, 16-byte chunk c at chunk c ^ (n & 7))
  pdl_wait();
  for (int i = tid; i < kScN * 16; i += kScThreads) {
    const int n = i >> 4, c = i & 15;  // head row, 16-byte chunk over the 256-byte row
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < G) v = *reinterpret_cast<const uint4*>(q + ((size_t)u * G + n) * WI_D + 8 * c);
    const int half = c >> 3, cc = c & 7;
    *reinterpret_cast<uint4*>(qB + half * (kScN * 128) + (n >> 3) * 1024 + (n & 7) * 128 + ((cc ^ (n & 7)) << 4)) = v;
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (warp == 0) {
    if (lane == 0) {
      int issued = min(ntile, STAGES);
      for (int it = STAGES; it < ntile; ++it) {
        const int s = it % STAGES, r = it / STAGES;
        if (!mbar_wait(&empty[s], (r - 1) & 1, err)) { *s_abort = 1; break; }
        issue(it);
        issued = it + 1;
      }
      if (*s_abort) drain_stages<STAGES>(full, issued, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = make_idesc(kScTile, kScN);
      const uint32_t q0 = smem_addr(qB);
      for (int it = 0; it < ntile; ++it) {
        const int s = it % STAGES, r = it / STAGES, b = it % kScAcc;
        if (!mbar_wait(&full[s], r & 1, err)) { *s_abort = 1; break; }
        if (it >= kScAcc && !mbar_wait(&tempty[b], (it / kScAcc - 1) & 1, err)) { *s_abort = 1; break; }
        tc_fence_after();
        const uint32_t a0 = smem_addr(A + (size_t)s * kScATile);
#pragma unroll
        for (int kk = 0; kk < WI_D / 16; ++kk) {
          const uint32_t ko = (uint32_t)(kk >> 2), kb = (uint32_t)(kk & 3) * 32;
          mma_bf16(tmem + (uint32_t)(b * kScN), make_desc_sw128(a0 + ko * (kScATile / 2) + kb),
                   make_desc_sw128(q0 + ko * (kScN * 128) + kb), idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(&tfull[b]);
        mma_commit(&empty[s]);
      }
    }
  } else {
    // epilogue: group grp = (warp - 2) / 4 takes the tiles it = grp (mod 2); warp w reads TMEM
    // lanes 32*(w%4).., i.e. clusters quarter*32 + lane of the tile; it also keeps the largest
    // key of the non-empty clusters per head (for the top-k)
    const int quarter = warp & 3, grp = (warp - 2) >> 2;
    bool ok = true;
    uint32_t kmx[G];
#pragma unroll
    for (int h = 0; h < G; ++h) kmx[h] = 0u;
    uint32_t kmxs = 0u;  // of the summed-score keys (group-shared retrieval)
    for (int it = grp; it < ntile; it += 2) {
      const int s = it % STAGES, r = it / STAGES, b = it % kScAcc;
      const int j0 = c0 + it * kScTile, nj = min(kScTile, c1 - j0);
      const int row = quarter * 32 + lane;
      uint32_t rr[16];
      if (ok) {
        if (!mbar_wait(&tfull[b], (it / kScAcc) & 1, err) || !mbar_wait(&full[s], r & 1, err)) {
          ok = false;
          *s_abort = 1;
        }
      }
      if (ok) {
        tc_fence_after();
        tmem_ld16_nowait(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * kScN), rr);
        tmem_wait_ld();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[b]);
      const int cn = (ok && row < nj) ? cnts[s * kScTile + row] : 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      const bool valid = ok && row < nj;
      if (valid) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const uint32_t key = cn > 0 ? float_key(__uint_as_float(rr[h])) : 0u;
          keys[((size_t)u * GK + h) * C + j0 + row] = key;
          kmx[h] = max(kmx[h], key);
        }
        if constexpr (GRP) {  // group-shared retrieval: row G holds the key of the heads' summed score
          float sum = 0.f;
#pragma unroll
          for (int h = 0; h < G; ++h) sum += __uint_as_float(rr[h]);
          const uint32_t key = cn > 0 ? float_key(sum) : 0u;
          keys[((size_t)u * GK + G) * C + j0 + row] = key;
          kmxs = max(kmxs, key);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < GK; ++h) {
      uint32_t m = h < G ? kmx[h < G ? h : 0] : kmxs;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) wmax[(warp - 2) * GK + h] = m;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (tid < GK) {  // this CTA's largest key per row: plain stores, the top-k takes the max over CTAs
    uint32_t m = 0u;
#pragma unroll
    for (int w8 = 0; w8 < kScEpiWarps; ++w8) m = max(m, wmax[w8 * GK + tid]);
    kmaxp[((size_t)u * P + p) * GK + tid] = m;
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kScAcc * kScN) : "memory");
  }
}

// ---- k_select_estimate: one launch, two kinds of CTA (kSThreads threads each).
//   blocks [0, U*G)           top-k of one head (role "select");
//   blocks [U*G, U*G + U*PE)  estimation over a range of one unit's clusters
//                             (role "estimate").
// The estimation only has to be ready for the final merge, so it shares the
// launch with the top-k instead of following it.

// -- estimate role: estimation partial over ALL non-empty clusters of the CTA's
// range, per head: m = max lam s_hj, Z = sum n_j e^{lam s - m},
// N = sum e^{lam s - m} valsum_j (online softmax per warp, merged per CTA).
constexpr int kEsStages = 3;
template <typename VT>  // value sums: float, or their bf16 copy
struct EsStage {
  VT vs[kSTile * WI_D];
  int cnt[kSTile];
  uint32_t sc[8][kSTile];  // score keys of up to 8 heads (0: empty cluster)
};
template <typename VT>
constexpr size_t es_smem() {
  return sizeof(EsStage<VT>) * kEsStages + 2 * kEsStages * sizeof(uint64_t) + sizeof(float) * kSWarps * 2 * 32 +
         sizeof(float) * kSWarps * 2 * 4 + 16;
}

template <int G, typename VT, int GK>
__device__ void estimate_role(unsigned char* raw, const VT* __restrict__ valsum, const int* __restrict__ cnt,
                              const uint32_t* __restrict__ scores, float* __restrict__ part, int C, int u, int p,
                              int P, float lam, int depth, int* err) {
  using HG = HeadGeo<G>;
  EsStage<VT>* st = reinterpret_cast<EsStage<VT>*>(raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(raw + sizeof(EsStage<VT>) * kEsStages);
  uint64_t* empty = full + kEsStages;
  float* pbuf = reinterpret_cast<float*>(empty + kEsStages);  // [warps][2][32]
  float* sbuf = pbuf + kSWarps * 2 * 32;                       // [warps][2][4]
  int* s_abort = reinterpret_cast<int*>(sbuf + kSWarps * 2 * 4);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int c0, c1;
  cluster_range(C, p, P, &c0, &c1);
  const int ntile = (c1 - c0 + kSTile - 1) / kSTile;
  if (tid == 0) {
    for (int s = 0; s < kEsStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSWarps);
    }
    *s_abort = 0;
  }
  __syncthreads();
  float m_l[HG::HB], z_l[HG::HB], N[G][4];
#pragma unroll
  for (int b = 0; b < HG::HB; ++b) { m_l[b] = -INFINITY; z_l[b] = 0.f; }
#pragma unroll
  for (int h = 0; h < G; ++h) N[h][0] = N[h][1] = N[h][2] = N[h][3] = 0.f;
  const int ci = lane >> 2;
  const int hl = (lane & 3) >> HG::SHIFT;
  const bool rep = (lane & ((1 << HG::SHIFT) - 1)) == 0;
  if (warp == kSWarps) {
    if (lane == 0) {
      // the value sums and counts (index data) of the first stages stream before the dependency
      // wait; the scores come from the previous kernel
      auto issue_index = [&](int it) {
        const int s = it % kEsStages;
        const int j0 = c0 + it * kSTile, nj = min(kSTile, c1 - j0);
        mbar_arrive_expect_tx(&full[s], (uint32_t)nj * (WI_D * (uint32_t)sizeof(VT) + 4 + 4 * G));
        const size_t row = (size_t)u * C + j0;
        bulk_g2s(st[s].vs, valsum + row * WI_D, nj * WI_D * (uint32_t)sizeof(VT), &full[s]);
        bulk_g2s(st[s].cnt, cnt + row, nj * 4, &full[s]);
      };
      auto issue_scores = [&](int it) {
        const int s = it % kEsStages;
        const int j0 = c0 + it * kSTile, nj = min(kSTile, c1 - j0);
        for (int h = 0; h < G; ++h) bulk_g2s(st[s].sc[h], scores + ((size_t)u * GK + h) * C + j0, nj * 4, &full[s]);
      };
      // at most `depth` tiles in flight (the ring has kEsStages slots): tile it is issued once tile
      // it - depth has been consumed
      depth = depth == 2 ? 2 : kEsStages;
      const int pre = min(ntile, depth);
      for (int it = 0; it < pre; ++it) issue_index(it);
      pdl_wait();
      for (int it = 0; it < pre; ++it) issue_scores(it);
      int issued = pre;
      for (int it = pre; it < ntile; ++it) {
        const int s = it % kEsStages, r = it / kEsStages;
        if (depth < kEsStages) {
          const int od = it - depth;  // phase (od / kEsStages) of its slot completes when it is consumed
          if (!mbar_wait(&empty[od % kEsStages], (od / kEsStages) & 1, err)) { *s_abort = 1; break; }
        }
        if (!mbar_wait(&empty[s], (r - 1) & 1, err)) { *s_abort = 1; break; }
        issue_index(it);
        issue_scores(it);
        issued = it + 1;
      }
      if (*s_abort) drain_stages<kEsStages>(full, issued, err);
    } else {
      pdl_wait();
    }
  } else {
    pdl_wait();
    float* pb = pbuf + warp * 2 * 32;
    float* sb = sbuf + warp * 2 * 4;
    for (int it = 0; it < ntile; ++it) {
      const int s = it % kEsStages, r = it / kEsStages;
      if (!mbar_wait(&full[s], r & 1, err)) { *s_abort = 1; break; }
      const EsStage<VT>& T = st[s];
      const int j0 = c0 + it * kSTile, nj = min(kSTile, c1 - j0);
      const int i0 = warp * 8;
      if (i0 < nj) {
        const bool valid_c = (i0 + ci) < nj;
        const int cn = valid_c ? T.cnt[i0 + ci] : 0;
#pragma unroll
        for (int b = 0; b < HG::HB; ++b) {
          const int head = b * 4 + hl;
          const bool valid = valid_c && head < G;
          const uint32_t key = T.sc[head < G ? head : 0][i0 + ci];
          const float se = (valid && cn > 0 && key != 0u) ? lam * key_float(key) : -INFINITY;
          float mx = fmaxf(se, __shfl_xor_sync(0xffffffffu, se, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float m_new = fmaxf(m_l[b], mx);
          const float sc = m_new == -INFINITY ? 1.f : __expf(m_l[b] - m_new);
          const float pr = (se == -INFINITY || !rep) ? 0.f : __expf(se - m_new);
          float zc = (float)cn * pr;
          zc += __shfl_xor_sync(0xffffffffu, zc, 4);
          zc += __shfl_xor_sync(0xffffffffu, zc, 8);
          zc += __shfl_xor_sync(0xffffffffu, zc, 16);
          z_l[b] = z_l[b] * sc + zc;
          m_l[b] = m_new;
          pb[b * 32 + lane] = pr;
          if (ci == 0 && rep) sb[b * 4 + hl] = sc;
        }
        __syncwarp();
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float sc = sb[(h >> 2) * 4 + (h & 3)];
          const float2 s2 = make_float2(sc, sc);
          const float2 lo = __fmul2_rn(make_float2(N[h][0], N[h][1]), s2);
          const float2 hi = __fmul2_rn(make_float2(N[h][2], N[h][3]), s2);
          N[h][0] = lo.x; N[h][1] = lo.y; N[h][2] = hi.x; N[h][3] = hi.y;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (i0 + i >= nj) break;  // rows past the tile hold stale shared memory
          float4 vv;
          if constexpr (sizeof(VT) == 4) {
            vv = *reinterpret_cast<const float4*>(&T.vs[(i0 + i) * WI_D + 4 * lane]);
          } else {
            float x[4];
            unpack_bf16x4(*reinterpret_cast<const uint2*>(&T.vs[(i0 + i) * WI_D + 4 * lane]), x);
            vv = make_float4(x[0], x[1], x[2], x[3]);
          }
          const float2 vlo = make_float2(vv.x, vv.y), vhi = make_float2(vv.z, vv.w);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float pr = pb[(h >> 2) * 32 + ((i * HG::GP + (h & 3)) << HG::SHIFT)];
            const float2 p2 = make_float2(pr, pr);
            const float2 lo = __ffma2_rn(p2, vlo, make_float2(N[h][0], N[h][1]));
            const float2 hi = __ffma2_rn(p2, vhi, make_float2(N[h][2], N[h][3]));
            N[h][0] = lo.x; N[h][1] = lo.y; N[h][2] = hi.x; N[h][3] = hi.y;
          }
        }
        __syncwarp();
      }
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  __syncthreads();
  if (*s_abort) return;
  float* red = reinterpret_cast<float*>(raw);  // [warps][G][WI_PART]; the stages are free now
  if (warp < kSWarps) {
#pragma unroll
    for (int b = 0; b < HG::HB; ++b) {
      const int head = b * 4 + hl;
      if (ci == 0 && rep && head < G) {
        red[((size_t)warp * G + head) * WI_PART + 0] = m_l[b];
        red[((size_t)warp * G + head) * WI_PART + 1] = z_l[b];
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
      *reinterpret_cast<float4*>(&red[((size_t)warp * G + h) * WI_PART + 4 + 4 * lane]) =
          make_float4(N[h][0], N[h][1], N[h][2], N[h][3]);
  }
  __syncthreads();
  for (int i = tid; i < G * WI_D; i += kSThreads) {
    const int h = i / WI_D, d = i % WI_D;
    float M = -INFINITY;
    for (int w = 0; w < kSWarps; ++w) M = fmaxf(M, red[((size_t)w * G + h) * WI_PART]);
    float z = 0.f, acc = 0.f;
    if (M > -INFINITY) {
      for (int w = 0; w < kSWarps; ++w) {
        const float mw = red[((size_t)w * G + h) * WI_PART];
        if (mw == -INFINITY) continue;
        const float f = __expf(mw - M);
        z = fmaf(f, red[((size_t)w * G + h) * WI_PART + 1], z);
        acc = fmaf(f, red[((size_t)w * G + h) * WI_PART + 4 + d], acc);
      }
    }
    float* o = part + (((size_t)u * G + h) * P + p) * WI_PART;
    if (d == 0) { o[0] = M; o[1] = z; }
    o[4 + d] = acc;
  }
}

// -- select role: top-k of one head.  The k largest keys (order-preserving
// bits of the scores; 0 = empty cluster) are the k smallest distances
// d = key_max - key.  One pass counts d on a logarithmic scale (2048 bins: the
// position of d's leading one, then its next 6 bits; monotone in d), which
// finds the bin holding the k-th key; the few keys in that bin are ranked by
// (key descending, id ascending) to pin the k-th one exactly (a radix select
// over (d, id) takes over when the bin holds more keys than threads).  The
// selected clusters are then listed in id order (a ballot per 32 ids and a
// prefix over those counts), each with its row run and weight (first row,
// rows, e^{lam s_j - m_sub}, id), m_sub = lam * s_max, together with the
// starts of NS row-balanced splits of the selected rows and
// Z_sub = sum n_j e^{lam s_j - m_sub} over them; their value-sum terms are
// summed where their rows are loaded (exact attention), and both are
// subtracted from the estimate at the merge.
//
// Every pass over the clusters is a short rolled loop with the CTA's stride:
// the role runs once per CTA per step and its instructions mostly miss the
// instruction cache, so the code executed once is kept small (the rare paths
// are out of line).  The keys are cached in shared memory when C <= kSelKeysMax;
// above it (up to 65536 clusters) the first pass streams them from global
// memory with 16-byte loads and keeps each key's distance bin (16 bits) in
// shared memory, which the later passes read; only the threshold bin's keys
// and the selected keys are read again.
constexpr int kSelThreads = 512;  // ranking capacity: candidates in the threshold bin
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kBinsPerLane = kTopkBins / kSelThreads;  // 4
constexpr int kSelKeysMax = 32768;
constexpr int kSNW = kSThreads / 32;  // warps of the CTA


// Logarithmic bin of a distance: 64 * (position of the leading one) + the next
// six bits (d = 0 and 1 share bin 0).  Non-decreasing in d; within a bin of
// leading position m >= 6 only the low m - 6 bits of d vary.  Computed from
// d converted to float with rounding toward zero: its exponent is m + 127 and
// the top six bits of its mantissa are the six bits after the leading one, so
// bits 30..17 of the float are 64 (m + 127) + those bits (branch-free).
__device__ __forceinline__ int log_bin(uint32_t d) {
  return max((int)(__float_as_uint(__uint2float_rz(d)) >> 17) - 127 * 64, 0);
}

// Smallest d with log_bin(d) >= b (b in [0, 2047]): bin b > 0 starts at the
// float 2^m (1 + sub / 64) (bits (b + 127 * 64) << 17), rounded up to an
// integer; rounding toward zero maps d to a float >= that value exactly when
// d >= it, since the value has 7 significant bits.
__device__ __forceinline__ uint32_t log_bin_start(int b) {
  return b == 0 ? 0u : __float2uint_ru(__uint_as_float((uint32_t)(b + 127 * 64) << 17));
}

struct TopkArgs {
  const uint32_t* scores;  // [U][G][C] score keys (order-preserving bits; 0 = empty cluster)
  const int* cnt;
  const int* off;
  const int* nonempty;
  const void* valsum;  // [U][C][128] value sums: float, or bf16 (the select_estimate instance says which)
  int* sel;
  int* selcnt;
  float* subpart;
  int4* runs;    // [U][G][kmax]  (first row, rows, weight bits e^{lam s - m_sub}, cluster id)
  int4* splits;  // [U][G][NS+2]  (position, row inside that cluster, split's first selected row, 0)
  int4* sruns;   // [U][G][NS+1][32] runs of positions splits[b].x .. +31 (one read for the split's CTA)
  const int* app_count;
  const int* kcur;   // budget of the clusters held so far (grows with the index)
  const int* grown;  // segments grown during decode: their seg_len rows each left the local window
  float* part1;  // estimation partials [U][G][PE]
  const unsigned* kmaxp;  // [U][P1][G] largest key over the non-empty clusters of each k_scores CTA
  int* err;
  int U, G, C, kmax, NS, PE, n_sink, W, P1, seg_len;
  int est_first;  // the estimation CTAs take the first block indices (they start before the top-k CTAs)
  int es_depth;   // estimation stages in flight per CTA (2 or kEsStages)
  float lam;
};

struct alignas(16) SelSmem {
  int hist[2][kTopkBins];
  int s_wsum[32];
  int s_bin, s_above, s_ncand, s_app;  // s_app, s_grown: the steady-row counters, fetched early
  int s_grown, s_pad[3];
  uint64_t s_bar, s_pad2;  // completion of the keys' bulk copy (cached keys)
  int s_spos[68];  // first position of each split
  int s_wt[32];
  float s_wf[32];
  uint32_t ckey[kSelThreads];
  int cid[kSelThreads];
};

static_assert(sizeof(SelSmem) % 16 == 0, "the cached keys follow SelSmem 16-byte aligned");
// Shared memory of the select role beyond SelSmem (a multiple of 16 bytes):
// the keys (16-byte aligned, when cached), then per 32-id chunk the take bits,
// then per selected position its id, rows, first row in the index and first
// row among the selected rows.
__host__ __device__ inline size_t sel_base_bytes(int C, int kmax) {
  return sizeof(SelSmem) + ((size_t)C + 31) / 32 * 4 + (size_t)kmax * 16;
}
// Row counts and first rows of the selected clusters land, while the top-k runs, in per-cluster
// slots next to the keys (asynchronous 4-byte copies) when that fits.
__host__ __device__ inline bool sel_rows_async(int C, int kmax) {
  return C <= kSelKeysMax && sel_base_bytes(C, kmax) + (size_t)C * 12 <= 200 * 1024;
}
// Above kSelKeysMax the keys do not fit: each key's logarithmic distance bin (16 bits) is kept instead.
__host__ __device__ inline size_t sel_keys_bytes(int C, int kmax) {
  return C <= kSelKeysMax ? (size_t)C * (sel_rows_async(C, kmax) ? 12 : 4) : ((size_t)C * 2 + 15) / 16 * 16;
}
__host__ __device__ inline size_t sel_smem_bytes(int C, int kmax) {
  return sel_base_bytes(C, kmax) + sel_keys_bytes(C, kmax);
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// Block-wide search over 2048 ascending bins (thread t < 512 owns bins 4t..4t+3):
// the bin where the running count first reaches `target` and the count below
// it.  Block-uniform result; false if the counts never reach `target`.
__device__ __forceinline__ bool find_bin(const int* hist, int target, SelSmem& sm, int* bin, int* above) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int c[kBinsPerLane] = {0, 0, 0, 0};
  if (warp < kSelWarps) {
    const int4 h4 = *reinterpret_cast<const int4*>(hist + kBinsPerLane * tid);
    c[0] = h4.x; c[1] = h4.y; c[2] = h4.z; c[3] = h4.w;
  }
  const int lsum = c[0] + c[1] + c[2] + c[3];
  const int inc = warp_inclusive_scan(lsum);
  if (lane == 31 && warp < kSelWarps) sm.s_wsum[warp] = inc;
  __syncthreads();
  const int ws = lane < kSelWarps ? sm.s_wsum[lane] : 0;
  const int wincl = warp_inclusive_scan(ws);
  const unsigned hit = __ballot_sync(0xffffffffu, wincl >= target);
  if (hit == 0u) return false;  // uniform: every warp sees the same totals
  const int wstar = __ffs(hit) - 1;
  if (warp == wstar) {
    int ex = __shfl_sync(0xffffffffu, wincl - ws, wstar) + inc - lsum;
#pragma unroll
    for (int i = 0; i < kBinsPerLane; ++i) {
      if (ex < target && target <= ex + c[i]) { sm.s_bin = kBinsPerLane * tid + i; sm.s_above = ex; }
      ex += c[i];
    }
  }
  __syncthreads();
  *bin = sm.s_bin;
  *above = sm.s_above;
  return true;
}

// The ids of the set take bits in ascending order: each thread owns a contiguous
// run of 32-id chunks, an exclusive prefix of their popcounts gives the position
// of its first id, and it writes its ids to sel[pos] for pos < min(limit, total).
// Returns the total number of set bits.
__device__ __forceinline__ int block_list_taken(const uint32_t* tm, int n, int* sel, int limit, SelSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + kSThreads - 1) / kSThreads;
  const int b0 = min(n, tid * per), b1 = min(n, b0 + per);
  int sum = 0;
  for (int i = b0; i < b1; ++i) sum += __popc(tm[i]);
  const int inc = warp_inclusive_scan(sum);
  if (lane == 31) sm.s_wt[warp] = inc;
  __syncthreads();
  const int x = lane < kSNW ? sm.s_wt[lane] : 0;
  int before = lane < warp ? x : 0, total = x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
  }
  const int lim = min(limit, total);
  int pos = before + inc - sum;
  for (int i = b0; i < b1; ++i) {
    for (uint32_t m = tm[i]; m != 0u; m &= m - 1u, ++pos)
      if (pos < lim) sel[pos] = i * 32 + __ffs(m) - 1;
  }
  return total;
}

// Key of cluster j recomputed from the scores and counts (when the keys do not
// fit in shared memory).  Out of line: it is the rare path.
__device__ __noinline__ uint32_t key_global(const uint32_t* s, int j) { return __ldcg(s + j); }

struct KeySrc {
  const uint32_t* ks;  // cached keys, or null
  const uint32_t* s;
  __device__ __forceinline__ uint32_t operator()(int j) const { return ks ? ks[j] : key_global(s, j); }
};

// The threshold bin holds more keys than threads (large ties): radix select
// (11-bit digits, ascending) over the 48-bit composite (d << 16) | id of the
// bin's keys (ids < 65536); the remaining-th one is the last taken, and every
// key of the bin up to it gets its take bit.  Out of line: the rare path.
__device__ __noinline__ void take_in_bin_radix(const KeySrc key_of, int C, uint32_t K0, int bstar, int remaining,
                                               uint32_t* tmask, SelSmem& sm) {
  const int tid = threadIdx.x;
  unsigned long long cpfx = 0ull, cmask = 0ull;
  int rem = remaining;
  bool ok = true;
  for (int i = tid; i < kTopkBins; i += kSThreads) sm.hist[1][i] = 0;
  __syncthreads();
  for (int pass = 0; pass < 5 && ok; ++pass) {
    const int sh = pass < 4 ? 37 - 11 * pass : 0;
    const unsigned long long dmask = pass < 4 ? 2047ull : 15ull;
    int* hc = sm.hist[(pass + 1) & 1];
    int* hn = sm.hist[pass & 1];
    for (int j = tid; j < C; j += kSThreads) {
      const uint32_t k = key_of(j);
      if (k == 0u) continue;
      const uint32_t d = K0 - k;
      const unsigned long long comp = ((unsigned long long)d << 16) | (unsigned)j;
      if (log_bin(d) == bstar && (comp & cmask) == cpfx) atomicAdd(&hc[(comp >> sh) & dmask], 1);
    }
    __syncthreads();
    for (int i = tid; i < kTopkBins; i += kSThreads) hn[i] = 0;
    int bin = 0, above = 0;
    ok = find_bin(hc, rem, sm, &bin, &above);
    rem -= above;
    cpfx |= (unsigned long long)bin << sh;
    cmask |= dmask << sh;
  }
  if (ok) {  // uniform
    for (int j = tid; j < C; j += kSThreads) {
      const uint32_t k = key_of(j);
      if (k == 0u) continue;
      const uint32_t d = K0 - k;
      const unsigned long long comp = ((unsigned long long)d << 16) | (unsigned)j;
      if (log_bin(d) == bstar && comp <= cpfx) atomicOr(&tmask[j >> 5], 1u << (j & 31));
    }
  }
}

// Top-k of key row h of unit u (a query head's scores, or with group-shared retrieval the heads'
// summed scores, row G), written out for that head or for every head of the unit.
template <int G, bool GRP>
__device__ __forceinline__ void select_role(unsigned char* raw, const TopkArgs& a, int u, int h) {
  SelSmem& sm = *reinterpret_cast<SelSmem*>(raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int GK = a.G + (GRP ? 1 : 0);    // key rows per unit
  const size_t uk = (size_t)u * GK + h;  // key row
  const int C = a.C, nch = (C + 31) / 32, kmax = a.kmax;
  uint32_t* ks = reinterpret_cast<uint32_t*>(raw + sizeof(SelSmem));                        // [C] if cached
  uint32_t* tmask = reinterpret_cast<uint32_t*>(raw + sizeof(SelSmem) + sel_keys_bytes(C, kmax));  // [nch]
  int* sel_s = reinterpret_cast<int*>(tmask + nch);                                           // [kmax] ids
  int* nc_s = sel_s + kmax;                                                                   // [kmax] rows
  int* of_s = nc_s + kmax;                                                                    // [kmax] first row
  int* rp_s = of_s + kmax;  // [kmax] first row among the selected rows
  const uint32_t* s = a.scores + uk * C;
  const int* cn = a.cnt + (size_t)u * C;
  const bool cached = C <= kSelKeysMax;
  bool rows_async = sel_rows_async(C, kmax);                  // uniform
  int* nc_a = reinterpret_cast<int*>(ks + C);                 // [C] counts of taken clusters, if rows_async
  int* of_a = nc_a + C;                                       // [C] their first rows
  const int* offu = a.off + (size_t)u * (C + 1);
  auto fetch_rows = [&](int j) {  // start the copies of cluster j's count and first row
    if (rows_async) {
      cp_async4(nc_a + j, cn + j);
      cp_async4(of_a + j, offu + j);
    }
  };
  const KeySrc key_of{cached ? ks : nullptr, s};
  uint16_t* kbin = reinterpret_cast<uint16_t*>(ks);  // [C] distance bins (0xFFFF: empty cluster) if !cached
  constexpr uint32_t kFarBin = 64 * 30;               // log_bin(2^30): the far keys' bins start here
  int kk = min(min(*a.kcur, kmax), a.nonempty[u]);
  // the first keys' loads are in flight across the K0 reduction and the barrier below
  const int n4 = C / 4;
  uint4 f[4];
  auto load4 = [&](int i0) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = i0 + r * kSThreads;
      f[r] = i < n4 ? __ldcg(reinterpret_cast<const uint4*>(s) + i) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  // cached keys: one bulk copy of the head's C keys into shared memory (the copy engine fetches them
  // as one request instead of every thread's vector loads); above kSelKeysMax, vector loads
  if (tid == 0) {  // the steady-row counters the split computation needs at the end, in flight meanwhile
    cp_async4(&sm.s_app, a.app_count);
    cp_async4(&sm.s_grown, a.grown);
  }
  if (cached) {
    if (tid == 0) {
      mbar_init(&sm.s_bar, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      mbar_arrive_expect_tx(&sm.s_bar, (uint32_t)C * 4u);
      bulk_g2s(ks, s, (uint32_t)C * 4u, &sm.s_bar);
    }
  } else {
    load4(tid);
  }
  // K0 = the largest key of a non-empty cluster, from k_scores' per-CTA maxima of the same
  // scores (every warp reduces them itself: no barrier)
  uint32_t K0 = 0u;
  for (int i = lane; i < a.P1; i += 32) K0 = max(K0, __ldcg(a.kmaxp + ((size_t)u * a.P1 + i) * GK + h));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) K0 = max(K0, __shfl_xor_sync(0xffffffffu, K0, o));
  for (int i = tid; i < kTopkBins; i += kSThreads) sm.hist[0][i] = 0;
  for (int i = tid; i < nch; i += kSThreads) tmask[i] = 0u;
  if (tid == 0) sm.s_ncand = 0;
  if (K0 == 0u) kk = 0;  // no non-empty cluster at all
  // ---- keys (C is a multiple of 16) and the logarithmic histogram of d = K0 - key.  Keys at
  // d >= 2^30 (in practice the negative scores, often half of all keys) fall into a handful of
  // bins where shared-memory atomics would serialize; they are counted (second round) only if
  // the nearer keys number fewer than k.
  auto count_key = [&](uint32_t k, bool far) {
    if (k != 0u && (K0 - k >= (1u << 30)) == far) atomicAdd(&sm.hist[0][log_bin(K0 - k)], 1);
  };
  if (cached) {
    __syncthreads();  // the histogram and the masks are zero; the barrier's init is visible
    // a timed-out wait is recorded; the CTA then selects nothing (uniformly), after waiting once more
    // (bounded) for its copy so that none lands after the CTA left
    if (__syncthreads_or(mbar_wait(&sm.s_bar, 0, a.err) ? 0 : 1)) {
      if (tid == 0) mbar_wait(&sm.s_bar, 0, a.err);
      kk = 0;
    }
    if (kk > 0)
      for (int i = tid; i < n4; i += kSThreads) {
        const uint4 k4 = reinterpret_cast<const uint4*>(ks)[i];
        count_key(k4.x, false);
        count_key(k4.y, false);
        count_key(k4.z, false);
        count_key(k4.w, false);
      }
  } else {
    __syncthreads();  // the histogram and the masks are zero
    auto bin_of = [&](uint32_t k) -> uint32_t { return k == 0u ? 0xFFFFu : (uint32_t)log_bin(K0 - k); };
    for (int i0 = tid; i0 < n4; i0 += 4 * kSThreads) {
      if (i0 != tid) load4(i0);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int i = i0 + r * kSThreads;
        if (i < n4) {
          const uint32_t b0 = bin_of(f[r].x), b1 = bin_of(f[r].y), b2 = bin_of(f[r].z), b3 = bin_of(f[r].w);
          reinterpret_cast<uint2*>(kbin)[i] = make_uint2(b0 | (b1 << 16), b2 | (b3 << 16));
          if (kk > 0) {
            if (b0 < kFarBin) atomicAdd(&sm.hist[0][b0], 1);
            if (b1 < kFarBin) atomicAdd(&sm.hist[0][b1], 1);
            if (b2 < kFarBin) atomicAdd(&sm.hist[0][b2], 1);
            if (b3 < kFarBin) atomicAdd(&sm.hist[0][b3], 1);
          }
        }
      }
    }
  }
  __syncthreads();
  bool found = kk == 0;
  int bstar = -1, remaining = 0;  // bstar -1: no bin, nothing is taken
  if (kk > 0) {
    int above = 0;
    found = find_bin(sm.hist[0], kk, sm, &bstar, &above);
    if (!found) {  // uniform: the k-th key is a far one; add the far keys and search again
      if (cached) {
        for (int j = tid; j < C; j += kSThreads) count_key(key_of(j), true);
      } else {
        for (int j = tid; j < C; j += kSThreads) {
          const uint32_t b = kbin[j];
          if (b != 0xFFFFu && b >= kFarBin) atomicAdd(&sm.hist[0][b], 1);
        }
      }
      __syncthreads();
      found = find_bin(sm.hist[0], kk, sm, &bstar, &above);
    }
    remaining = kk - above;
    if (!found) bstar = -1;
  }
  // ---- one pass: keys in bins below the threshold bin are taken (their bit set in the chunk
  // masks, about k of them), keys in it are candidates; bins are ranges of d, the threshold
  // bin is [dlo, dhi)
  const uint32_t dlo = bstar >= 0 ? log_bin_start(bstar) : 0u;
  const uint32_t dhi = bstar >= 0 && bstar < kTopkBins - 1 ? log_bin_start(bstar + 1) : 0xffffffffu;
  const bool top_open = bstar == kTopkBins - 1;  // the last bin also holds d = 2^32 - 1
  auto classify = [&](uint32_t k, int j) -> uint32_t {  // the take bit of j within its chunk, or 0
    const uint32_t d = K0 - k;
    if (k == 0u || d >= dhi && !top_open) return 0u;
    if (d < dlo) {
      fetch_rows(j);
      return 1u << (j & 31);
    }
    const int slot = atomicAdd(&sm.s_ncand, 1);
    if (slot < kSelThreads) { sm.ckey[slot] = k; sm.cid[slot] = j; }
    return 0u;
  };
  if (bstar >= 0) {
    if (cached) {  // four cached keys per load; their take bits share one chunk word
      for (int i = tid; i < C / 4; i += kSThreads) {
        const uint4 k4 = reinterpret_cast<const uint4*>(ks)[i];
        const int j = 4 * i;
        const uint32_t bits = classify(k4.x, j) | classify(k4.y, j + 1) | classify(k4.z, j + 2) |
                              classify(k4.w, j + 3);
        if (bits) atomicOr(&tmask[j >> 5], bits);
      }
    } else {  // four bins per load; the threshold bin's keys are read again from global memory
      for (int i = tid; i < C / 4; i += kSThreads) {
        const uint2 b2 = reinterpret_cast<const uint2*>(kbin)[i];
        const uint32_t bq[4] = {b2.x & 0xFFFFu, b2.x >> 16, b2.y & 0xFFFFu, b2.y >> 16};
        uint32_t bits = 0u;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int j = 4 * i + q;
          if (bq[q] == 0xFFFFu || (int)bq[q] > bstar) continue;
          if ((int)bq[q] < bstar) {
            bits |= 1u << (j & 31);
          } else {
            const uint32_t k = __ldcg(s + j);
            const int slot = atomicAdd(&sm.s_ncand, 1);
            if (slot < kSelThreads) { sm.ckey[slot] = k; sm.cid[slot] = j; }
          }
        }
        if (bits) atomicOr(&tmask[(4 * i) >> 5], bits);
      }
    }
  }
  __syncthreads();
  const int ncand = sm.s_ncand;
  if (kk > 0 && found) {
    if (ncand <= kSelThreads) {
      // rank of candidate tid in (key descending, id ascending) order: the first `remaining` are taken
      if (tid < ncand) {
        const uint32_t mk = sm.ckey[tid];
        const int mi = sm.cid[tid];
        int rank = 0;
        for (int i = 0; i < ncand; ++i) {
          const uint32_t ki = sm.ckey[i];
          rank += (ki > mk || (ki == mk && sm.cid[i] < mi)) ? 1 : 0;
        }
        if (rank < remaining) {
          atomicOr(&tmask[mi >> 5], 1u << (mi & 31));
          fetch_rows(mi);
        }
      }
    } else {
      take_in_bin_radix(key_of, C, K0, bstar, remaining, tmask, sm);
      rows_async = false;  // uniform: that path sets take bits only
    }
  }
  __syncthreads();
  // ---- the selection in id order
  const int total = block_list_taken(tmask, nch, sel_s, kk, sm);
  if (total != kk) {  // uniform; cannot happen with consistent counts
    if (tid == 0) atomicOr(a.err, WI_DEVERR_TOPK);
    kk = min(kk, total);  // every position below kk got an id
  }
  asm volatile("cp.async.wait_all;" ::: "memory");  // this thread's row copies have landed
  __syncthreads();
  // ---- per selected cluster (position p = tid + rounds of kSThreads): rows and their prefix
  int R = 0;
  for (int r0 = 0; r0 < kk; r0 += kSThreads) {  // uniform
    const int p = r0 + tid;
    const int j = p < kk ? sel_s[p] : 0;
    const int nc = p < kk ? (rows_async ? nc_a[j] : __ldg(cn + j)) : 0;
    const int of = p < kk ? (rows_async ? of_a[j] : __ldg(offu + j)) : 0;
    const int inc = warp_inclusive_scan(nc);
    if (lane == 31) sm.s_wt[warp] = inc;
    __syncthreads();
    const int x = lane < kSNW ? sm.s_wt[lane] : 0;
    int b = lane < warp ? x : 0, t = x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      b += __shfl_xor_sync(0xffffffffu, b, o);
      t += __shfl_xor_sync(0xffffffffu, t, o);
    }
    if (p < kk) {
      nc_s[p] = nc;
      of_s[p] = of;
      rp_s[p] = R + b + inc - nc;
    }
    R += t;
    __syncthreads();  // s_wt is reused by the next round; the position arrays are complete
  }
  if constexpr (!GRP) {
    const size_t uh = uk;  // key row = output head
    int* out = a.sel + uh * kmax;
    // ---- NSP = NS + 1 row-balanced splits of the head's exact rows [steady rows | selected rows]
    // (T = S + R rows): split b starts at row floor(T b / NSP), i.e. at selected row
    // max(0, floor(T b / NSP) - S): (position of the cluster holding that row, row inside it, the
    // selected row); entry NSP is the end.  Split 0 also takes the S steady rows.
    const float m_sub = kk > 0 ? a.lam * key_float(K0) : -INFINITY;
    const int NSP = a.NS + 1;
    int4* runs = a.runs + uh * kmax;
    int4* splits = a.splits + uh * (NSP + 1);
    int4* sruns = a.sruns + uh * NSP * 32;
    if (tid < NSP) {
      int4 sp = make_int4(0, 0, 0, 0);
      const long long S = (long long)a.n_sink + a.W + max(sm.s_app, 0) - (long long)sm.s_grown * a.seg_len,
                      T = S + R;
      const int rb = (int)max(0LL, (T * tid) / NSP - S);
      if (R > 0 && rb < R) {
        int lo = 0, hi = kk - 1;  // largest position whose first row is <= rb
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (rp_s[mid] <= rb) lo = mid; else hi = mid - 1;
        }
        sp = make_int4(lo, rb - rp_s[lo], rb, 0);
      } else {
        sp = make_int4(kk, 0, R, 0);
      }
      splits[tid] = sp;
      sm.s_spos[tid] = sp.x;
    }
    __syncthreads();
    // ---- row run and weight per selected cluster; copies into the run windows of the splits
    float zpart = 0.f;
    for (int p = tid; p < kk; p += kSThreads) {
      const int j = sel_s[p], nc = nc_s[p];
      const float w = __expf(a.lam * key_float(key_of(j)) - m_sub);
      const int4 run = make_int4(of_s[p], nc, __float_as_int(w), j);
      out[p] = j;
      runs[p] = run;
      for (int b = 0; b < NSP; ++b) {
        const int p0 = sm.s_spos[b];
        if (p0 > p) break;
        if (p < p0 + 32) sruns[b * 32 + (p - p0)] = run;
      }
      zpart = fmaf((float)nc, w, zpart);
    }
    for (int i = kk + tid; i < kmax; i += kSThreads) out[i] = -1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zpart += __shfl_xor_sync(0xffffffffu, zpart, o);
    if (lane == 0) sm.s_wf[warp] = zpart;
    __syncthreads();
    // the retrieved clusters' value-sum terms are summed by the exact-attention CTAs that load them
    if (tid == 0) {
      a.selcnt[uh] = kk;
      splits[NSP] = make_int4(kk, 0, R, 0);
      float zz = 0.f;
      for (int w = 0; w < kSNW; ++w) zz += sm.s_wf[w];
      float* sp = a.subpart + uh * WI_PART;
      sp[0] = m_sub;
      sp[1] = zz;
    }
  } else {
    // ---- NSP = NS + 1 row-balanced splits of the head's exact rows [steady rows | selected rows]
    // (T = S + R rows): split b starts at row floor(T b / NSP), i.e. at selected row
    // max(0, floor(T b / NSP) - S): (position of the cluster holding that row, row inside it, the
    // selected row); entry NSP is the end.  Split 0 also takes the S steady rows.  The rows do not
    // depend on the head: with group-shared retrieval every head of the unit gets these splits.
    const int NSP = a.NS + 1;
    int4 sp = make_int4(kk, 0, R, 0);
    if (tid < NSP) {
      const long long S = (long long)a.n_sink + a.W + max(sm.s_app, 0) - (long long)sm.s_grown * a.seg_len,
                      T = S + R;
      const int rb = (int)max(0LL, (T * tid) / NSP - S);
      if (R > 0 && rb < R) {
        int lo = 0, hi = kk - 1;  // largest position whose first row is <= rb
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (rp_s[mid] <= rb) lo = mid; else hi = mid - 1;
        }
        sp = make_int4(lo, rb - rp_s[lo], rb, 0);
      }
      sm.s_spos[tid] = sp.x;
    }
    __syncthreads();
    // every head's largest key (its m_sub) and its key of this thread's first selected cluster,
    // requested together: one round trip for all heads
    uint32_t K0g[G], keyg[G];
    const int pf = tid < kk ? sel_s[tid] : 0;
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      K0g[hh] = 0u;
      for (int i = lane; i < a.P1; i += 32) K0g[hh] = max(K0g[hh], __ldcg(a.kmaxp + ((size_t)u * a.P1 + i) * GK + hh));
      keyg[hh] = tid < kk ? __ldcg(a.scores + ((size_t)u * GK + hh) * C + pf) : 0u;
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) K0g[hh] = max(K0g[hh], __shfl_xor_sync(0xffffffffu, K0g[hh], o));
    }
    // ---- every (selected cluster, head) pair in one pass: the head's row run with its weight
    // e^{lam s_hj - m_sub_h}, the copies into its split windows, its share of the retrieved Z term
    float msub[G], zp[G];
#pragma unroll
    for (int ho = 0; ho < G; ++ho) {
      msub[ho] = kk > 0 ? a.lam * key_float(K0g[ho]) : -INFINITY;
      zp[ho] = 0.f;
    }
    for (int p = tid; p < kk; p += kSThreads) {
      const int j = sel_s[p], nc = nc_s[p], of = of_s[p];
#pragma unroll
      for (int ho = 0; ho < G; ++ho) {
        const size_t uo = (size_t)u * a.G + ho;
        const uint32_t key = p == tid ? keyg[ho] : __ldcg(a.scores + ((size_t)u * GK + ho) * C + j);
        const float w = __expf(a.lam * key_float(key) - msub[ho]);
        const int4 run = make_int4(of, nc, __float_as_int(w), j);
        a.sel[uo * kmax + p] = j;
        a.runs[uo * kmax + p] = run;
        int4* sruns = a.sruns + uo * NSP * 32;
        for (int b = 0; b < NSP; ++b) {
          const int p0 = sm.s_spos[b];
          if (p0 > p) break;
          if (p < p0 + 32) sruns[b * 32 + (p - p0)] = run;
        }
        zp[ho] = fmaf((float)nc, w, zp[ho]);
      }
    }
#pragma unroll
    for (int ho = 0; ho < G; ++ho) {
      const size_t uo = (size_t)u * a.G + ho;
      for (int i = kk + tid; i < kmax; i += kSThreads) a.sel[uo * kmax + i] = -1;
      if (tid < NSP) a.splits[uo * (NSP + 1) + tid] = sp;
    }
    // per-head Z terms: warp sums into shared scratch (the second histogram is free by now)
    float* wz = reinterpret_cast<float*>(sm.hist[1]);  // [warps][G]
#pragma unroll
    for (int ho = 0; ho < G; ++ho) {
      float z = zp[ho];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
      if (lane == 0) wz[warp * G + ho] = z;
    }
    __syncthreads();
    // the retrieved clusters' value-sum terms are summed by the exact-attention CTAs that load them
#pragma unroll
    for (int ho = 0; ho < G; ++ho) {
      if (tid == ho) {
        const size_t uo = (size_t)u * a.G + ho;
        float zz = 0.f;
        for (int w = 0; w < kSNW; ++w) zz += wz[w * G + ho];
        a.selcnt[uo] = kk;
        a.splits[uo * (NSP + 1) + NSP] = make_int4(kk, 0, R, 0);
        float* spp = a.subpart + uo * WI_PART;
        spp[0] = msub[ho];
        spp[1] = zz;
      }
    }
  }
}

template <int G, typename VT, bool GRP>
__global__ void __launch_bounds__(kSThreads, 1) k_select_estimate(TopkArgs a) {
  extern __shared__ __align__(128) unsigned char se_raw[];
  pdl_trigger();
  const int nsel = GRP ? a.U : a.U * a.G, nest = a.U * a.PE;
  // block order: the top-k CTAs first, or (when the estimation CTAs fit in one wave beside them) the
  // estimation CTAs first, so that their HBM stream overlaps the top-k instead of following it
  const int bi = blockIdx.x;
  const bool sel = a.est_first ? bi >= nest : bi < nsel;
  if (sel) {
    const int si = a.est_first ? bi - nest : bi;
    pdl_wait();
    // a query head's row, or with group-shared retrieval the unit's summed-score row G
    select_role<G, GRP>(se_raw, a, GRP ? si : si / a.G, GRP ? a.G : si % a.G);
  } else {
    const int e = a.est_first ? bi : bi - nsel;
    estimate_role<G, VT, G + (GRP ? 1 : 0)>(se_raw, static_cast<const VT*>(a.valsum), a.cnt, a.scores, a.part1,
                                            a.C, e / a.PE, e % a.PE, a.PE, a.lam, a.es_depth, a.err);
  }
}

// ---------------------------------------------------------- exact_merge ----
// CTA = (split, head, unit).  The head's exact rows -- the steady rows (sinks,
// local window, appended tokens) followed by its selected clusters' rows in
// position order -- are cut into NS+1 row-balanced splits by the top-k; split
// 0 starts with the steady rows (sinks and window copied before the
// dependency wait).  A producer lane packs the row runs into ROWS-row stages
// (K and V rows bulk-copied into shared memory; a stage with no rows ends the
// stream for the warps that take it); the 8 consumer warps form 8 / (ROWS /
// 8) groups, group g taking stages g, g + groups, ..., each warp 8 rows of a
// stage, flash-decode style.  The last CTA of the head (ticket counter) merges
// all partials into the output row.  96 KB of stages either way: 64-row
// stages take fewer bulk copies (a run is cut at every stage boundary), which
// rules when the CTAs come in several waves; 32-row stages hand the first
// rows to the consumers sooner, which rules a launch of one wave.
constexpr int kD3Warps = 8;
constexpr int kD3Threads = 32 * (kD3Warps + 1);
constexpr int kD3StageBytes = 96 * 1024;
constexpr int kTierPf = 8;  // host memory tier: page slots of a run looked up ahead (more: row by row)

template <int ROWS>
struct D3Geo {
  static constexpr int Rows = ROWS;
  static constexpr int Stages = kD3StageBytes / (ROWS * WI_D * 4);
  static constexpr int WPS = ROWS / 8;              // consumer warps per stage
  static constexpr int Groups = kD3Warps / WPS;     // stages consumed at once
  static_assert(ROWS % 8 == 0 && kD3Warps % WPS == 0 && Groups <= Stages, "stage geometry");
  struct Stage {
    bf16 k[ROWS * WI_D];
    bf16 v[ROWS * WI_D];
  };
  static constexpr size_t SMEM = sizeof(Stage) * Stages + 2 * Stages * sizeof(uint64_t) + 4 * Stages * sizeof(int) +
                                 sizeof(float) * kD3Warps * (WI_PART + WI_D) + 32 + 32 * kTierPf * sizeof(int);
};

struct ExactArgs {
  const bf16* q;
  const bf16* K;
  const bf16* V;
  const bf16* appK;
  const bf16* appV;
  const int* app_count;
  const bf16* grownK;  // [gmax][U][seg_len][128]: rows of the segments grown during decode
  const bf16* grownV;
  const int* grown;    // segments grown so far
  int gmax, seg_len, U;
  const int* selcnt;
  const int4* runs;
  const int4* splits;
  const int4* sruns;
  const void* valsum;  // [U][C][128] the value sums the estimate read: float, or their bf16 copy
  const int* nonempty;
  const float* part1;    // [U][G][P]
  const float* subpart;  // [U][G]
  float* part3;          // [U][G][NS+1]  exact partials
  float* subn;           // [U][G][NS+1]  value-sum terms of the retrieved clusters whose first row is here
  unsigned int* ticket;  // [U][G]
  unsigned long long* rows_total;
  float* out;
  int* err;
  long long n;
  int G, C, kmax, P, NS, n_sink, W, max_append;
  float lam;
  WiTierDev tier;  // host memory tier: clustered rows from cached pages or host memory (TIER instances)
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// The clustered rows of one unit seen through the host memory tier: page p (rows 16p .. 16p+15 of the
// unit's row space) is read from cache slot slot_of[p] when it holds one, else from host memory.
struct TierRows {
  const int* slot_of;
  const bf16* poolK;
  const bf16* poolV;
  const bf16* hostK;
  const bf16* hostV;
  int* use;
  int step;
  int (*pslot)[kTierPf];  // shared memory: [lane][page of its run] slots
  unsigned long long n_cache = 0, n_host = 0;  // rows copied: this lane's from cached pages; the warp's
                                               // from host memory (every lane counts them all)
};

// Producer of exact_merge: the whole producer warp.  The CTA's rows form one
// stream cut into 64-row stages; a batch of up to 32 runs (one per lane) is
// placed by a prefix sum of their lengths, then for every stage the batch
// touches, lane 0 opens the stage (waits until the consumers freed it) and
// announces its bytes, and each lane bulk-copies the part of its own run that
// falls in the stage (the copy engine takes ~60-100 cycles per copy, so the
// copies of a stage are issued by several lanes at once); a stage is closed
// once its 64 rows are placed.
template <int ROWS>
struct StagePacker {
  using Geo = D3Geo<ROWS>;
  static constexpr int kD3Rows = Geo::Rows, kD3Stages = Geo::Stages, kD3Groups = Geo::Groups;
  typename Geo::Stage* st;
  uint64_t* full;
  uint64_t* empty;
  int* nrows;
  int* err;
  int fpos = 0;     // rows placed so far (uniform in the warp)
  int opened = -1;  // last stage opened
  bool ok = true;   // uniform

  // this lane's run: rows [0, len) at kb / vb (len 0: no run)
  __device__ void push(const bf16* kb, const bf16* vb, int len) {
    const int lane = threadIdx.x & 31;
    const int incl = warp_inclusive_scan(len);
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    const int my0 = fpos + incl - len, my1 = my0 + len;
    const int A = fpos, B = fpos + total;
    for (int t = A / kD3Rows; ok && t * kD3Rows < B; ++t) {
      const int s = t % kD3Stages, r = t / kD3Stages;
      const int lo = max(A, t * kD3Rows), hi = min(B, (t + 1) * kD3Rows);
      if (lane == 0) {
        if (t > opened && r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, err)) ok = false;
        if (ok)
          asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&full[s])),
                       "r"((uint32_t)(hi - lo) * WI_D * 4)
                       : "memory");
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      opened = max(opened, t);
      if (!ok) break;
      const int p0 = max(my0, lo), p1 = min(my1, hi);
      if (p1 > p0) {
        const uint32_t bytes = (uint32_t)(p1 - p0) * WI_D * 2;
        const int d = p0 - t * kD3Rows;
        bulk_g2s(&st[s].k[d * WI_D], kb + (size_t)(p0 - my0) * WI_D, bytes, &full[s]);
        bulk_g2s(&st[s].v[d * WI_D], vb + (size_t)(p0 - my0) * WI_D, bytes, &full[s]);
      }
      if (hi == (t + 1) * kD3Rows && lane == 0) {  // the stage is full: hand it over
        nrows[s] = kD3Rows;
        mbar_arrive(&full[s]);
      }
    }
    if (ok) fpos = B;
  }

  // The same stream through the host memory tier: this lane's run is rows [row0, row0 + len) of the
  // unit's row space.  Its pages' slots are looked up first (one round trip for the warp).  For every
  // stage, each lane bulk-copies the pieces of its part that sit in cached pages (a piece ends at a
  // page boundary), after lane 0 announced their bytes; then the warp copies the rows of the pages
  // not cached, one row per instruction (16 bytes per lane: lanes 0-15 the key row, 16-31 the value
  // row) with cp.async from host memory, and every lane arms the stage's barrier with an arrive on
  // completion of its copies.
  __device__ void push_tier(TierRows& tr, int row0, int len) {
    const int lane = threadIdx.x & 31;
    const int pg0 = row0 >> 4;
    const int npg = len > 0 ? ((row0 + len - 1) >> 4) - pg0 + 1 : 0;
#pragma unroll
    for (int i = 0; i < kTierPf; ++i)
      if (i < npg) tr.pslot[lane][i] = __ldcg(tr.slot_of + pg0 + i);
    for (int i = 0; i < npg; ++i) tr.use[pg0 + i] = tr.step;
    __syncwarp();
    const int incl = warp_inclusive_scan(len);
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    const int my0 = fpos + incl - len, my1 = my0 + len;
    const int A = fpos, B = fpos + total;
    for (int t = A / kD3Rows; ok && t * kD3Rows < B; ++t) {
      const int s = t % kD3Stages, r = t / kD3Stages;
      const int lo = max(A, t * kD3Rows), hi = min(B, (t + 1) * kD3Rows);
      if (lane == 0 && t > opened && r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, err)) ok = false;
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      opened = max(opened, t);
      if (!ok) break;
      // this lane's part of the stage, page piece by page piece: the cached pieces by bulk copy
      const int q0 = max(my0, lo), q1 = min(my1, hi);
      auto piece_slot = [&](int sr) {
        const int pgi = (sr >> 4) - pg0;
        return pgi < kTierPf ? tr.pslot[lane][pgi] : __ldcg(tr.slot_of + (sr >> 4));
      };
      int cbytes = 0, hrows = 0;
      for (int i = q0; i < q1;) {
        const int sr = row0 + (i - my0), e = min(q1, i + kWiPageRows - (sr & 15));
        if (piece_slot(sr) >= 0) cbytes += (e - i) * WI_D * 4; else hrows += e - i;
        i = e;
      }
      const int cb = __reduce_add_sync(0xffffffffu, cbytes);
      if (lane == 0 && cb > 0)
        asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&full[s])),
                     "r"((uint32_t)cb)
                     : "memory");
      __syncwarp();
      for (int i = q0; i < q1;) {
        const int sr = row0 + (i - my0), e = min(q1, i + kWiPageRows - (sr & 15));
        const int slot = piece_slot(sr);
        if (slot >= 0) {
          const size_t o = ((size_t)slot * kWiPageRows + (sr & 15)) * WI_D;
          const uint32_t bytes = (uint32_t)(e - i) * WI_D * 2;
          bulk_g2s(&st[s].k[(i - t * kD3Rows) * WI_D], tr.poolK + o, bytes, &full[s]);
          bulk_g2s(&st[s].v[(i - t * kD3Rows) * WI_D], tr.poolV + o, bytes, &full[s]);
          tr.n_cache += e - i;  // this lane's cached rows
        }
        i = e;
      }
      // the rows of pages not cached: the lanes that own some, one row per warp instruction
      unsigned own = __ballot_sync(0xffffffffu, hrows > 0);
      bf16* dbase = (lane < 16 ? st[s].k : st[s].v) + (lane & 15) * 8;
      while (own) {
        const int L = __ffs(own) - 1;
        own &= own - 1;
        const int L0 = __shfl_sync(0xffffffffu, my0, L), L1 = __shfl_sync(0xffffffffu, my1, L);
        const int Lrow0 = __shfl_sync(0xffffffffu, row0, L);
        for (int i = max(L0, lo); i < min(L1, hi); ++i) {  // uniform
          const int sr = Lrow0 + (i - L0);
          const int pgi = (sr >> 4) - (Lrow0 >> 4);
          const int slot = pgi < kTierPf ? tr.pslot[L][pgi] : __ldcg(tr.slot_of + (sr >> 4));
          if (slot >= 0) continue;  // bulk-copied above (uniform)
          const bf16* src = (lane < 16 ? tr.hostK : tr.hostV) + (size_t)sr * WI_D;
          cp_async16(dbase + (i - t * kD3Rows) * WI_D, src + (lane & 15) * 8);
          ++tr.n_host;
        }
      }
      asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_addr(&full[s])) : "memory");
      __syncwarp();
      if (hi == (t + 1) * kD3Rows && lane == 0) {  // the stage is full: hand it over
        nrows[s] = kD3Rows;
        mbar_arrive(&full[s]);
      }
    }
    if (ok) fpos = B;
    __syncwarp();  // the slot scratch is rewritten by the next batch
  }
  // Close the partial last stage and send the end markers (kD3Groups consecutive stages with no
  // rows: one for every consumer group); on failure, close what is open and wait for the copies in
  // flight, so that none lands after the CTA left.
  __device__ void finish(int* abort_flag) {
    const int lane = threadIdx.x & 31;
    if (lane != 0) return;
    int t = fpos / kD3Rows;
    bool closed = fpos % kD3Rows == 0;  // no stage is half filled
    if (ok && !closed) {  // opened stage with rows: close it
      const int s = t % kD3Stages;
      nrows[s] = fpos % kD3Rows;
      mbar_arrive(&full[s]);
      closed = true;
      ++t;
    }
    for (int e = 0; ok && e < kD3Groups; ++e, ++t) {  // the end markers
      const int s = t % kD3Stages, r = t / kD3Stages;
      if (t > opened && r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, err)) ok = false;
      if (ok) {
        nrows[s] = 0;
        mbar_arrive(&full[s]);
      }
    }
    if (!ok) {
      *abort_flag = 1;
      if (!closed) {  // the stage being filled has rows in flight: let it complete
        const int s = (fpos / kD3Rows) % kD3Stages;
        nrows[s] = fpos % kD3Rows;
        mbar_arrive(&full[s]);
      }
      for (int tt = max(0, opened - kD3Stages + 1); tt <= opened; ++tt)  // bounded waits
        mbar_wait(&full[tt % kD3Stages], (tt / kD3Stages) & 1, err);
    }
  }
};

template <typename VT, int ROWS, bool TIER>
__global__ void __launch_bounds__(kD3Threads, 2) k_exact_merge(ExactArgs a) {
  using Geo = D3Geo<ROWS>;
  constexpr int kD3Stages = Geo::Stages, kD3WPS = Geo::WPS, kD3Groups = Geo::Groups;
  extern __shared__ __align__(128) unsigned char d3_raw[];
  typename Geo::Stage* st = reinterpret_cast<typename Geo::Stage*>(d3_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(d3_raw + sizeof(typename Geo::Stage) * kD3Stages);
  uint64_t* empty = full + kD3Stages;
  int* nrows = reinterpret_cast<int*>(empty + kD3Stages);        // [4 * stages]
  float* red = reinterpret_cast<float*>(nrows + 4 * kD3Stages);  // [warps][WI_PART]
  float* vred = red + kD3Warps * WI_PART;                         // [warps][WI_D] value-sum terms
  int* flags = reinterpret_cast<int*>(vred + kD3Warps * WI_D);    // abort, last CTA, kk, non-empty
  int(*pslot)[kTierPf] = reinterpret_cast<int(*)[kTierPf]>(flags + 8);  // [32][kTierPf] (tier only)
  const int split = blockIdx.x, h = blockIdx.y, u = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t uh = (size_t)u * a.G + h;
  const int nsp = a.NS + 1;  // CTAs per head
  pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < kD3Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kD3WPS);
    }
    flags[0] = 0;
    flags[1] = 0;
  }
  __syncthreads();
  float m = -INFINITY, Z = 0.f, N[4] = {0.f, 0.f, 0.f, 0.f};
  if (warp == kD3Warps) {
    const bf16* Ku = a.K + (size_t)u * a.n * WI_D;
    const bf16* Vu = a.V + (size_t)u * a.n * WI_D;
    StagePacker<ROWS> pk{st, full, empty, nrows, a.err};
    const long long ntier = (long long)a.n_sink + a.W;  // rows per unit of the tier's steady copy
    TierRows tr{};
    if constexpr (TIER) {
      const size_t pu = (size_t)u * a.tier.pages, su = (size_t)u * a.tier.slots * kWiPageRows * WI_D;
      tr.slot_of = a.tier.slot_of + pu;
      tr.poolK = static_cast<const bf16*>(a.tier.poolK) + su;
      tr.poolV = static_cast<const bf16*>(a.tier.poolV) + su;
      tr.hostK = static_cast<const bf16*>(a.tier.hostK) + (size_t)u * a.n * WI_D;
      tr.hostV = static_cast<const bf16*>(a.tier.hostV) + (size_t)u * a.n * WI_D;
      tr.use = a.tier.use + pu;
      tr.step = a.tier.step;
      tr.pslot = pslot;
    }
    const int amax = a.max_append > 0 ? a.max_append : 1;
    if (split == 0) {
      // ---- steady rows first: the sinks and (in an index that cannot grow) the build's local window
      // are fixed since the build (copied before the wait), the rest of the window after it
      const size_t w0 = (size_t)(a.n - a.W) * WI_D;
      const int wl = a.gmax == 0 ? a.W : 0;
      if constexpr (TIER) {  // the tier's device copy of the sinks and the window, [n_sink | W] rows
        const bf16* Ks = static_cast<const bf16*>(a.tier.steadyK) + (size_t)u * ntier * WI_D;
        const bf16* Vs = static_cast<const bf16*>(a.tier.steadyV) + (size_t)u * ntier * WI_D;
        const size_t ws = (size_t)a.n_sink * WI_D;
        pk.push(lane == 0 ? Ks : Ks + ws, lane == 0 ? Vs : Vs + ws, lane == 0 ? a.n_sink : (lane == 1 ? wl : 0));
      } else {
        pk.push(lane == 0 ? Ku : Ku + w0, lane == 0 ? Vu : Vu + w0, lane == 0 ? a.n_sink : (lane == 1 ? wl : 0));
      }
    }
    pdl_wait();
    const int ngrown = a.gmax > 0 ? min(*a.grown, a.gmax) : 0;
    if (split == 0) {
      const int na = *a.app_count;
      const bf16* Ka = a.appK + (size_t)u * amax * WI_D;
      const bf16* Va = a.appV + (size_t)u * amax * WI_D;
      if (a.gmax == 0) {
        pk.push(Ka, Va, lane == 0 ? na : 0);
      } else {
        // the window starts past the grown segments: the build's window rows not grown yet, then the
        // appended rows not grown yet
        const int gs = ngrown * a.seg_len;
        const int wrem = max(a.W - gs, 0), a0 = min(max(gs - a.W, 0), na);
        const size_t wr = (size_t)(a.n - wrem) * WI_D;
        pk.push(lane == 0 ? Ku + wr : Ka + (size_t)a0 * WI_D, lane == 0 ? Vu + wr : Va + (size_t)a0 * WI_D,
                lane == 0 ? wrem : (lane == 1 ? na - a0 : 0));
      }
    }
    // ---- selected clusters: rows [b_s, b_{s+1}) of the head's row-balanced split, 32 runs per
    // batch; one round trip gives the split bounds and the copies of its first 32 runs
    const int4 sa = a.splits[uh * (nsp + 1) + split];
    const int4 sb = a.splits[uh * (nsp + 1) + split + 1];
    const int kk = min(a.selcnt[uh], a.kmax);
    const int4 r0 = a.sruns[(uh * nsp + split) * 32 + lane];
    int rows_left = sb.z - sa.z;
    int pos = max(sa.x, 0), in = sa.y;
    const int4* runs = a.runs + uh * a.kmax;
    while (rows_left > 0 && pos < kk && pk.ok) {
      const int4 rr = (pos + lane < kk) ? (pos == sa.x ? r0 : runs[pos + lane]) : make_int4(0, 0, 0, 0);
      const int i_in = lane == 0 ? in : 0;
      const bool valid = pos + lane < kk;
      // a run must lie inside the build's clustered rows or (rows n.. : a grown segment's slots, seg_len
      // per segment) inside one grown segment; anything else is reported, never copied
      const bool in_grown = valid && (long long)rr.x >= a.n;
      const int gr = in_grown ? (int)((long long)rr.x - a.n) : 0;
      const int gseg = in_grown ? gr / a.seg_len : 0, goff = in_grown ? gr % a.seg_len : 0;
      const bool sane = !valid || (i_in >= 0 && i_in <= rr.y &&
                                   (in_grown ? (gseg < ngrown && goff + rr.y <= a.seg_len)
                                             : (rr.x >= a.n_sink && (long long)rr.x + rr.y <= a.n - a.W)));
      if (__any_sync(0xffffffffu, !sane)) {
        if (lane == 0) atomicOr(a.err, WI_DEVERR_BAD_ROW);
        break;
      }
      const int len = valid ? rr.y - i_in : 0;
      const int before = warp_inclusive_scan(len) - len;
      const int take = max(0, min(len, rows_left - before));
      if constexpr (TIER) {  // no grown segments with the tier
        pk.push_tier(tr, rr.x + i_in, take);  // whole warp
      } else {
        const size_t o = in_grown ? (((size_t)gseg * a.U + u) * a.seg_len + goff + i_in) * WI_D
                                  : (size_t)(rr.x + i_in) * WI_D;
        pk.push((in_grown ? a.grownK : Ku) + o, (in_grown ? a.grownV : Vu) + o, take);  // whole warp
      }
      rows_left -= __shfl_sync(0xffffffffu, warp_inclusive_scan(take), 31);
      in = 0;
      pos += 32;
    }
    pk.finish(&flags[0]);
    if (lane == 0) atomicAdd(a.rows_total, (unsigned long long)pk.fpos);
    if constexpr (TIER) {
      asm volatile("cp.async.wait_all;" ::: "memory");  // none of the copies lands after the CTA left
      const unsigned nc = __reduce_add_sync(0xffffffffu, (unsigned)tr.n_cache);
      if (lane == 0) {
        atomicAdd(a.tier.rows_src, (unsigned long long)nc);
        atomicAdd(a.tier.rows_src + 1, tr.n_host);
      }
    }
  } else {
    // ---- consumers
    pdl_wait();
    if (tid == 0) {  // the merge needs these; fetch them now, off the tail
      flags[2] = a.selcnt[uh];
      flags[3] = a.nonempty[u];
    }
    float qr[4];
    load_bf16x4(a.q + uh * WI_D + 4 * lane, qr);
    // value-sum terms sum_j w_j valsum_j of the retrieved clusters whose first row lies in this
    // split (clusters [first, last) of the selection), one round trip while the first stage lands
    float4 sub = make_float4(0.f, 0.f, 0.f, 0.f);
    {
      // the copies of the split's first 32 runs are read with the split bounds: window index
      // o + warp + 8x, o = 1 if the split starts inside a cluster (both offsets are fetched)
      const int4* sr = a.sruns + (uh * nsp + split) * 32;
      int4 e0[4], e1[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int i = warp + 8 * x;
        e0[x] = sr[i];
        e1[x] = i + 1 < 32 ? sr[i + 1] : make_int4(0, 0, 0, 0);
      }
      const int4 sa = a.splits[uh * (nsp + 1) + split];
      const int4 sb = a.splits[uh * (nsp + 1) + split + 1];
      const int kk = min(a.selcnt[uh], a.kmax);
      const int o = sa.y > 0 ? 1 : 0;
      const int first = max(sa.x, 0) + o;
      const int last = min(sb.x + (sb.y > 0 ? 1 : 0), kk);
      const int4* runs = a.runs + uh * a.kmax;
      // the terms subtracted are the ones the estimate added: from the same copy of the value sums
      // (the instance's type; no pointer of the other type exists in it)
      const VT* vsu = static_cast<const VT*>(a.valsum) + (size_t)u * a.C * WI_D + 4 * lane;
      auto ldvs = [&](int j) -> float4 {
        if constexpr (sizeof(VT) == 4) {
          return __ldg(reinterpret_cast<const float4*>(vsu + (size_t)j * WI_D));
        } else {
          float x[4];
          load_bf16x4(reinterpret_cast<const bf16*>(vsu) + (size_t)j * WI_D, x);
          return make_float4(x[0], x[1], x[2], x[3]);
        }
      };
      auto add_terms = [&](const float (&ww)[4], const float4 (&vv)[4]) {
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          sub.x = fmaf(ww[x], vv[x].x, sub.x);
          sub.y = fmaf(ww[x], vv[x].y, sub.y);
          sub.z = fmaf(ww[x], vv[x].z, sub.z);
          sub.w = fmaf(ww[x], vv[x].w, sub.w);
        }
      };
      {
        float4 vv[4];
        float ww[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int c = first + warp + 8 * x;
          const int4 rr = o ? e1[x] : e0[x];
          const bool v = c < last && o + warp + 8 * x < 32;
          const int j = (v && rr.w >= 0 && rr.w < a.C) ? rr.w : 0;
          ww[x] = v ? __int_as_float(rr.z) : 0.f;
          vv[x] = ldvs(j);
        }
        add_terms(ww, vv);
      }
      // clusters beyond the window
      for (int c0 = max(sa.x, 0) + 32 + warp; c0 < last; c0 += 4 * kD3Warps) {
        float4 vv[4];
        float ww[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int c = c0 + x * kD3Warps;
          const int4 rr = c < last ? runs[c] : make_int4(0, 0, 0, 0);
          const int j = (rr.w >= 0 && rr.w < a.C) ? rr.w : 0;
          ww[x] = c < last ? __int_as_float(rr.z) : 0.f;
          vv[x] = ldvs(j);
        }
        add_terms(ww, vv);
      }
    }
    const int ri = lane >> 2;  // the row (of the warp's 8) whose logit this lane ends with
    const int i0 = (warp % kD3WPS) * 8;  // the warp's rows of each stage its group takes
    for (int it = warp / kD3WPS;; it += kD3Groups) {
      const int s = it % kD3Stages, r = it / kD3Stages;
      if (!mbar_wait(&full[s], r & 1, a.err)) { flags[0] = 1; break; }
      const int nr = nrows[s];
      if (nr == 0) break;
      if (i0 < nr) {
        const typename Geo::Stage& T = st[s];
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float x[4];
          unpack_bf16x4(*reinterpret_cast<const uint2*>(&T.k[(i0 + i) * WI_D + 4 * lane]), x);
          float2 acc = __fmul2_rn(make_float2(qr[0], qr[1]), make_float2(x[0], x[1]));
          acc = __ffma2_rn(make_float2(qr[2], qr[3]), make_float2(x[2], x[3]), acc);
          v[i] = (i0 + i < nr) ? acc.x + acc.y : 0.f;
        }
        const float dot = transpose_reduce<8>(v);
        const float l = (i0 + ri < nr) ? a.lam * dot : -INFINITY;
        float mx = fmaxf(l, __shfl_xor_sync(0xffffffffu, l, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float m_new = fmaxf(m, mx);  // finite: row i0 is valid
        const float sc = __expf(m - m_new);
        const float pr = __expf(l - m_new);
        float zs = pr;  // each row's p sits in 4 lanes; these xors add each row once
        zs += __shfl_xor_sync(0xffffffffu, zs, 4);
        zs += __shfl_xor_sync(0xffffffffu, zs, 8);
        zs += __shfl_xor_sync(0xffffffffu, zs, 16);
        Z = Z * sc + zs;
        float2 nlo = __fmul2_rn(make_float2(N[0], N[1]), make_float2(sc, sc));
        float2 nhi = __fmul2_rn(make_float2(N[2], N[3]), make_float2(sc, sc));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float pi = __shfl_sync(0xffffffffu, pr, i * 4);
          if (i0 + i < nr) {
            float x[4];
            unpack_bf16x4(*reinterpret_cast<const uint2*>(&T.v[(i0 + i) * WI_D + 4 * lane]), x);
            nlo = __ffma2_rn(make_float2(pi, pi), make_float2(x[0], x[1]), nlo);
            nhi = __ffma2_rn(make_float2(pi, pi), make_float2(x[2], x[3]), nhi);
          }
        }
        N[0] = nlo.x; N[1] = nlo.y; N[2] = nhi.x; N[3] = nhi.y;
        m = m_new;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (lane == 0) {
      red[warp * WI_PART + 0] = m;
      red[warp * WI_PART + 1] = Z;
    }
    *reinterpret_cast<float4*>(&red[warp * WI_PART + 4 + 4 * lane]) = make_float4(N[0], N[1], N[2], N[3]);
    *reinterpret_cast<float4*>(&vred[warp * WI_D + 4 * lane]) = sub;
  }
  __syncthreads();
  if (flags[0]) return;
  // CTA partial
  float* o3 = a.part3 + (uh * nsp + split) * WI_PART;
  if (tid < WI_D) {
    float M = -INFINITY;
    for (int w = 0; w < kD3Warps; ++w) M = fmaxf(M, red[w * WI_PART]);
    float z = 0.f, acc = 0.f;
    if (M > -INFINITY)
      for (int w = 0; w < kD3Warps; ++w) {
        const float mw = red[w * WI_PART];
        if (mw == -INFINITY) continue;
        const float f = __expf(mw - M);
        z = fmaf(f, red[w * WI_PART + 1], z);
        acc = fmaf(f, red[w * WI_PART + 4 + tid], acc);
      }
    if (tid == 0) {
      o3[0] = M;
      o3[1] = z;
    }
    o3[4 + tid] = acc;
    float vs = 0.f;
#pragma unroll
    for (int w = 0; w < kD3Warps; ++w) vs += vred[w * WI_D + tid];
    a.subn[(uh * nsp + split) * WI_PART + 4 + tid] = vs;
  }
  // Publish this CTA's partial and take a ticket: the barrier orders the CTA's writes before
  // thread 0's release; the acquire side makes every earlier CTA's partial visible to the last one.
  __syncthreads();
  if (tid == 0) flags[1] = ticket_acq_rel(&a.ticket[uh]) == (unsigned)(nsp - 1);
  __syncthreads();
  if (!flags[1]) return;
  // ---- the last CTA of this head: estimate over all clusters - retrieved terms, plus exact, by LSE.
  // Rows: P estimation partials, nsp exact partials, nsp retrieved value-sum partials, then
  // (m_sub, Z_sub).  Every warp fetches the headers (m, Z) of all rows and the value columns of
  // its own rows in one round trip; the column sums meet in shared memory (the stages are free).
  const int kk = flags[2];
  const int nonempty = flags[3];
  constexpr int kMW = kD3Warps + 1;  // all warps of the CTA
  constexpr int kMR = 4;             // rows per warp per round trip
  const int P = a.P, rx = P, rs = P + nsp, rsub = P + 2 * nsp, nrow = rsub + 1;
  const float* p1 = a.part1 + uh * P * WI_PART;
  const float* p3 = a.part3 + uh * nsp * WI_PART;
  const float* ps = a.subn + uh * nsp * WI_PART;
  const float* sp = a.subpart + uh * WI_PART;
  auto grow = [&](int r) -> const float* {
    return r < rx ? p1 + (size_t)r * WI_PART
                  : (r < rs ? p3 + (size_t)(r - rx) * WI_PART
                            : (r < rsub ? ps + (size_t)(r - rs) * WI_PART : sp));
  };
  float* mz = reinterpret_cast<float*>(d3_raw);  // [nrow][2]
  float* wred = mz + 2 * ((nrow + 31) & ~31);   // [kMW][3][WI_D]: estimate, exact, value-sum columns
  float* zred = wred + kMW * 3 * WI_D;           // [kMW][2]
  float4 colv[kMR];
#pragma unroll
  for (int i = 0; i < kMR; ++i) {
    const int r = warp + i * kMW;
    colv[i] = r < nrow ? __ldcg(reinterpret_cast<const float4*>(grow(r) + 4) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int r = tid; r < nrow; r += kD3Threads) {
    const float2 h2 = __ldcg(reinterpret_cast<const float2*>(grow(r)));
    mz[2 * r] = h2.x;
    mz[2 * r + 1] = h2.y;
  }
  __syncthreads();
  float Me = -INFINITY, Mx = -INFINITY;
  for (int r = lane; r < rs; r += 32) {
    if (r < rx) Me = fmaxf(Me, mz[2 * r]);
    else Mx = fmaxf(Mx, mz[2 * r]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Me = fmaxf(Me, __shfl_xor_sync(0xffffffffu, Me, o));
    Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, o));
  }
  const bool use_est = Me > -INFINITY && kk < nonempty;
  float4 ce = make_float4(0.f, 0.f, 0.f, 0.f), cx = ce, cs = ce;
  float ze = 0.f, zx = 0.f;
  for (int r0 = warp; r0 < nrow; r0 += kMR * kMW) {
    if (r0 != warp) {  // rows beyond the first round trip (more partials than warps * kMR)
#pragma unroll
      for (int i = 0; i < kMR; ++i) {
        const int r = r0 + i * kMW;
        colv[i] = r < nrow ? __ldcg(reinterpret_cast<const float4*>(grow(r) + 4) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int i = 0; i < kMR; ++i) {
      const int r = r0 + i * kMW;
      if (r >= rsub) continue;
      const float mr = mz[2 * r], zr = mz[2 * r + 1];
      if (r < rx) {
        const float f = (use_est && mr > -INFINITY) ? __expf(mr - Me) : 0.f;
        ze = fmaf(f, zr, ze);
        ce.x = fmaf(f, colv[i].x, ce.x); ce.y = fmaf(f, colv[i].y, ce.y);
        ce.z = fmaf(f, colv[i].z, ce.z); ce.w = fmaf(f, colv[i].w, ce.w);
      } else if (r < rs) {
        const float f = mr > -INFINITY ? __expf(mr - Mx) : 0.f;
        zx = fmaf(f, zr, zx);
        cx.x = fmaf(f, colv[i].x, cx.x); cx.y = fmaf(f, colv[i].y, cx.y);
        cx.z = fmaf(f, colv[i].z, cx.z); cx.w = fmaf(f, colv[i].w, cx.w);
      } else {
        cs.x += colv[i].x; cs.y += colv[i].y; cs.z += colv[i].z; cs.w += colv[i].w;
      }
    }
  }
  reinterpret_cast<float4*>(wred + (warp * 3 + 0) * WI_D)[lane] = ce;
  reinterpret_cast<float4*>(wred + (warp * 3 + 1) * WI_D)[lane] = cx;
  reinterpret_cast<float4*>(wred + (warp * 3 + 2) * WI_D)[lane] = cs;
  if (lane == 0) {
    zred[2 * warp] = ze;
    zred[2 * warp + 1] = zx;
  }
  __syncthreads();
  if (tid < WI_D) {
    const int d = tid;
    float Ze = 0.f, Ne = 0.f, Zx = 0.f, Nx = 0.f, Ns = 0.f;
#pragma unroll
    for (int w = 0; w < kMW; ++w) {
      Ze += zred[2 * w];
      Zx += zred[2 * w + 1];
      Ne += wred[(w * 3 + 0) * WI_D + d];
      Nx += wred[(w * 3 + 1) * WI_D + d];
      Ns += wred[(w * 3 + 2) * WI_D + d];
    }
    if (use_est) {
      const float msub = mz[2 * rsub];
      if (msub > -INFINITY) {
        const float f = __expf(msub - Me);
        Ze = fmaf(-f, mz[2 * rsub + 1], Ze);
        Ne = fmaf(-f, Ns, Ne);
      }
      Ze = fmaxf(Ze, 0.f);
    } else {
      Ze = 0.f;
      Ne = 0.f;
    }
    const float M = fmaxf(Mx, Me);
    const float fx = Mx > -INFINITY ? __expf(Mx - M) : 0.f;
    const float fe = (use_est && Ze > 0.f) ? __expf(Me - M) : 0.f;
    a.out[uh * WI_D + d] = (Nx * fx + Ne * fe) / (Zx * fx + Ze * fe);
  }
  if (tid == 0) a.ticket[uh] = 0u;  // ready for the next step
}

// ------------------------------------------------------------- host copy ----
// 16-byte words from src to dst, either side possibly host memory mapped into the device's
// address space (the host-buffer step reads its query and writes its output this way).
__global__ void k_copy16(const uint4* __restrict__ src, uint4* __restrict__ dst, int n16) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += gridDim.x * blockDim.x) dst[i] = src[i];
}

// ---------------------------------------------------------------- append ----
__global__ void k_append(const bf16* __restrict__ k_new, const bf16* __restrict__ v_new, bf16* __restrict__ appK,
                         bf16* __restrict__ appV, int* __restrict__ app_count, int t, int max_append) {
  const int u = blockIdx.x, lane = threadIdx.x;
  const size_t dst = ((size_t)u * max_append + t) * WI_D;
  reinterpret_cast<uint2*>(appK + dst)[lane] = ldg_u2(k_new + (size_t)u * WI_D + 4 * lane);
  reinterpret_cast<uint2*>(appV + dst)[lane] = ldg_u2(v_new + (size_t)u * WI_D + 4 * lane);
  if (u == 0 && lane == 0) *app_count = t + 1;
}

// Optional timing events: ev[0] before the first kernel, ev[i] after the i-th.
inline cudaError_t mark(const cudaEvent_t* ev, int i, cudaStream_t st) {
  return ev ? cudaEventRecordWithFlags(ev[i], st, cudaEventRecordExternal) : cudaSuccess;
}

// Launch with programmatic dependent launch: the kernel may be scheduled
// while the previous kernel in the stream is still running; it calls
// griddepcontrol.wait before touching anything that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int G, typename VT, bool GRP>
cudaError_t launch_select_vt(const WiGeom& g, const WiDecodeBufs& b, const TopkArgs& t, cudaStream_t st) {
  const size_t sel = sel_smem_bytes(g.C, g.kmax), es = es_smem<VT>();
  const size_t smem = sel > es ? sel : es;
  static int smem_set[kWiSmemDevices] = {};
  cudaError_t e = wi_ensure_smem(k_select_estimate<G, VT, GRP>, smem, smem_set);
  if (e != cudaSuccess) return e;
  const int nsel = GRP ? g.U : g.U * G;
  return launch_pdl(k_select_estimate<G, VT, GRP>, dim3(nsel + g.U * b.p_es), dim3(kSThreads), smem, st, t);
}

template <int G, bool GRP>
cudaError_t launch_scores(const WiGeom& g, const WiDecodeBufs& b, const bf16* q, cudaStream_t st) {
  static int smem_set[kWiSmemDevices] = {};
  cudaError_t e = wi_ensure_smem(k_scores<G, GRP>, ScCfg<G>::SMEM, smem_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_scores<G, GRP>, dim3(b.p1, g.U), dim3(kScThreads), ScCfg<G>::SMEM, st, b.map_mu, q, b.cnt,
                    reinterpret_cast<uint32_t*>(b.scores), b.kmaxp, g.C, b.p1, b.err);
}

template <typename VT, int ROWS, bool TIER>
cudaError_t launch_exact_rows(const WiGeom& g, const WiDecodeBufs& b, const ExactArgs& a, cudaStream_t st) {
  static int smem_set[kWiSmemDevices] = {};
  constexpr size_t smem = D3Geo<ROWS>::SMEM;
  cudaError_t e = wi_ensure_smem(k_exact_merge<VT, ROWS, TIER>, smem, smem_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_exact_merge<VT, ROWS, TIER>, dim3(b.nsplit + 1, g.G, g.U), dim3(kD3Threads), smem, st, a);
}

template <typename VT>
cudaError_t launch_exact(const WiGeom& g, const WiDecodeBufs& b, const ExactArgs& a, cudaStream_t st) {
  if constexpr (sizeof(VT) == 4) {  // the tier holds fp32 value-sum indexes only
    if (b.tier.on)
      return b.d3_rows == 32 ? launch_exact_rows<VT, 32, true>(g, b, a, st) : launch_exact_rows<VT, 64, true>(g, b, a, st);
  }
  return b.d3_rows == 32 ? launch_exact_rows<VT, 32, false>(g, b, a, st) : launch_exact_rows<VT, 64, false>(g, b, a, st);
}

template <int G>
cudaError_t launch_select(const WiGeom& g, const WiDecodeBufs& b, const TopkArgs& t, cudaStream_t st) {
  if (g.grp)
    return b.valsum16 ? launch_select_vt<G, bf16, true>(g, b, t, st) : launch_select_vt<G, float, true>(g, b, t, st);
  return b.valsum16 ? launch_select_vt<G, bf16, false>(g, b, t, st) : launch_select_vt<G, float, false>(g, b, t, st);
}

template <int G>
cudaError_t launch_g(const WiGeom& g, const WiDecodeBufs& b, const void* qv, float* out, cudaStream_t st,
                     const cudaEvent_t* ev, unsigned mask) {
  const bf16* q = static_cast<const bf16*>(qv);
  const float lam = 1.0f / sqrtf((float)WI_D);
  cudaError_t e = mark(ev, 0, st);
  if (e != cudaSuccess) return e;
  // scores
  if (mask & 1u) e = g.grp ? launch_scores<G, true>(g, b, q, st) : launch_scores<G, false>(g, b, q, st);
  if (e != cudaSuccess || (e = mark(ev, 1, st)) != cudaSuccess) return e;
  TopkArgs t;
  t.scores = reinterpret_cast<const uint32_t*>(b.scores);
  t.cnt = b.cnt;
  t.off = b.off;
  t.nonempty = b.nonempty;
  t.valsum = b.valsum16 ? b.valsum16 : static_cast<const void*>(b.valsum);
  t.sel = b.sel;
  t.selcnt = b.selcnt;
  t.subpart = b.subpart;
  t.runs = b.runs;
  t.splits = b.splits;
  t.kmaxp = b.kmaxp;
  t.app_count = b.app_count;
  t.kcur = b.kcur;
  t.grown = b.grown;
  t.seg_len = g.S;
  t.W = g.W;
  t.P1 = b.p1;
  t.sruns = b.sruns;
  t.part1 = b.part1;
  t.err = b.err;
  t.U = g.U;
  t.G = G;
  t.C = g.C;
  t.kmax = g.kmax;
  t.NS = b.nsplit;
  t.PE = b.p_es;
  t.lam = lam;
  t.n_sink = g.n_sink;
  t.est_first = b.est_first;
  t.es_depth = b.es_depth;
  if (mask & 2u) e = launch_select<G>(g, b, t, st);
  if (e != cudaSuccess || (e = mark(ev, 2, st)) != cudaSuccess) return e;
  ExactArgs a;
  a.q = q;
  a.K = static_cast<const bf16*>(b.K);
  a.V = static_cast<const bf16*>(b.V);
  a.appK = static_cast<const bf16*>(b.appK);
  a.appV = static_cast<const bf16*>(b.appV);
  a.app_count = b.app_count;
  a.grownK = static_cast<const bf16*>(b.grownK);
  a.grownV = static_cast<const bf16*>(b.grownV);
  a.grown = b.grown;
  a.gmax = g.Gmax;
  a.seg_len = g.S;
  a.U = g.U;
  a.selcnt = b.selcnt;
  a.runs = b.runs;
  a.splits = b.splits;
  a.sruns = b.sruns;
  a.valsum = b.valsum16 ? b.valsum16 : static_cast<const void*>(b.valsum);
  a.subn = b.subn;
  a.C = g.C;
  a.nonempty = b.nonempty;
  a.part1 = b.part1;
  a.subpart = b.subpart;
  a.part3 = b.part3;
  a.ticket = b.ticket;
  a.rows_total = b.rows_total;
  a.out = out;
  a.err = b.err;
  a.n = g.n;
  a.G = G;
  a.kmax = g.kmax;
  a.P = b.p_es;
  a.NS = b.nsplit;
  a.n_sink = g.n_sink;
  a.W = g.W;
  a.max_append = g.max_append;
  a.lam = lam;
  a.tier = b.tier;
  if (mask & 4u) e = b.valsum16 ? launch_exact<bf16>(g, b, a, st) : launch_exact<float>(g, b, a, st);
  if (e != cudaSuccess) return e;
  return mark(ev, 3, st);
}

}  // namespace

cudaError_t wi_launch_decode(const WiGeom& g, const WiDecodeBufs& b, const void* q, float* out, cudaStream_t st,
                             const cudaEvent_t* ev, unsigned mask) {
  switch (g.G) {
    case 1: return launch_g<1>(g, b, q, out, st, ev, mask);
    case 2: return launch_g<2>(g, b, q, out, st, ev, mask);
    case 3: return launch_g<3>(g, b, q, out, st, ev, mask);
    case 4: return launch_g<4>(g, b, q, out, st, ev, mask);
    case 5: return launch_g<5>(g, b, q, out, st, ev, mask);
    case 6: return launch_g<6>(g, b, q, out, st, ev, mask);
    case 7: return launch_g<7>(g, b, q, out, st, ev, mask);
    case 8: return launch_g<8>(g, b, q, out, st, ev, mask);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t wi_launch_copy16(const void* src, void* dst, size_t bytes, cudaStream_t st) {
  const int n16 = (int)(bytes / 16);
  const int blocks = (n16 + 255) / 256 < 64 ? (n16 + 255) / 256 : 64;
  k_copy16<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16);
  return cudaGetLastError();
}

cudaError_t wi_launch_append(const WiGeom& g, const WiDecodeBufs& b, const void* k_new, const void* v_new, int t,
                             cudaStream_t st) {
  k_append<<<g.U, 32, 0, st>>>(static_cast<const bf16*>(k_new), static_cast<const bf16*>(v_new),
                               static_cast<bf16*>(b.appK), static_cast<bf16*>(b.appV), b.app_count, t,
                               g.max_append);
  return cudaGetLastError();
}
