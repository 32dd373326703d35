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
// Three kernels per step, each over the whole batch:
//   score_estimate  streams every cluster's mu / valsum / count through shared
//                   memory (bulk copies, mbarrier pipeline) once: the scores
//                   s_hj = q_h . mu_j of the G heads of the group, and the
//                   estimation partial (m, Z, N) over ALL non-empty clusters;
//   topk_sub        per head: radix select of the k best non-empty clusters
//                   (ties to the lowest id, ids ascending) and the estimation
//                   terms of exactly those clusters, to be taken back out;
//   exact_merge     per head and row split: flash-decode over the steady rows
//                   and the retrieved clusters' contiguous rows (bulk copies
//                   into shared memory); the last CTA of a head merges
//                   estimate - retrieved terms + exact partials by LSE.
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
constexpr int kTopkBins = 2048;  // first radix digit: the top 11 bits of the score key

// G query heads per kv head, in blocks of 4 heads (HB blocks); GP = heads per
// block rounded up to a power of two; NV = values per transpose-reduction
// (8 clusters x GP heads); lane l ends with cluster l >> 2 and in-block head
// (l & 3) >> SHIFT.
template <int G>
struct HeadGeo {
  static constexpr int HB = G > 4 ? 2 : 1;
  static constexpr int GP = G > 2 ? 4 : (G > 1 ? 2 : 1);
  static constexpr int NV = 8 * GP;
  static constexpr int SHIFT = GP == 4 ? 0 : (GP == 2 ? 1 : 2);
};

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

// ---- k_scores: s_hj = q_h . mu_j for every cluster on the tensor cores, and
// the histogram of the first radix digit of the score keys per head (for the
// top-k).  Per 128-cluster tile: TMA loads the mean keys (A, 128 x 128 bf16,
// K-major, 128-byte swizzle) and the counts; one thread issues eight
// tcgen05.mma (M = 128 clusters, N = 16 heads (G used, the rest zero), K = 16)
// into one of two 16-column TMEM accumulators; four epilogue warps read one
// cluster row each per lane (tcgen05.ld 32x32b.x16) and store the G scores.
// Warp 0: TMA producer; warp 1: TMEM allocation + MMA; warps 2..5: epilogue.
constexpr int kScTile = 128;
constexpr int kScEpiWarps = 4;
constexpr int kScThreads = 32 * (2 + kScEpiWarps);
constexpr int kScATile = kScTile * WI_D * 2;  // 32 KB: two 16 KB halves of 64 columns
constexpr int kScN = 16;                        // MMA N: heads padded to 16
constexpr int kScQBytes = kScN * WI_D * 2;      // 4 KB, the B operand

template <int G>
struct ScCfg {
  static constexpr int STAGES = G > 4 ? 4 : 5;
  static constexpr size_t A_OFF = kScQBytes;
  static constexpr size_t HIST_OFF = A_OFF + (size_t)STAGES * kScATile;
  static constexpr size_t CNT_OFF = HIST_OFF + sizeof(int) * G * kTopkBins;
  static constexpr size_t BAR_OFF = CNT_OFF + sizeof(int) * STAGES * kScTile;
  static constexpr size_t SMEM = BAR_OFF + sizeof(uint64_t) * (2 * STAGES + 4) + 16;
};

template <int G>
__global__ void __launch_bounds__(kScThreads, 1) k_scores(const __grid_constant__ CUtensorMap map_mu,
                                                         const bf16* __restrict__ q, const int* __restrict__ cnt,
                                                         float* __restrict__ scores, int* __restrict__ ghist, int C,
                                                         int P, int* err) {
  using CF = ScCfg<G>;
  constexpr int STAGES = CF::STAGES;
  extern __shared__ __align__(1024) unsigned char sc_raw[];
  unsigned char* qB = sc_raw;                                              // [k half][16 rows][128 B]
  unsigned char* A = sc_raw + CF::A_OFF;                                   // [stage][k half][128 rows][128 B]
  int* hist = reinterpret_cast<int*>(sc_raw + CF::HIST_OFF);              // [G][kTopkBins]
  int* cnts = reinterpret_cast<int*>(sc_raw + CF::CNT_OFF);               // [stage][128]
  uint64_t* full = reinterpret_cast<uint64_t*>(sc_raw + CF::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tbase = reinterpret_cast<uint32_t*>(tempty + 2);
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
      mbar_init(&empty[s], 1 + kScEpiWarps);  // the MMA commit and every epilogue warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kScEpiWarps);
    }
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;" ::"r"(smem_addr(tbase))
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
  for (int i = tid; i < G * kTopkBins; i += kScThreads) hist[i] = 0;
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
        const int s = it % STAGES, r = it / STAGES, b = it & 1;
        if (!mbar_wait(&full[s], r & 1, err)) { *s_abort = 1; break; }
        if (it >= 2 && !mbar_wait(&tempty[b], ((it >> 1) - 1) & 1, err)) { *s_abort = 1; break; }
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
    // epilogue: warp w reads TMEM lanes 32*(w%4).., i.e. clusters quarter*32 + lane of the tile
    const int quarter = warp & 3;
    bool ok = true;
    for (int it = 0; it < ntile; ++it) {
      const int s = it % STAGES, r = it / STAGES, b = it & 1;
      const int j0 = c0 + it * kScTile, nj = min(kScTile, c1 - j0);
      const int row = quarter * 32 + lane;
      uint32_t rr[16];
      if (ok) {
        if (!mbar_wait(&tfull[b], (it >> 1) & 1, err) || !mbar_wait(&full[s], r & 1, err)) {
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
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float sdot = __uint_as_float(rr[h]);
        if (valid) scores[((size_t)u * G + h) * C + j0 + row] = sdot;
        const int slot = (valid && cn > 0) ? h * kTopkBins + (int)(float_key(sdot) >> 21) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, slot);  // lanes of one digit add once
        if (slot >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[slot], __popc(peers));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;" ::"r"(tmem) : "memory");
  }
  if (*s_abort) return;
  for (int i = tid; i < G * kTopkBins; i += kScThreads) {
    const int c = hist[i];
    if (c) atomicAdd(&ghist[((size_t)u * G + i / kTopkBins) * kTopkBins + (i % kTopkBins)], c);
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
struct EsStage {
  float vs[kSTile * WI_D];
  int cnt[kSTile];
  float sc[8][kSTile];  // scores of up to 8 heads
};
constexpr size_t kEsSmem = sizeof(EsStage) * kEsStages + 2 * kEsStages * sizeof(uint64_t) +
                           sizeof(float) * kSWarps * 2 * 32 + sizeof(float) * kSWarps * 2 * 4 + 16;

template <int G>
__device__ void estimate_role(unsigned char* raw, const float* __restrict__ valsum, const int* __restrict__ cnt,
                              const float* __restrict__ scores, float* __restrict__ part, int C, int u, int p,
                              int P, float lam, int* err) {
  using HG = HeadGeo<G>;
  EsStage* st = reinterpret_cast<EsStage*>(raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(raw + sizeof(EsStage) * kEsStages);
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
      int issued = 0;
      for (int it = 0; it < ntile; ++it) {
        const int s = it % kEsStages, r = it / kEsStages;
        if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, err)) { *s_abort = 1; break; }
        const int j0 = c0 + it * kSTile, nj = min(kSTile, c1 - j0);
        mbar_arrive_expect_tx(&full[s], (uint32_t)nj * (WI_D * 4 + 4 + 4 * G));
        const size_t row = (size_t)u * C + j0;
        bulk_g2s(st[s].vs, valsum + row * WI_D, nj * WI_D * 4, &full[s]);
        bulk_g2s(st[s].cnt, cnt + row, nj * 4, &full[s]);
        for (int h = 0; h < G; ++h) bulk_g2s(st[s].sc[h], scores + ((size_t)u * G + h) * C + j0, nj * 4, &full[s]);
        issued = it + 1;
      }
      if (*s_abort) drain_stages<kEsStages>(full, issued, err);
    }
  } else {
    float* pb = pbuf + warp * 2 * 32;
    float* sb = sbuf + warp * 2 * 4;
    for (int it = 0; it < ntile; ++it) {
      const int s = it % kEsStages, r = it / kEsStages;
      if (!mbar_wait(&full[s], r & 1, err)) { *s_abort = 1; break; }
      const EsStage& T = st[s];
      const int j0 = c0 + it * kSTile, nj = min(kSTile, c1 - j0);
      const int i0 = warp * 8;
      if (i0 < nj) {
        const bool valid_c = (i0 + ci) < nj;
        const int cn = valid_c ? T.cnt[i0 + ci] : 0;
#pragma unroll
        for (int b = 0; b < HG::HB; ++b) {
          const int head = b * 4 + hl;
          const bool valid = valid_c && head < G;
          const float se = (valid && cn > 0) ? lam * T.sc[head < G ? head : 0][i0 + ci] : -INFINITY;
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
          const float4 vv = *reinterpret_cast<const float4*>(&T.vs[(i0 + i) * WI_D + 4 * lane]);
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

// -- select role: top-k of one head.  KPT consecutive clusters per thread
// (threads 0..511; the remaining warp only meets the barriers), held as
// order-preserving keys in registers (0 = empty cluster / padding).  Three
// radix passes (11, 11, 10 bits) find the k-th largest key T -- the first
// digit's histogram comes from k_scores -- then the keys > T and the first (in
// id order) keys == T are written in id order, with each selected cluster's
// row run and weight (first row, rows, e^{lam s_j - m_sub}, id), m_sub =
// lam * s_max, and the starts of NS row-balanced splits of the selected rows.
// Also Z_sub = sum n_j e^{lam s_j - m_sub} over the selected clusters; their
// value-sum terms are summed where their rows are loaded (exact attention),
// and both are subtracted from the estimate at the merge.
constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kBinsPerLane = kTopkBins / kSelThreads;  // 4

// Inverse of float_key for finite scores.
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

struct TopkArgs {
  int* ghist;    // [U][G][kTopkBins] first-digit histogram from k_scores; cleared here after use
  const float* scores;
  const int* cnt;
  const int* off;
  const int* nonempty;
  const float* valsum;
  int* sel;
  int* selcnt;
  float* subpart;
  int4* runs;    // [U][G][kmax]  (first row, rows, weight bits e^{lam s - m_sub}, cluster id)
  int4* splits;  // [U][G][NS+1]  (position, row inside that cluster, split's first row, 0)
  float* part1;  // estimation partials [U][G][PE]
  int* err;
  int U, G, C, kmax, NS, PE, n_sink;
  float lam;
};

// Inclusive warp scan of 64-bit counts.
__device__ __forceinline__ unsigned long long warp_scan_u64(unsigned long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Exclusive block-wide prefix of a 64-bit count per thread, one barrier: warp
// totals go through `wt` (>= 32 entries); returns the prefix, sets *total.
__device__ __forceinline__ unsigned long long block_prefix_u64(unsigned long long v, unsigned long long* wt,
                                                               unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const unsigned long long inc = warp_scan_u64(v);
  if (lane == 31) wt[warp] = inc;
  __syncthreads();
  const unsigned long long x = lane < nw ? wt[lane] : 0ull;
  unsigned long long before = lane < warp ? x : 0ull, all = x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    all += __shfl_xor_sync(0xffffffffu, all, o);
  }
  *total = all;
  return before + inc - v;
}

struct SelSmem {
  int hist[2][kTopkBins];
  int s_wsum[32];
  int s_bin, s_above;
  uint32_t s_maxkey;
  int pad;
  unsigned long long s_wt[3][32];
  float zred[32];
};

template <int KPT>
__device__ void select_role(unsigned char* raw, const TopkArgs& a, int u, int h) {
  static_assert(KPT % 4 == 0, "vector loads of 4");
  SelSmem& sm = *reinterpret_cast<SelSmem*>(raw);
  int* s_row = reinterpret_cast<int*>(raw + sizeof(SelSmem));  // [kmax + 1] row prefix in selection order
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t uh = (size_t)u * a.G + h;
  const int C = a.C;
  const float* s = a.scores + uh * C;
  const int* cn = a.cnt + (size_t)u * C;
  int* out = a.sel + uh * a.kmax;
  // every global read this CTA needs is issued here, before the first use (all of it is in L2:
  // the scores and the histogram were just written, the counts just read, by k_scores)
  uint32_t key[KPT];
  int nc[KPT];
  int4 g4 = make_int4(0, 0, 0, 0);
  const bool scan_lane = warp < kSelWarps;
  const int rb0 = kBinsPerLane * tid;  // this lane's reversed bins rb0 .. rb0+3 (bins 2047-rb0 .. 2044-rb0)
  int* gh = a.ghist + uh * kTopkBins;
  if (scan_lane) g4 = __ldcg(reinterpret_cast<const int4*>(gh + kTopkBins - kBinsPerLane - rb0));
  const int base = tid * KPT;
  if (base + KPT <= C) {
#pragma unroll
    for (int e = 0; e < KPT; e += 4) {
      const int4 c4 = __ldg(reinterpret_cast<const int4*>(cn + base + e));
      const float4 f4 = __ldcg(reinterpret_cast<const float4*>(s + base + e));
      nc[e] = c4.x; nc[e + 1] = c4.y; nc[e + 2] = c4.z; nc[e + 3] = c4.w;
      key[e] = float_key(f4.x); key[e + 1] = float_key(f4.y);
      key[e + 2] = float_key(f4.z); key[e + 3] = float_key(f4.w);
    }
  } else {
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
      const int j = base + e;
      nc[e] = j < C ? __ldg(cn + j) : 0;
      key[e] = j < C ? float_key(__ldcg(s + j)) : 0u;
    }
  }
  int kk = min(a.kmax, a.nonempty[u]);
#pragma unroll
  for (int e = 0; e < KPT; ++e)
    if (nc[e] <= 0) key[e] = 0u;  // empty clusters are never candidates
  if (scan_lane) *reinterpret_cast<int4*>(gh + kTopkBins - kBinsPerLane - rb0) = make_int4(0, 0, 0, 0);
  for (int i = tid; i < a.kmax; i += kSThreads) out[i] = -1;
  for (int i = tid; i < kTopkBins; i += kSThreads) sm.hist[1][i] = 0;
  if (tid == 0) { a.selcnt[uh] = kk; sm.s_maxkey = 0u; }
  // ---- radix select: three passes of (count, barrier, scan, barrier, pick, barrier)
  uint32_t prefix = 0, pmask = 0;
  int remaining = kk;
  bool found = true;
#pragma unroll 1
  for (int pass = 0; pass < 3 && kk > 0; ++pass) {
    const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t dmask = pass == 2 ? 1023u : 2047u;
    int* hc = sm.hist[pass & 1];
    int* hn = sm.hist[(pass + 1) & 1];
    if (pass > 0) {
#pragma unroll
      for (int e = 0; e < KPT; ++e)
        if (key[e] != 0u && (key[e] & pmask) == prefix) atomicAdd(&hc[(key[e] >> sh) & dmask], 1);
    }
    __syncthreads();
    int c[kBinsPerLane];
    if (pass == 0) {  // the first digit's counts came from k_scores, in ascending bin order
      c[0] = g4.w; c[1] = g4.z; c[2] = g4.y; c[3] = g4.x;
    } else {
#pragma unroll
      for (int i = 0; i < kBinsPerLane; ++i) c[i] = scan_lane ? hc[kTopkBins - 1 - rb0 - i] : 0;
    }
    int lsum = 0;
#pragma unroll
    for (int i = 0; i < kBinsPerLane; ++i) lsum += c[i];
    const int inc = warp_inclusive_scan(lsum);
    if (lane == 31) sm.s_wsum[warp] = inc;
    if (pass + 1 < 3)
      for (int i = tid; i < kTopkBins; i += kSThreads) hn[i] = 0;
    __syncthreads();
    const int ws = lane < kSelWarps ? sm.s_wsum[lane] : 0;
    const int wincl = warp_inclusive_scan(ws);
    const unsigned hit = __ballot_sync(0xffffffffu, wincl >= remaining);
    const int wstar = __ffs(hit) - 1;  // warp whose bins hold the remaining-th largest key
    if (wstar < 0) {                   // inconsistent counts: select nothing, report it
      found = false;
      break;
    }
    if (warp == wstar) {
      int ex = __shfl_sync(0xffffffffu, wincl - ws, wstar) + inc - lsum;
#pragma unroll
      for (int i = 0; i < kBinsPerLane; ++i) {
        if (ex < remaining && remaining <= ex + c[i]) { sm.s_bin = kTopkBins - 1 - rb0 - i; sm.s_above = ex; }
        ex += c[i];
      }
    }
    __syncthreads();
    remaining -= sm.s_above;
    prefix |= (uint32_t)sm.s_bin << sh;
    pmask |= dmask << sh;
  }
  if (!found) {
    if (tid == 0) atomicOr(a.err, WI_DEVERR_TOPK);
    kk = 0;
    if (tid == 0) a.selcnt[uh] = 0;
  }
  const uint32_t T = kk > 0 ? prefix : 0xffffffffu;  // nothing is taken when kk == 0
  // ---- compaction in id order
  uint32_t kmx = 0u;
  int cgt = 0, ceq = 0;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    kmx = max(kmx, key[e]);
    cgt += key[e] > T;
    ceq += (key[e] != 0u && key[e] == T);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) kmx = max(kmx, __shfl_xor_sync(0xffffffffu, kmx, o));
  if (lane == 0) atomicMax(&sm.s_maxkey, kmx);
  unsigned long long tot;
  const unsigned long long pre =
      block_prefix_u64(((unsigned long long)cgt << 32) | (unsigned)ceq, sm.s_wt[0], &tot);
  const int pre_gt = (int)(pre >> 32), pre_eq = (int)(pre & 0xffffffffu);
  const int tot_gt = (int)(tot >> 32), tot_eq = (int)(tot & 0xffffffffu);
  const float m_sub = kk > 0 ? a.lam * key_float(sm.s_maxkey) : -INFINITY;
  int eq_seen = pre_eq, my_rows = 0;
  uint32_t takemask = 0u;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    const bool is_eq = key[e] != 0u && key[e] == T;
    const bool take = key[e] > T || (is_eq && eq_seen < remaining);
    eq_seen += is_eq ? 1 : 0;
    if (take) { takemask |= 1u << e; my_rows += nc[e]; }
  }
  unsigned long long rtot, ctot;
  const int row_pre = (int)block_prefix_u64((unsigned long long)my_rows, sm.s_wt[1], &rtot);
  // a cluster's first row = n_sink + the counts of all lower ids (the cluster-contiguous layout)
  int csum = 0;
#pragma unroll
  for (int e = 0; e < KPT; ++e) csum += nc[e];
  int of = a.n_sink + (int)block_prefix_u64((unsigned long long)csum, sm.s_wt[2], &ctot);
  int pos = pre_gt + min(pre_eq, remaining);
  int rp = row_pre;
  float zpart = 0.f;
  int4* runs = a.runs + uh * a.kmax;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    if (takemask & (1u << e)) {
      if (pos < kk) {
        const int j = base + e;
        const float w = __expf(a.lam * key_float(key[e]) - m_sub);
        out[pos] = j;
        s_row[pos] = rp;
        runs[pos] = make_int4(of, nc[e], __float_as_int(w), j);
        zpart = fmaf((float)nc[e], w, zpart);
      }
      rp += nc[e];
      ++pos;
    }
    of += nc[e];
  }
  if (tid == 0) {
    s_row[kk] = (int)rtot;
    if (tot_gt + min(tot_eq, remaining) != kk) atomicOr(a.err, WI_DEVERR_TOPK);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) zpart += __shfl_xor_sync(0xffffffffu, zpart, o);
  if (lane == 0) sm.zred[warp] = zpart;
  __syncthreads();
  // split s starts at row b_s = R * s / NS: (position of its first cluster, row inside it, b_s)
  if (tid <= a.NS) {
    const int R = s_row[kk];
    const int b = (int)((long long)R * tid / a.NS);
    int lo = 0, hi = kk;  // largest position with s_row[pos] <= b
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_row[mid] <= b) lo = mid; else hi = mid - 1;
    }
    if (b >= R) lo = kk;
    a.splits[uh * (a.NS + 1) + tid] = make_int4(lo, b - (lo < kk ? s_row[lo] : R), b, 0);
  }
  // the retrieved clusters' value-sum terms are summed by the exact-attention CTAs that load them
  if (tid == 0) {
    float* sp = a.subpart + uh * WI_PART;
    float zz = 0.f;
    for (int w = 0; w < kSelWarps; ++w) zz += sm.zred[w];
    sp[0] = m_sub;
    sp[1] = zz;
  }
}

template <int G, int KPT>
__global__ void __launch_bounds__(kSThreads, 1) k_select_estimate(TopkArgs a) {
  extern __shared__ __align__(128) unsigned char se_raw[];
  pdl_trigger();
  pdl_wait();
  const int nsel = a.U * a.G;
  if ((int)blockIdx.x < nsel) {
    select_role<KPT>(se_raw, a, blockIdx.x / a.G, blockIdx.x % a.G);
  } else {
    const int e = blockIdx.x - nsel;
    estimate_role<G>(se_raw, a.valsum, a.cnt, a.scores, a.part1, a.C, e / a.PE, e % a.PE, a.PE, a.lam, a.err);
  }
}

// ---------------------------------------------------------- exact_merge ----
// CTA = (split, head, unit).  Splits 0..NS-1 take row-balanced shares of the
// head's selected clusters (the split starts come from topk_sub); split NS
// takes the steady rows (sinks and local window, which it starts copying
// before the previous kernel has finished, then the appended tokens).  A
// producer lane packs the row runs into 64-row stages (K and V rows
// bulk-copied into shared memory; a stage with no rows ends the stream); 8
// consumer warps take 8 rows each per stage, flash-decode style.  The last
// CTA of the head (ticket counter) merges all partials into the output row.
constexpr int kD3Rows = 64;
constexpr int kD3Stages = 3;
constexpr int kD3Warps = 8;
constexpr int kD3Threads = 32 * (kD3Warps + 1);

struct D3Stage {
  bf16 k[kD3Rows * WI_D];
  bf16 v[kD3Rows * WI_D];
};
constexpr size_t kD3Smem = sizeof(D3Stage) * kD3Stages + 2 * kD3Stages * sizeof(uint64_t) +
                           4 * kD3Stages * sizeof(int) + sizeof(float) * kD3Warps * WI_PART + 32;

struct ExactArgs {
  const bf16* q;
  const bf16* K;
  const bf16* V;
  const bf16* appK;
  const bf16* appV;
  const int* app_count;
  const int* selcnt;
  const int4* runs;
  const int4* splits;
  const float* valsum;
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
};

// Producer state of exact_merge (lane 0 of the producer warp only).
struct RunPacker {
  D3Stage* st;
  uint64_t* full;
  uint64_t* empty;
  int* nrows;
  int* err;
  int stage_it = 0, fill = 0;
  bool opened = false;
  long long rows_done = 0;

  __device__ bool open() {
    const int s = stage_it % kD3Stages, r = stage_it / kD3Stages;
    if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, err)) return false;
    fill = 0;
    opened = true;
    return true;
  }
  __device__ void close() {
    const int s = stage_it % kD3Stages;
    nrows[s] = fill;
    mbar_arrive(&full[s]);  // completes the stage once its announced bytes have landed
    ++stage_it;
    opened = false;
  }
  // rows [0, len) of the runs starting at kb / vb
  __device__ bool push(const bf16* kb, const bf16* vb, int len) {
    while (len > 0) {
      if (!opened && !open()) return false;
      const int s = stage_it % kD3Stages;
      const int take = min(len, kD3Rows - fill);
      const uint32_t bytes = (uint32_t)take * WI_D * 2;
      asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&full[s])),
                   "r"(2 * bytes)
                   : "memory");
      bulk_g2s(&st[s].k[fill * WI_D], kb, bytes, &full[s]);
      bulk_g2s(&st[s].v[fill * WI_D], vb, bytes, &full[s]);
      fill += take;
      rows_done += take;
      kb += (size_t)take * WI_D;
      vb += (size_t)take * WI_D;
      len -= take;
      if (fill == kD3Rows) close();
    }
    return true;
  }
};

__global__ void __launch_bounds__(kD3Threads, 2) k_exact_merge(ExactArgs a) {
  extern __shared__ __align__(128) unsigned char d3_raw[];
  D3Stage* st = reinterpret_cast<D3Stage*>(d3_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(d3_raw + sizeof(D3Stage) * kD3Stages);
  uint64_t* empty = full + kD3Stages;
  int* nrows = reinterpret_cast<int*>(empty + kD3Stages);        // [4 * stages]
  float* red = reinterpret_cast<float*>(nrows + 4 * kD3Stages);  // [warps][WI_PART]
  int* flags = reinterpret_cast<int*>(red + kD3Warps * WI_PART);  // abort, last CTA, kk, non-empty
  const int split = blockIdx.x, h = blockIdx.y, u = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t uh = (size_t)u * a.G + h;
  const int nsp = a.NS + 1;  // CTAs per head
  pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < kD3Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kD3Warps);
    }
    flags[0] = 0;
    flags[1] = 0;
  }
  __syncthreads();
  float m = -INFINITY, Z = 0.f, N[4] = {0.f, 0.f, 0.f, 0.f};
  if (warp == kD3Warps) {
    const bf16* Ku = a.K + (size_t)u * a.n * WI_D;
    const bf16* Vu = a.V + (size_t)u * a.n * WI_D;
    RunPacker pk{st, full, empty, nrows, a.err};
    bool ok = true;
    if (split == a.NS) {
      // ---- steady rows: sinks and local window are fixed since the build; appended rows after the wait
      if (lane == 0) {
        ok = ok && pk.push(Ku, Vu, a.n_sink);
        ok = ok && pk.push(Ku + (size_t)(a.n - a.W) * WI_D, Vu + (size_t)(a.n - a.W) * WI_D, a.W);
      }
      pdl_wait();
      reinterpret_cast<float4*>(a.subn + (uh * nsp + split) * WI_PART + 4)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (lane == 0) {
        const int amax = a.max_append > 0 ? a.max_append : 1;
        ok = ok && pk.push(a.appK + (size_t)u * amax * WI_D, a.appV + (size_t)u * amax * WI_D, *a.app_count);
      }
    } else {
      // ---- selected clusters: rows [b_s, b_{s+1}) of the head's row-balanced split
      pdl_wait();
      const int4 sa = a.splits[uh * nsp + split];
      const int4 sb = a.splits[uh * nsp + split + 1];
      const int kk = min(a.selcnt[uh], a.kmax);
      int rows_left = sb.z - sa.z;
      int pos = max(sa.x, 0), in = sa.y;
      const int4* runs = a.runs + uh * a.kmax;
      const float4* vsu = reinterpret_cast<const float4*>(a.valsum + (size_t)u * a.C * WI_D) + lane;
      float4 sub = make_float4(0.f, 0.f, 0.f, 0.f);  // value-sum terms of the clusters that start here
      while (rows_left > 0 && pos < kk) {
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
        const int4 rr = (pos + lane < kk) ? runs[pos + lane] : make_int4(0, 0, 0, 0);
        const int nb = min(32, kk - pos);
        int used = 0;
        const int first_in = in;
        for (int i = 0; i < nb && rows_left > 0; ++i) {
          const int o = __shfl_sync(0xffffffffu, rr.x, i);
          const int z = __shfl_sync(0xffffffffu, rr.y, i);
          const int take = min(z - in, rows_left);
          // a run must lie inside the clustered rows; anything else is reported, never copied
          const bool sane = in >= 0 && in <= z && o >= a.n_sink && (long long)o + z <= a.n - a.W;
          if (!sane) {
            if (lane == 0) atomicOr(a.err, WI_DEVERR_BAD_ROW);
            rows_left = 0;
            break;
          }
          if (lane == 0 && ok && take > 0)
            ok = pk.push(Ku + (size_t)(o + in) * WI_D, Vu + (size_t)(o + in) * WI_D, take);
          rows_left -= take;
          in = 0;
          used = i + 1;
        }
        // clusters of this batch whose first row lies in this split: four value rows in flight
        for (int i0 = (first_in > 0 ? 1 : 0); i0 < used; i0 += 4) {
          float4 vv[4];
          float ww[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const int i = min(i0 + x, used - 1);
            int j = __shfl_sync(0xffffffffu, rr.w, i);
            j = (j >= 0 && j < a.C) ? j : 0;
            ww[x] = i0 + x < used ? __int_as_float(__shfl_sync(0xffffffffu, rr.z, i)) : 0.f;
            vv[x] = __ldg(vsu + (size_t)j * (WI_D / 4));
          }
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            sub.x = fmaf(ww[x], vv[x].x, sub.x);
            sub.y = fmaf(ww[x], vv[x].y, sub.y);
            sub.z = fmaf(ww[x], vv[x].z, sub.z);
            sub.w = fmaf(ww[x], vv[x].w, sub.w);
          }
        }
        pos += nb;
      }
      reinterpret_cast<float4*>(a.subn + (uh * nsp + split) * WI_PART + 4)[lane] = sub;
    }
    if (lane == 0) {
      if (ok && pk.opened) pk.close();
      if (ok) ok = pk.open();  // the end marker: a stage with no rows
      if (ok) pk.close();
      if (!ok) {
        flags[0] = 1;
        const int issued = pk.stage_it;
        for (int s = 0; s < kD3Stages && s < issued; ++s) {
          const int last = ((issued - 1 - s) / kD3Stages) * kD3Stages + s;
          mbar_wait(&full[s], (last / kD3Stages) & 1, a.err);
        }
      }
      atomicAdd(a.rows_total, (unsigned long long)pk.rows_done);
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
    const int ri = lane >> 2;  // the row (of the warp's 8) whose logit this lane ends with
    for (int it = 0;; ++it) {
      const int s = it % kD3Stages, r = it / kD3Stages;
      if (!mbar_wait(&full[s], r & 1, a.err)) { flags[0] = 1; break; }
      const int nr = nrows[s];
      if (nr == 0) break;
      const int i0 = warp * 8;
      if (i0 < nr) {
        const D3Stage& T = st[s];
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
  }
  // Publish this CTA's partial and take a ticket: the barrier orders the CTA's writes before
  // thread 0's release; the acquire side makes every earlier CTA's partial visible to the last one.
  __syncthreads();
  if (tid == 0) flags[1] = ticket_acq_rel(&a.ticket[uh]) == (unsigned)(nsp - 1);
  __syncthreads();
  if (!flags[1]) return;
  // ---- the last CTA of this head: estimate over all clusters - retrieved terms, plus exact, by LSE.
  // One parallel gather of every partial row into shared memory (the K/V stages are free now),
  // then each output dim sums its column there.  Rows: P estimation partials, nsp exact
  // partials, nsp retrieved value-sum partials, then (m_sub, Z_sub).
  const int kk = flags[2];
  const int nonempty = flags[3];
  const int nrow = a.P + 2 * nsp + 1;
  const float* p1 = a.part1 + uh * a.P * WI_PART;
  const float* p3 = a.part3 + uh * nsp * WI_PART;
  const float* ps = a.subn + uh * nsp * WI_PART;
  const float* sp = a.subpart + uh * WI_PART;
  auto grow = [&](int r) -> const float* {
    return r < a.P ? p1 + (size_t)r * WI_PART
                   : (r < a.P + nsp ? p3 + (size_t)(r - a.P) * WI_PART
                                    : (r < a.P + 2 * nsp ? ps + (size_t)(r - a.P - nsp) * WI_PART : sp));
  };
  float* rows = reinterpret_cast<float*>(d3_raw);
  const int maxrows = (int)(sizeof(D3Stage) * kD3Stages / (WI_PART * sizeof(float)));
  const int nst = nrow < maxrows ? nrow : maxrows;
  for (int i = tid; i < nst * (WI_PART / 4); i += kD3Threads) {
    const int r = i / (WI_PART / 4), c4 = i % (WI_PART / 4);
    reinterpret_cast<float4*>(rows)[i] = __ldcg(reinterpret_cast<const float4*>(grow(r)) + c4);
  }
  __syncthreads();
  auto row = [&](int r) -> const float* { return r < nst ? rows + (size_t)r * WI_PART : grow(r); };
  if (tid < WI_D) {
    const int d = tid;
    float Me = -INFINITY, Mx = -INFINITY;
    for (int c = 0; c < a.P; ++c) Me = fmaxf(Me, row(c)[0]);
    for (int c = 0; c < nsp; ++c) Mx = fmaxf(Mx, row(a.P + c)[0]);
    float Ze = 0.f, Ne = 0.f;
    if (Me > -INFINITY && kk < nonempty) {
      for (int c = 0; c < a.P; ++c) {
        const float* r = row(c);
        const float f = r[0] == -INFINITY ? 0.f : __expf(r[0] - Me);
        Ze = fmaf(f, r[1], Ze);
        Ne = fmaf(f, r[4 + d], Ne);
      }
      const float* r = row(a.P + 2 * nsp);
      if (r[0] > -INFINITY) {
        float nsub = 0.f;
        for (int c = 0; c < nsp; ++c) nsub += row(a.P + nsp + c)[4 + d];
        const float f = __expf(r[0] - Me);
        Ze = fmaf(-f, r[1], Ze);
        Ne = fmaf(-f, nsub, Ne);
      }
      Ze = fmaxf(Ze, 0.f);
    }
    float Zx = 0.f, Nx = 0.f;
    if (Mx > -INFINITY) {
      for (int c = 0; c < nsp; ++c) {
        const float* r = row(a.P + c);
        const float f = r[0] == -INFINITY ? 0.f : __expf(r[0] - Mx);
        Zx = fmaf(f, r[1], Zx);
        Nx = fmaf(f, r[4 + d], Nx);
      }
    }
    const float M = fmaxf(Mx, Me);
    const float fx = Mx > -INFINITY ? __expf(Mx - M) : 0.f;
    const float fe = (Me > -INFINITY && Ze > 0.f) ? __expf(Me - M) : 0.f;
    a.out[uh * WI_D + d] = (Nx * fx + Ne * fe) / (Zx * fx + Ze * fe);
  }
  if (tid == 0) a.ticket[uh] = 0u;  // ready for the next step
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

template <int G, int KPT>
cudaError_t launch_select(const WiGeom& g, const WiDecodeBufs& b, const TopkArgs& t, cudaStream_t st) {
  const size_t sel = sizeof(SelSmem) + (size_t)(g.kmax + 1) * sizeof(int);
  const size_t smem = sel > kEsSmem ? sel : kEsSmem;
  static int smem_set = 0;
  cudaError_t e = wi_ensure_smem(k_select_estimate<G, KPT>, smem, &smem_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_select_estimate<G, KPT>, dim3(g.U * G + g.U * b.p_es), dim3(kSThreads), smem, st, t);
}

template <int G>
cudaError_t launch_g(const WiGeom& g, const WiDecodeBufs& b, const void* qv, float* out, cudaStream_t st,
                     const cudaEvent_t* ev) {
  const bf16* q = static_cast<const bf16*>(qv);
  const float lam = 1.0f / sqrtf((float)WI_D);
  cudaError_t e = mark(ev, 0, st);
  if (e != cudaSuccess) return e;
  // scores (+ first-digit histogram)
  static int smem_sc = 0;
  if ((e = wi_ensure_smem(k_scores<G>, ScCfg<G>::SMEM, &smem_sc)) != cudaSuccess) return e;
  e = launch_pdl(k_scores<G>, dim3(b.p1, g.U), dim3(kScThreads), ScCfg<G>::SMEM, st, b.map_mu, q, b.cnt, b.scores,
                 b.ghist, g.C, b.p1, b.err);
  if (e != cudaSuccess || (e = mark(ev, 1, st)) != cudaSuccess) return e;
  TopkArgs t;
  t.ghist = b.ghist;
  t.scores = b.scores;
  t.cnt = b.cnt;
  t.off = b.off;
  t.nonempty = b.nonempty;
  t.valsum = b.valsum;
  t.sel = b.sel;
  t.selcnt = b.selcnt;
  t.subpart = b.subpart;
  t.runs = b.runs;
  t.splits = b.splits;
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
  const int kpt = (g.C + kSelThreads - 1) / kSelThreads;
  if (kpt <= 16) e = launch_select<G, 16>(g, b, t, st);
  else if (kpt <= 32) e = launch_select<G, 32>(g, b, t, st);
  else if (kpt <= 64) e = launch_select<G, 64>(g, b, t, st);
  else e = launch_select<G, 128>(g, b, t, st);
  if (e != cudaSuccess || (e = mark(ev, 2, st)) != cudaSuccess) return e;
  ExactArgs a;
  a.q = q;
  a.K = static_cast<const bf16*>(b.K);
  a.V = static_cast<const bf16*>(b.V);
  a.appK = static_cast<const bf16*>(b.appK);
  a.appV = static_cast<const bf16*>(b.appV);
  a.app_count = b.app_count;
  a.selcnt = b.selcnt;
  a.runs = b.runs;
  a.splits = b.splits;
  a.valsum = b.valsum;
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
  static int smem3_set = 0;
  if ((e = wi_ensure_smem(k_exact_merge, kD3Smem, &smem3_set)) != cudaSuccess) return e;
  e = launch_pdl(k_exact_merge, dim3(b.nsplit + 1, G, g.U), dim3(kD3Threads), kD3Smem, st, a);
  if (e != cudaSuccess) return e;
  return mark(ev, 3, st);
}

}  // namespace

cudaError_t wi_launch_decode(const WiGeom& g, const WiDecodeBufs& b, const void* q, float* out, cudaStream_t st,
                             const cudaEvent_t* ev) {
  switch (g.G) {
    case 1: return launch_g<1>(g, b, q, out, st, ev);
    case 2: return launch_g<2>(g, b, q, out, st, ev);
    case 3: return launch_g<3>(g, b, q, out, st, ev);
    case 4: return launch_g<4>(g, b, q, out, st, ev);
    case 5: return launch_g<5>(g, b, q, out, st, ev);
    case 6: return launch_g<6>(g, b, q, out, st, ev);
    case 7: return launch_g<7>(g, b, q, out, st, ev);
    case 8: return launch_g<8>(g, b, q, out, st, ev);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t wi_launch_append(const WiGeom& g, const WiDecodeBufs& b, const void* k_new, const void* v_new, int t,
                             cudaStream_t st) {
  k_append<<<g.U, 32, 0, st>>>(static_cast<const bf16*>(k_new), static_cast<const bf16*>(v_new),
                               static_cast<bf16*>(b.appK), static_cast<bf16*>(b.appV), b.app_count, t,
                               g.max_append);
  return cudaGetLastError();
}
