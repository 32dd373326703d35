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

namespace {

// ------------------------------------------------------- score_estimate ----
constexpr int kD1Warps = 16;            // consumer warps; one more warp issues the copies
constexpr int kD1Tile = 8 * kD1Warps;   // clusters per stage (8 per consumer warp)
constexpr int kD1Stages = 2;
constexpr int kD1Threads = 32 * (kD1Warps + 1);

struct D1Stage {
  bf16 mu[kD1Tile * WI_D];
  float vs[kD1Tile * WI_D];
  int cnt[kD1Tile];
};

constexpr size_t kD1Smem = sizeof(D1Stage) * kD1Stages + 2 * kD1Stages * sizeof(uint64_t) +
                           sizeof(float) * kD1Warps * 2 * 32 + sizeof(float) * kD1Warps * 2 * 4 + 16;

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

template <int G>
__global__ void __launch_bounds__(kD1Threads, 1) k_score_estimate(
    const bf16* __restrict__ q, const bf16* __restrict__ mu, const float* __restrict__ valsum,
    const int* __restrict__ cnt, float* __restrict__ scores, float* __restrict__ part, int C, int P, float lam,
    int* err) {
  using HG = HeadGeo<G>;
  extern __shared__ __align__(128) unsigned char d1_raw[];
  D1Stage* st = reinterpret_cast<D1Stage*>(d1_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(d1_raw + sizeof(D1Stage) * kD1Stages);
  uint64_t* empty = full + kD1Stages;
  float* pbuf = reinterpret_cast<float*>(empty + kD1Stages);  // [warps][2][32]
  float* sbuf = pbuf + kD1Warps * 2 * 32;                      // [warps][2][4]
  int* s_abort = reinterpret_cast<int*>(sbuf + kD1Warps * 2 * 4);
  const int u = blockIdx.y, p = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // clusters [c0, c1) of the unit, split evenly across the P CTAs (boundaries on multiples of 16 so
  // that every bulk copy stays 16-byte aligned); tiles of kD1Tile clusters, the last one partial
  const int c0 = (int)(((long long)C * p / P) & ~15LL);
  const int c1 = p + 1 == P ? C : (int)(((long long)C * (p + 1) / P) & ~15LL);
  const int ntile = (c1 - c0 + kD1Tile - 1) / kD1Tile;
  pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < kD1Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kD1Warps);
    }
    *s_abort = 0;
  }
  __syncthreads();
  // The producer streams the index (written only by build / import, which have
  // completed) while the previous kernel may still run; everything else waits.
  // consumer state (lane l: the head it ends each reduction with; dims 4l..4l+3)
  float m_l[HG::HB], z_l[HG::HB], N[G][4];
#pragma unroll
  for (int b = 0; b < HG::HB; ++b) { m_l[b] = -INFINITY; z_l[b] = 0.f; }
#pragma unroll
  for (int h = 0; h < G; ++h) N[h][0] = N[h][1] = N[h][2] = N[h][3] = 0.f;
  const int ci = lane >> 2;
  const int hl = (lane & 3) >> HG::SHIFT;
  const bool rep = (lane & ((1 << HG::SHIFT) - 1)) == 0;  // one writer per (cluster, head)
  if (warp == kD1Warps) {
    // ---- producer: one lane issues the bulk copies of each tile
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      for (int it = 0; it < ntile; ++it) {
        const int s = it % kD1Stages, r = it / kD1Stages;
        if (r > 0 && !mbar_wait(&empty[s], (r - 1) & 1, err)) { ok = false; break; }
        const int j0 = c0 + it * kD1Tile, nj = min(kD1Tile, c1 - j0);
        mbar_arrive_expect_tx(&full[s], (uint32_t)nj * (WI_D * 2 + WI_D * 4 + 4));
        const size_t row = (size_t)u * C + j0;
        bulk_g2s(st[s].mu, mu + row * WI_D, nj * WI_D * 2, &full[s]);
        bulk_g2s(st[s].vs, valsum + row * WI_D, nj * WI_D * 4, &full[s]);
        bulk_g2s(st[s].cnt, cnt + row, nj * 4, &full[s]);
        issued = it + 1;
      }
      if (!ok) {  // never leave with copies in flight: wait for the last round of every stage
        *s_abort = 1;
        for (int s = 0; s < kD1Stages && s < issued; ++s) {
          const int last = ((issued - 1 - s) / kD1Stages) * kD1Stages + s;
          mbar_wait(&full[s], (last / kD1Stages) & 1, err);
        }
      }
    }
  } else {
    // ---- consumers: warp w owns clusters [8w, 8w+8) of every tile
    pdl_wait();
    float qr[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) load_bf16x4(q + ((size_t)u * G + h) * WI_D + 4 * lane, qr[h]);
    // head pairs (h, h+1) as float2 for the packed FMA; an odd last head pairs with zeros
    constexpr int GPAIR = (G + 1) / 2;
    float2 qp[GPAIR][4];
#pragma unroll
    for (int hp = 0; hp < GPAIR; ++hp)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        qp[hp][e] = make_float2(qr[2 * hp][e], 2 * hp + 1 < G ? qr[(2 * hp + 1) < G ? 2 * hp + 1 : 0][e] : 0.f);
    float* pb = pbuf + warp * 2 * 32;
    float* sb = sbuf + warp * 2 * 4;
    for (int it = 0; it < ntile; ++it) {
      const int s = it % kD1Stages, r = it / kD1Stages;
      if (!mbar_wait(&full[s], r & 1, err)) { *s_abort = 1; break; }
      const D1Stage& T = st[s];
      const int j0 = c0 + it * kD1Tile, nj = min(kD1Tile, c1 - j0);
      const int i0 = warp * 8;
      if (i0 < nj) {
        float x[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          unpack_bf16x4(*reinterpret_cast<const uint2*>(&T.mu[(i0 + i) * WI_D + 4 * lane]), x[i]);
          if (i0 + i >= nj) x[i][0] = x[i][1] = x[i][2] = x[i][3] = 0.f;  // stale rows past the tile
        }
        const bool valid_c = (i0 + ci) < nj;
        const int cn = valid_c ? T.cnt[i0 + ci] : 0;
#pragma unroll
        for (int b = 0; b < HG::HB; ++b) {
          float v[HG::NV];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if constexpr (HG::GP == 1) {
              // one head: pair up dims instead
              float2 acc = __fmul2_rn(make_float2(qr[0][0], qr[0][1]), make_float2(x[i][0], x[i][1]));
              acc = __ffma2_rn(make_float2(qr[0][2], qr[0][3]), make_float2(x[i][2], x[i][3]), acc);
              v[i] = acc.x + acc.y;
            } else {
#pragma unroll
              for (int h = 0; h < HG::GP; h += 2) {
                const int hp = (b * 4 + h) / 2;
                const int hq = hp < GPAIR ? hp : 0;
                float2 acc = __fmul2_rn(qp[hq][0], make_float2(x[i][0], x[i][0]));
                acc = __ffma2_rn(qp[hq][1], make_float2(x[i][1], x[i][1]), acc);
                acc = __ffma2_rn(qp[hq][2], make_float2(x[i][2], x[i][2]), acc);
                acc = __ffma2_rn(qp[hq][3], make_float2(x[i][3], x[i][3]), acc);
                v[i * HG::GP + h] = (b * 4 + h) < G ? acc.x : 0.f;
                v[i * HG::GP + h + 1] = (b * 4 + h + 1) < G ? acc.y : 0.f;
              }
            }
          }
          const float sdot = transpose_reduce<HG::NV>(v);
          const int head = b * 4 + hl;
          const bool valid = valid_c && head < G;
          if (valid && rep) scores[((size_t)u * G + head) * C + j0 + i0 + ci] = sdot;
          const float se = (valid && cn > 0) ? lam * sdot : -INFINITY;
          float mx = fmaxf(se, __shfl_xor_sync(0xffffffffu, se, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float m_new = fmaxf(m_l[b], mx);
          const float sc = m_new == -INFINITY ? 1.f : __expf(m_l[b] - m_new);
          const float pr = se == -INFINITY ? 0.f : __expf(se - m_new);
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
        // N_h = N_h * sc_h + sum_i p_ih valsum_i
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float sc = sb[(h >> 2) * 4 + (h & 3)];
          const float2 s2 = make_float2(sc, sc);
          float2 lo = __fmul2_rn(make_float2(N[h][0], N[h][1]), s2);
          float2 hi = __fmul2_rn(make_float2(N[h][2], N[h][3]), s2);
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
  pdl_wait();
  __syncthreads();
  if (*s_abort) return;
  float* red = reinterpret_cast<float*>(d1_raw);  // [warps][G][WI_PART]; the stages are free now
  if (warp < kD1Warps) {
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
  for (int i = tid; i < G * WI_D; i += kD1Threads) {
    const int h = i / WI_D, d = i % WI_D;
    float M = -INFINITY;
    for (int w = 0; w < kD1Warps; ++w) M = fmaxf(M, red[((size_t)w * G + h) * WI_PART]);
    float z = 0.f, acc = 0.f;
    if (M > -INFINITY) {
      for (int w = 0; w < kD1Warps; ++w) {
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

// ------------------------------------------------------------- topk_sub ----
// CTA = (head, unit), 1024 threads, KPT consecutive clusters per thread held
// as order-preserving keys in registers (0 = empty cluster / padding).
// Three radix passes (11, 11, 10 bits) find the k-th largest key T; keys > T
// and the first (in id order) keys == T are written in id order.  For the
// exact-attention kernel it also writes each selected cluster's row run
// (first row, rows) and the starts of NS row-balanced splits of the selected
// rows.  Finally the estimation terms of the selected clusters, relative to
// m_sub = lam * s_max: Z_sub = sum n_j exp(lam s_j - m_sub),
// N_sub = sum exp(lam s_j - m_sub) valsum_j.
constexpr int kTopkThreads = 1024;

// Inverse of float_key for finite scores.
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

struct TopkArgs {
  const float* scores;
  const int* cnt;
  const int* off;
  const int* nonempty;
  const float* valsum;
  int* sel;
  int* selcnt;
  float* subpart;
  int2* runs;    // [U][G][kmax]  (first row, rows)
  int4* splits;  // [U][G][NS+1]  (position, row inside that cluster, split's first row, 0)
  int* err;
  int G, C, kmax, NS;
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

// Exclusive block-wide prefix of a 64-bit count per thread, with one barrier:
// warp totals go through `wt` (32 entries); returns the prefix, sets *total.
__device__ __forceinline__ unsigned long long block_prefix_u64(unsigned long long v, unsigned long long* wt,
                                                               unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned long long inc = warp_scan_u64(v);
  if (lane == 31) wt[warp] = inc;
  __syncthreads();
  const unsigned long long x = wt[lane];
  unsigned long long before = lane < warp ? x : 0ull, all = x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    all += __shfl_xor_sync(0xffffffffu, all, o);
  }
  *total = all;
  return before + inc - v;
}

template <int KPT>
__global__ void __launch_bounds__(kTopkThreads) k_topk_sub(TopkArgs a) {
  static_assert(kTopkThreads == 1024, "the scans below assume 32 warps");
  __shared__ int hist[2][2048];
  __shared__ int s_wsum[32];
  __shared__ int s_bin, s_above;
  __shared__ uint32_t s_maxkey;
  __shared__ unsigned long long s_wt[2][32];
  __shared__ __align__(16) float red[32][WI_D];
  __shared__ float zred[32];
  extern __shared__ __align__(16) unsigned char tk_dyn[];
  int* s_id = reinterpret_cast<int*>(tk_dyn);            // [kmax]
  float* s_w = reinterpret_cast<float*>(s_id + a.kmax);  // [kmax]
  int* s_row = reinterpret_cast<int*>(s_w + a.kmax);     // [kmax + 1] row prefix in selection order
  pdl_trigger();
  const int h = blockIdx.x, u = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 2048; i += kTopkThreads) hist[0][i] = 0;
  if (tid == 0) s_maxkey = 0u;
  pdl_wait();
  const size_t uh = (size_t)u * a.G + h;
  const int C = a.C;
  const float* s = a.scores + uh * C;
  const int* cn = a.cnt + (size_t)u * C;
  int* out = a.sel + uh * a.kmax;
  const int kk = min(a.kmax, a.nonempty[u]);
  uint32_t key[KPT];
  int nc[KPT];
  const int base = tid * KPT;
  if (base + KPT <= C) {  // vector loads, all issued before use
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
#pragma unroll
  for (int e = 0; e < KPT; ++e)
    if (nc[e] <= 0) key[e] = 0u;  // empty clusters are never candidates
  for (int i = tid; i < a.kmax; i += kTopkThreads) out[i] = -1;
  if (tid == 0) a.selcnt[uh] = kk;
  __syncthreads();
  // ---- radix select: three passes, three barriers each (the next pass's histogram is cleared meanwhile)
  uint32_t prefix = 0, pmask = 0;
  int remaining = kk;
#pragma unroll 1
  for (int pass = 0; pass < 3 && kk > 0; ++pass) {
    const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    int* hc = hist[pass & 1];
    int* hn = hist[(pass + 1) & 1];
#pragma unroll
    for (int e = 0; e < KPT; ++e)
      if (key[e] != 0u && (key[e] & pmask) == prefix) atomicAdd(&hc[(key[e] >> sh) & (nb - 1)], 1);
    __syncthreads();
    // warp w owns reversed bins [64w, 64w+64) (bin = nb-1-rb), lane l the pair 2l, 2l+1
    const int rb0 = 64 * warp + 2 * lane;
    const int b0 = rb0 < nb ? hc[nb - 1 - rb0] : 0;
    const int b1 = rb0 + 1 < nb ? hc[nb - 2 - rb0] : 0;
    const int inc = warp_inclusive_scan(b0 + b1);
    if (lane == 31) s_wsum[warp] = inc;
    for (int i = tid; i < 2048; i += kTopkThreads) hn[i] = 0;
    __syncthreads();
    int ws = s_wsum[lane];
    int wincl = warp_inclusive_scan(ws);
    const unsigned hit = __ballot_sync(0xffffffffu, wincl >= remaining);
    const int wstar = __ffs(hit) - 1;  // warp whose range holds the remaining-th largest key
    if (warp == wstar) {
      const int before = __shfl_sync(0xffffffffu, wincl - ws, wstar);
      const int ex = before + inc - (b0 + b1);
      if (ex < remaining && remaining <= ex + b0) { s_bin = nb - 1 - rb0; s_above = ex; }
      else if (ex + b0 < remaining && remaining <= ex + b0 + b1) { s_bin = nb - 2 - rb0; s_above = ex + b0; }
    }
    __syncthreads();
    remaining -= s_above;
    prefix |= (uint32_t)s_bin << sh;
    pmask |= (uint32_t)(nb - 1) << sh;
  }
  const uint32_t T = kk > 0 ? prefix : 0xffffffffu;  // nothing is taken when kk == 0
  // ---- compaction in id order: counts of keys > T and == T, and the rows they bring
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
  if (lane == 0) atomicMax(&s_maxkey, kmx);
  unsigned long long tot;
  const unsigned long long pre = block_prefix_u64(((unsigned long long)cgt << 32) | (unsigned)ceq, s_wt[0], &tot);
  const int pre_gt = (int)(pre >> 32), pre_eq = (int)(pre & 0xffffffffu);
  const int tot_gt = (int)(tot >> 32), tot_eq = (int)(tot & 0xffffffffu);
  const float m_sub = kk > 0 ? a.lam * key_float(s_maxkey) : -INFINITY;
  // which of my keys are taken, and their rows
  int eq_seen = pre_eq, my_rows = 0;
  uint32_t takemask = 0u;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    const bool is_eq = key[e] != 0u && key[e] == T;
    const bool take = key[e] > T || (is_eq && eq_seen < remaining);
    eq_seen += is_eq ? 1 : 0;
    if (take) { takemask |= 1u << e; my_rows += nc[e]; }
  }
  unsigned long long rtot;
  const int row_pre = (int)block_prefix_u64((unsigned long long)my_rows, s_wt[1], &rtot);
  int pos = pre_gt + min(pre_eq, remaining);
  int rp = row_pre;
  float zpart = 0.f;
  const int* offu = a.off + (size_t)u * (C + 1);
  int2* runs = a.runs + uh * a.kmax;
#pragma unroll
  for (int e = 0; e < KPT; ++e) {
    if (takemask & (1u << e)) {
      if (pos < kk) {
        const int j = base + e;
        const float w = __expf(a.lam * key_float(key[e]) - m_sub);
        out[pos] = j;
        s_id[pos] = j;
        s_w[pos] = w;
        s_row[pos] = rp;
        runs[pos] = make_int2(__ldg(offu + j), nc[e]);
        zpart = fmaf((float)nc[e], w, zpart);
      }
      rp += nc[e];
      ++pos;
    }
  }
  if (tid == 0) {
    s_row[kk] = (int)rtot;
    if (tot_gt + min(tot_eq, remaining) != kk) atomicOr(a.err, WI_DEVERR_TOPK);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) zpart += __shfl_xor_sync(0xffffffffu, zpart, o);
  if (lane == 0) zred[warp] = zpart;
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
  // N_sub: warp w sums selected clusters w, w+32, ...; four value rows in flight per lane
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* vsu = reinterpret_cast<const float4*>(a.valsum + (size_t)u * C * WI_D) + lane;
  for (int i = warp; i < kk; i += 4 * 32) {
    float4 vv[4];
    float ww[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int ii = i + x * 32;
      ww[x] = 0.f;
      vv[x] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ii < kk) {
        ww[x] = s_w[ii];
        vv[x] = __ldg(vsu + (size_t)s_id[ii] * (WI_D / 4));
      }
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      acc.x = fmaf(ww[x], vv[x].x, acc.x);
      acc.y = fmaf(ww[x], vv[x].y, acc.y);
      acc.z = fmaf(ww[x], vv[x].z, acc.z);
      acc.w = fmaf(ww[x], vv[x].w, acc.w);
    }
  }
  *reinterpret_cast<float4*>(&red[warp][4 * lane]) = acc;
  __syncthreads();
  float* sp = a.subpart + uh * WI_PART;
  if (tid < WI_D) {
    float acc2 = 0.f;
    for (int w = 0; w < 32; ++w) acc2 += red[w][tid];
    sp[4 + tid] = acc2;
  }
  if (tid == 0) {
    float zz = 0.f;
    for (int w = 0; w < 32; ++w) zz += zred[w];
    sp[0] = m_sub;
    sp[1] = zz;
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
  const int2* runs;
  const int4* splits;
  const int* nonempty;
  const float* part1;    // [U][G][P]
  const float* subpart;  // [U][G]
  float* part3;          // [U][G][NS+1]
  unsigned int* ticket;  // [U][G]
  unsigned long long* rows_total;
  float* out;
  int* err;
  long long n;
  int G, kmax, P, NS, n_sink, W, max_append;
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
  int* flags = reinterpret_cast<int*>(red + kD3Warps * WI_PART);  // [0] abort, [1] last CTA
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
      if (lane == 0) {
        const int amax = a.max_append > 0 ? a.max_append : 1;
        ok = ok && pk.push(a.appK + (size_t)u * amax * WI_D, a.appV + (size_t)u * amax * WI_D, *a.app_count);
      }
    } else {
      // ---- selected clusters: rows [b_s, b_{s+1}) of the head's row-balanced split
      pdl_wait();
      const int4 sa = a.splits[uh * nsp + split];
      const int4 sb = a.splits[uh * nsp + split + 1];
      const int kk = a.selcnt[uh];
      int rows_left = sb.z - sa.z;
      int pos = sa.x, in = sa.y;
      const int2* runs = a.runs + uh * a.kmax;
      while (rows_left > 0 && pos < kk) {
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
        const int2 rr = (pos + lane < kk) ? runs[pos + lane] : make_int2(0, 0);
        const int nb = min(32, kk - pos);
        for (int i = 0; i < nb && rows_left > 0; ++i) {
          const int o = __shfl_sync(0xffffffffu, rr.x, i);
          const int z = __shfl_sync(0xffffffffu, rr.y, i);
          const int take = min(z - in, rows_left);
          if (lane == 0 && ok && take > 0)
            ok = pk.push(Ku + (size_t)(o + in) * WI_D, Vu + (size_t)(o + in) * WI_D, take);
          rows_left -= take;
          in = 0;
        }
        pos += nb;
      }
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
  __threadfence();
  __syncthreads();
  if (tid == 0) flags[1] = atomicAdd(&a.ticket[uh], 1u) == (unsigned)(nsp - 1);
  __syncthreads();
  if (!flags[1]) return;
  __threadfence();
  // ---- the last CTA of this head: estimate over all clusters - retrieved terms, plus exact, by LSE.
  // Partial maxima and sums are gathered in parallel first (one thread per partial), then every
  // output dim sums its column with independent loads.
  const int kk = a.selcnt[uh];
  float* pm = red;                  // [P + nsp] maxima (reuses red)
  float* pz = red + (a.P + nsp);    // matching sums
  const float* p1 = a.part1 + uh * a.P * WI_PART;
  const float* p3 = a.part3 + uh * nsp * WI_PART;
  for (int c = tid; c < a.P + nsp; c += kD3Threads) {
    const float* src = c < a.P ? p1 + (size_t)c * WI_PART : p3 + (size_t)(c - a.P) * WI_PART;
    pm[c] = __ldcg(src);
    pz[c] = __ldcg(src + 1);
  }
  __syncthreads();
  if (tid < WI_D) {
    const int d = tid;
    float Me = -INFINITY, Mx = -INFINITY;
    for (int c = 0; c < a.P; ++c) Me = fmaxf(Me, pm[c]);
    for (int c = 0; c < nsp; ++c) Mx = fmaxf(Mx, pm[a.P + c]);
    float Ze = 0.f, Ne = 0.f;
    if (Me > -INFINITY && kk < a.nonempty[u]) {
#pragma unroll 8
      for (int c = 0; c < a.P; ++c) {
        const float f = pm[c] == -INFINITY ? 0.f : __expf(pm[c] - Me);
        Ze = fmaf(f, pz[c], Ze);
        Ne = fmaf(f, __ldcg(p1 + (size_t)c * WI_PART + 4 + d), Ne);
      }
      const float* sp = a.subpart + uh * WI_PART;
      const float ms = __ldcg(sp);
      if (ms > -INFINITY) {
        const float f = __expf(ms - Me);
        Ze = fmaf(-f, __ldcg(sp + 1), Ze);
        Ne = fmaf(-f, __ldcg(sp + 4 + d), Ne);
      }
      Ze = fmaxf(Ze, 0.f);
    }
    float Zx = 0.f, Nx = 0.f;
    if (Mx > -INFINITY) {
#pragma unroll 8
      for (int c = 0; c < nsp; ++c) {
        const float mc = pm[a.P + c];
        const float f = mc == -INFINITY ? 0.f : __expf(mc - Mx);
        Zx = fmaf(f, pz[a.P + c], Zx);
        Nx = fmaf(f, __ldcg(p3 + (size_t)c * WI_PART + 4 + d), Nx);
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

template <int KPT>
cudaError_t launch_topk(const WiGeom& g, const TopkArgs& t, cudaStream_t st) {
  const size_t smem = (size_t)(3 * g.kmax + 1) * sizeof(int);
  static int smem_set = 0;
  cudaError_t e = wi_ensure_smem(k_topk_sub<KPT>, smem, &smem_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_topk_sub<KPT>, dim3(g.G, g.U), dim3(kTopkThreads), smem, st, t);
}

template <int G>
cudaError_t launch_g(const WiGeom& g, const WiDecodeBufs& b, const void* qv, float* out, cudaStream_t st,
                     const cudaEvent_t* ev) {
  const bf16* q = static_cast<const bf16*>(qv);
  const float lam = 1.0f / sqrtf((float)WI_D);
  cudaError_t e = mark(ev, 0, st);
  if (e != cudaSuccess) return e;
  static int smem1_set = 0;
  if ((e = wi_ensure_smem(k_score_estimate<G>, kD1Smem, &smem1_set)) != cudaSuccess) return e;
  e = launch_pdl(k_score_estimate<G>, dim3(b.p1, g.U), dim3(kD1Threads), kD1Smem, st, q,
                 static_cast<const bf16*>(b.mu), b.valsum, b.cnt, b.scores, b.part1, g.C, b.p1, lam, b.err);
  if (e != cudaSuccess || (e = mark(ev, 1, st)) != cudaSuccess) return e;
  TopkArgs t;
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
  t.err = b.err;
  t.G = G;
  t.C = g.C;
  t.kmax = g.kmax;
  t.NS = b.nsplit;
  t.lam = lam;
  const int kpt = (g.C + kTopkThreads - 1) / kTopkThreads;
  if (kpt <= 8) e = launch_topk<8>(g, t, st);
  else if (kpt <= 16) e = launch_topk<16>(g, t, st);
  else if (kpt <= 32) e = launch_topk<32>(g, t, st);
  else e = launch_topk<64>(g, t, st);
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
  a.P = b.p1;
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
