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
// Kernel chain per step (all units of the batch in each launch):
//   D1 score_estimate  s_hj = q_h . mu_j for every cluster (written out) and,
//                      fused in the same pass over mu / valsum, the
//                      estimation partials (m, Z, N) per cluster chunk;
//   D2 topk            radix select of the k best non-empty clusters per head,
//                      ties to the lowest id, ids ascending;
//   D2b union          union of the group's selections: the exact rows of the
//                      unit (steady rows, then the clusters' contiguous rows),
//                      each tagged with the mask of heads that attend to it;
//   D3 exact           split-K flash-decode over those rows: (m, Z, N) per
//                      head per split;
//   D4+D5 merge        remove the retrieved clusters' terms from the
//                      estimate, merge estimate and exact partials by LSE.
#include <cuda_runtime.h>

#include "wi_common.cuh"
#include "wi_internal.h"

namespace {

constexpr int kD1Threads = 256;
constexpr int kD3Threads = 256;
constexpr int kTopkThreads = 1024;
constexpr int kUnionThreads = 512;

template <int G>
__device__ __forceinline__ void load_q(const bf16* q, int u, int lane, float (&qr)[G][4]) {
#pragma unroll
  for (int h = 0; h < G; ++h) load_bf16x4(q + ((size_t)u * G + h) * WI_D + 4 * lane, qr[h]);
}

// ---------------------------------------------------------------- D1 ----
// CTA = (cluster chunk, unit).  Phase A: warp-per-cluster dot products with
// the G query heads (lane l holds dims 4l..4l+3).  Phase B: with the chunk's
// per-head max m_h, Z_h = sum n_j exp(lam s_hj - m_h) and
// N_h = sum exp(lam s_hj - m_h) valsum_j over non-empty j.
template <int G>
__global__ void __launch_bounds__(kD1Threads) k_d1_score_estimate(
    const bf16* __restrict__ q, const bf16* __restrict__ mu, const float* __restrict__ valsum,
    const int* __restrict__ cnt, float* __restrict__ scores, float* __restrict__ part, int C, int CH, int nchunk,
    float lam) {
  extern __shared__ __align__(16) float d1s[];
  float* sc = d1s;                 // [G][CH], lam * s or -inf for empty clusters
  float* red = d1s + G * CH;       // [8][G][WI_PART]
  const int u = blockIdx.y, c = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NW = kD1Threads / 32;
  const int j0 = c * CH;
  const int nj = min(CH, C - j0);
  float qr[G][4];
  load_q<G>(q, u, lane, qr);
  const bf16* mub = mu + ((size_t)u * C + j0) * WI_D + 4 * lane;
  const int* cb = cnt + (size_t)u * C + j0;
  // phase A: four clusters per warp in flight
  for (int jj = warp; jj < nj; jj += 4 * NW) {
    uint2 w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (jj + i * NW < nj) w[i] = ldg_u2(mub + (size_t)(jj + i * NW) * WI_D);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int jx = jj + i * NW;
      if (jx >= nj) break;
      float x[4];
      unpack_bf16x4(w[i], x);
      const int cn = __ldg(cb + jx);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float dsum = qr[h][0] * x[0];
        dsum = fmaf(qr[h][1], x[1], dsum);
        dsum = fmaf(qr[h][2], x[2], dsum);
        dsum = fmaf(qr[h][3], x[3], dsum);
        dsum = warp_sum(dsum);
        if (lane == 0) {
          scores[((size_t)u * G + h) * C + j0 + jx] = dsum;
          sc[h * CH + jx] = cn > 0 ? lam * dsum : -INFINITY;
        }
      }
    }
  }
  __syncthreads();
  float mh[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float v = -INFINITY;
    for (int jj = lane; jj < nj; jj += 32) v = fmaxf(v, sc[h * CH + jj]);
    mh[h] = warp_max(v);
  }
  float Z[G], N[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    Z[h] = 0.f;
    N[h][0] = N[h][1] = N[h][2] = N[h][3] = 0.f;
  }
  const float* vb = valsum + ((size_t)u * C + j0) * WI_D + 4 * lane;
  for (int jj = warp; jj < nj; jj += 4 * NW) {
    float4 vv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (jj + i * NW < nj) vv[i] = __ldg(reinterpret_cast<const float4*>(vb + (size_t)(jj + i * NW) * WI_D));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int jx = jj + i * NW;
      if (jx >= nj) break;
      const float cn = (float)__ldg(cb + jx);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float sv = sc[h * CH + jx];
        const float p = sv == -INFINITY ? 0.f : __expf(sv - mh[h]);
        Z[h] = fmaf(cn, p, Z[h]);
        N[h][0] = fmaf(p, vv[i].x, N[h][0]);
        N[h][1] = fmaf(p, vv[i].y, N[h][1]);
        N[h][2] = fmaf(p, vv[i].z, N[h][2]);
        N[h][3] = fmaf(p, vv[i].w, N[h][3]);
      }
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float* r = red + ((size_t)warp * G + h) * WI_PART;
    if (lane == 0) r[1] = Z[h];
    *reinterpret_cast<float4*>(r + 4 + 4 * lane) = make_float4(N[h][0], N[h][1], N[h][2], N[h][3]);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * (WI_D + 2); i += kD1Threads) {
    const int h = i / (WI_D + 2), e = i % (WI_D + 2);
    float* o = part + (((size_t)u * G + h) * nchunk + c) * WI_PART;
    if (e == 0) {
      // every warp computed the same mh; recompute from shared scores
      float v = -INFINITY;
      for (int jj = 0; jj < nj; ++jj) v = fmaxf(v, sc[h * CH + jj]);
      o[0] = v;
    } else if (e == 1) {
      float z = 0.f;
      for (int w = 0; w < NW; ++w) z += red[((size_t)w * G + h) * WI_PART + 1];
      o[1] = z;
    } else {
      const int dd = e - 2;
      float a = 0.f;
      for (int w = 0; w < NW; ++w) a += red[((size_t)w * G + h) * WI_PART + 4 + dd];
      o[4 + dd] = a;
    }
  }
}

// ---------------------------------------------------------------- D2 ----
// Radix select per (head, unit): three passes (11, 11, 10 bits) over the
// order-preserving keys of the scores find the k-th largest key T; then the
// keys > T and the first (in id order) keys == T are compacted in id order.
__global__ void __launch_bounds__(kTopkThreads) k_d2_topk(const float* __restrict__ scores,
                                                         const int* __restrict__ cnt,
                                                         const int* __restrict__ nonempty, int* __restrict__ sel,
                                                         int* __restrict__ selcnt, int G, int C, int kmax,
                                                         int* err) {
  __shared__ int hist[2048];
  __shared__ int tmp[32];
  __shared__ int s_bin, s_above;
  const int h = blockIdx.x, u = blockIdx.y, tid = threadIdx.x;
  const size_t uh = (size_t)u * G + h;
  const float* s = scores + uh * C;
  const int* cn = cnt + (size_t)u * C;
  int* out = sel + uh * kmax;
  const int kk = min(kmax, nonempty[u]);
  for (int i = tid; i < kmax; i += kTopkThreads) out[i] = -1;
  if (tid == 0) selcnt[uh] = kk;
  if (kk <= 0) return;
  uint32_t prefix = 0, pmask = 0;
  int remaining = kk;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = shifts[pass], nb = 1 << widths[pass];
    for (int i = tid; i < 2048; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int j = tid; j < C; j += kTopkThreads) {
      const uint32_t key = __ldg(cn + j) > 0 ? float_key(__ldg(s + j)) : 0u;
      if (key != 0u && (key & pmask) == prefix) atomicAdd(&hist[(key >> sh) & (nb - 1)], 1);
    }
    __syncthreads();
    // suffix counts from the top bin down: thread t owns reversed bins 2t, 2t+1
    const int r0 = 2 * tid, r1 = 2 * tid + 1;
    const int c0 = r0 < nb ? hist[nb - 1 - r0] : 0;
    const int c1 = r1 < nb ? hist[nb - 1 - r1] : 0;
    int tot;
    const int ex = block_exclusive_scan(c0 + c1, tmp, &tot);
    // the bin holding the remaining-th largest key: count above < remaining <= count above + bin
    if (r0 < nb && ex < remaining && remaining <= ex + c0) { s_bin = nb - 1 - r0; s_above = ex; }
    if (r1 < nb && ex + c0 < remaining && remaining <= ex + c0 + c1) { s_bin = nb - 1 - r1; s_above = ex + c0; }
    __syncthreads();
    const int bin = s_bin, above = s_above;
    __syncthreads();
    remaining -= above;
    prefix |= (uint32_t)bin << sh;
    pmask |= (uint32_t)(nb - 1) << sh;
  }
  const uint32_t T = prefix;  // the k-th largest key; take `remaining` keys equal to T
  const int need_eq = remaining;
  int base_out = 0, base_eq = 0;
  for (int j0 = 0; j0 < C; j0 += kTopkThreads) {
    const int j = j0 + tid;
    uint32_t key = 0u;
    if (j < C) key = __ldg(cn + j) > 0 ? float_key(__ldg(s + j)) : 0u;
    const int is_eq = (key != 0u && key == T) ? 1 : 0;
    int tot_eq;
    const int eq_rank = base_eq + block_exclusive_scan(is_eq, tmp, &tot_eq);
    const int take = (key > T) || (is_eq && eq_rank < need_eq) ? 1 : 0;
    int tot_take;
    const int pos = base_out + block_exclusive_scan(take, tmp, &tot_take);
    if (take) {
      if (pos < kk) out[pos] = j;
      else atomicOr(err, WI_DEVERR_TOPK);
    }
    base_out += tot_take;
    base_eq += tot_eq;
  }
  if (tid == 0 && base_out != kk) atomicOr(err, WI_DEVERR_TOPK);
}

// --------------------------------------------------------------- D2b ----
// Union of the group's selections as the unit's exact row list.  Row entry =
// (row << 8) | head mask; rows >= n address the append buffer (row - n).
// Order: sinks, local window, appended tokens, then the union's clusters in
// ascending id, each cluster's rows contiguous.
__global__ void __launch_bounds__(kUnionThreads) k_d2_union(const int* __restrict__ sel,
                                                           const int* __restrict__ selcnt,
                                                           const int* __restrict__ cnt, const int* __restrict__ off,
                                                           const int* __restrict__ app_count,
                                                           uint32_t* __restrict__ rows, int* __restrict__ rcount,
                                                           unsigned long long* __restrict__ rows_total, int G, int C,
                                                           int kmax, long long n, int n_sink, int W,
                                                           long long rows_cap, int* err) {
  extern __shared__ __align__(16) uint32_t us[];
  const int words = (C + 31) / 32;
  uint32_t* bm = us;                               // [G][words]
  int* ent_id = reinterpret_cast<int*>(bm + (size_t)G * words);   // [G * kmax]
  uint32_t* ent_mask = reinterpret_cast<uint32_t*>(ent_id + (size_t)G * kmax);  // [G * kmax]
  int* ent_row = reinterpret_cast<int*>(ent_mask + (size_t)G * kmax);           // [G * kmax + 1]
  __shared__ int tmp[32];
  const int u = blockIdx.x, tid = threadIdx.x;
  const uint32_t all = (1u << G) - 1u;
  for (int i = tid; i < G * words; i += kUnionThreads) bm[i] = 0u;
  __syncthreads();
  for (int h = 0; h < G; ++h) {
    const int m = selcnt[(size_t)u * G + h];
    const int* sh = sel + ((size_t)u * G + h) * kmax;
    for (int i = tid; i < m; i += kUnionThreads) {
      const int id = sh[i];
      if (id >= 0 && id < C) atomicOr(&bm[(size_t)h * words + (id >> 5)], 1u << (id & 31));
      else atomicOr(err, WI_DEVERR_BAD_CLUSTER);
    }
  }
  __syncthreads();
  // entries in id order: each thread owns a contiguous run of words
  const int per = (words + kUnionThreads - 1) / kUnionThreads;
  const int w0 = min(words, tid * per), w1 = min(words, w0 + per);
  int mine = 0;
  for (int w = w0; w < w1; ++w) {
    uint32_t o = 0u;
    for (int h = 0; h < G; ++h) o |= bm[(size_t)h * words + w];
    mine += __popc(o);
  }
  int nent;
  int pos = block_exclusive_scan(mine, tmp, &nent);
  for (int w = w0; w < w1; ++w) {
    uint32_t o = 0u;
    for (int h = 0; h < G; ++h) o |= bm[(size_t)h * words + w];
    while (o) {
      const int b = __ffs(o) - 1;
      o &= o - 1u;
      uint32_t mk = 0u;
      for (int h = 0; h < G; ++h) mk |= ((bm[(size_t)h * words + w] >> b) & 1u) << h;
      ent_id[pos] = w * 32 + b;
      ent_mask[pos] = mk;
      ++pos;
    }
  }
  __syncthreads();
  // row offsets of the entries inside the unit's exact row list
  const int t_app = *app_count;
  const int nsteady = n_sink + W + t_app;
  int running = nsteady;
  for (int e0 = 0; e0 < nent; e0 += kUnionThreads) {
    const int e = e0 + tid;
    const int sz = e < nent ? cnt[(size_t)u * C + ent_id[e]] : 0;
    int tot;
    const int ex = block_exclusive_scan(sz, tmp, &tot);
    if (e < nent) ent_row[e] = running + ex;
    running += tot;
  }
  __syncthreads();
  const int R = running;
  if (R > rows_cap) {
    if (tid == 0) { atomicOr(err, WI_DEVERR_UNION_OVERFLOW); rcount[u] = 0; }
    return;
  }
  uint32_t* ro = rows + (size_t)u * rows_cap;
  for (int r = tid; r < nsteady; r += kUnionThreads) {
    long long row;
    if (r < n_sink) row = r;
    else if (r < n_sink + W) row = n - W + (r - n_sink);
    else row = n + (r - n_sink - W);
    ro[r] = ((uint32_t)row << 8) | all;
  }
  // one warp per entry writes its cluster's contiguous rows
  const int lane = tid & 31, warp = tid >> 5;
  for (int e = warp; e < nent; e += kUnionThreads / 32) {
    const int id = ent_id[e];
    const int b = off[(size_t)u * (C + 1) + id];
    const int sz = cnt[(size_t)u * C + id];
    const uint32_t mk = ent_mask[e];
    for (int i = lane; i < sz; i += 32) ro[ent_row[e] + i] = ((uint32_t)(b + i) << 8) | mk;
  }
  if (tid == 0) {
    rcount[u] = R;
    atomicAdd(rows_total, (unsigned long long)R);  // exact rows of the step, for byte accounting
  }
}

// ---------------------------------------------------------------- D3 ----
// CTA = (split, unit): rows [R*s/NS, R*(s+1)/NS) of the unit's exact row
// list.  Each warp walks groups of 8 rows: 8 K rows and 8 V rows in flight,
// per-head online softmax (m, Z, N[4 dims per lane]); warps merge at the end.
template <int G>
__global__ void __launch_bounds__(kD3Threads) k_d3_exact(const bf16* __restrict__ q, const bf16* __restrict__ K,
                                                        const bf16* __restrict__ V, const bf16* __restrict__ appK,
                                                        const bf16* __restrict__ appV,
                                                        const uint32_t* __restrict__ rows,
                                                        const int* __restrict__ rcount, float* __restrict__ part,
                                                        long long n, int max_append, long long rows_cap, int NS,
                                                        float lam, int* err) {
  __shared__ __align__(16) float red[kD3Threads / 32][G][WI_PART];
  const int u = blockIdx.y, s = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NW = kD3Threads / 32;
  const long long R = rcount[u];
  const long long r0 = R * s / NS, r1 = R * (s + 1) / NS;
  float qr[G][4];
  load_q<G>(q, u, lane, qr);
  float m[G], Z[G], N[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    Z[h] = 0.f;
    N[h][0] = N[h][1] = N[h][2] = N[h][3] = 0.f;
  }
  const uint32_t* ro = rows + (size_t)u * rows_cap;
  const bf16* Ku = K + (size_t)u * n * WI_D;
  const bf16* Vu = V + (size_t)u * n * WI_D;
  const bf16* Ka = appK + (size_t)u * max_append * WI_D;
  const bf16* Va = appV + (size_t)u * max_append * WI_D;
  for (long long rb = r0 + warp * 8; rb < r1; rb += 8 * NW) {
    const int nr = (int)min(8LL, r1 - rb);
    const uint32_t mine = lane < nr ? ro[rb + lane] : 0u;
    uint2 kw[8], vw[8];
    uint32_t mk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t e = __shfl_sync(0xffffffffu, mine, i);
      mk[i] = i < nr ? (e & 0xFFu) : 0u;
      kw[i] = make_uint2(0u, 0u);  // rows past the range contribute p = 0 times a finite value
      vw[i] = make_uint2(0u, 0u);
      if (i < nr) {
        const long long row = e >> 8;
        const bf16* kp;
        const bf16* vp;
        if (row < n) { kp = Ku + row * WI_D; vp = Vu + row * WI_D; }
        else { kp = Ka + (row - n) * WI_D; vp = Va + (row - n) * WI_D; }
        kw[i] = ldg_u2(kp + 4 * lane);
        vw[i] = ldg_u2(vp + 4 * lane);
      }
    }
    float l[8][G];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float x[4];
      unpack_bf16x4(kw[i], x);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float dsum = qr[h][0] * x[0];
        dsum = fmaf(qr[h][1], x[1], dsum);
        dsum = fmaf(qr[h][2], x[2], dsum);
        dsum = fmaf(qr[h][3], x[3], dsum);
        dsum = warp_sum(dsum);
        l[i][h] = ((mk[i] >> h) & 1u) ? lam * dsum : -INFINITY;
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float mx = m[h];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx = fmaxf(mx, l[i][h]);
      if (mx == -INFINITY) continue;
      const float sc = __expf(m[h] - mx);  // m == -inf gives 0
      Z[h] *= sc;
      N[h][0] *= sc; N[h][1] *= sc; N[h][2] *= sc; N[h][3] *= sc;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float p = __expf(l[i][h] - mx);  // -inf gives 0
        float x[4];
        unpack_bf16x4(vw[i], x);
        Z[h] += p;
        N[h][0] = fmaf(p, x[0], N[h][0]);
        N[h][1] = fmaf(p, x[1], N[h][1]);
        N[h][2] = fmaf(p, x[2], N[h][2]);
        N[h][3] = fmaf(p, x[3], N[h][3]);
      }
      m[h] = mx;
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    if (lane == 0) { red[warp][h][0] = m[h]; red[warp][h][1] = Z[h]; }
    *reinterpret_cast<float4*>(&red[warp][h][4 + 4 * lane]) = make_float4(N[h][0], N[h][1], N[h][2], N[h][3]);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * WI_D; i += kD3Threads) {
    const int h = i / WI_D, dd = i % WI_D;
    float M = -INFINITY;
    for (int w = 0; w < NW; ++w) M = fmaxf(M, red[w][h][0]);
    float z = 0.f, a = 0.f;
    if (M > -INFINITY) {
      for (int w = 0; w < NW; ++w) {
        const float mw = red[w][h][0];
        if (mw == -INFINITY) continue;
        const float f = __expf(mw - M);
        z = fmaf(f, red[w][h][1], z);
        a = fmaf(f, red[w][h][4 + dd], a);
      }
    }
    float* o = part + (((size_t)u * G + h) * NS + s) * WI_PART;
    if (dd == 0) { o[0] = M; o[1] = z; }
    o[4 + dd] = a;
  }
}

// ------------------------------------------------------------- D4 + D5 ----
// CTA = (head, unit), thread = output dim.  Estimate: merge D1's chunk
// partials, subtract the retrieved clusters' terms (they are counted exactly
// in D3), clamp at zero.  Exact: merge D3's split partials.  Output: LSE
// merge of the two.
__global__ void __launch_bounds__(WI_D) k_d5_merge(const float* __restrict__ part1,
                                                  const float* __restrict__ part3,
                                                  const float* __restrict__ scores, const int* __restrict__ sel,
                                                  const int* __restrict__ selcnt, const int* __restrict__ nonempty,
                                                  const int* __restrict__ cnt, const float* __restrict__ valsum,
                                                  float* __restrict__ out, int G, int C, int kmax, int nchunk,
                                                  int NS, float lam) {
  const int h = blockIdx.x, u = blockIdx.y, d = threadIdx.x;
  const size_t uh = (size_t)u * G + h;
  const float* p1 = part1 + uh * nchunk * WI_PART;
  float Me = -INFINITY;
  for (int c = 0; c < nchunk; ++c) Me = fmaxf(Me, p1[(size_t)c * WI_PART]);
  float Ze = 0.f, Ne = 0.f;
  const int ns = selcnt[uh];
  if (Me > -INFINITY && ns < nonempty[u]) {
    for (int c = 0; c < nchunk; ++c) {
      const float mc = p1[(size_t)c * WI_PART];
      if (mc == -INFINITY) continue;
      const float f = __expf(mc - Me);
      Ze = fmaf(f, p1[(size_t)c * WI_PART + 1], Ze);
      Ne = fmaf(f, p1[(size_t)c * WI_PART + 4 + d], Ne);
    }
    const int* sh = sel + uh * kmax;
    const float* sch = scores + uh * C;
    for (int i = 0; i < ns; ++i) {
      const int j = sh[i];
      const float w = __expf(lam * sch[j] - Me);
      Ze = fmaf(-(float)cnt[(size_t)u * C + j], w, Ze);
      Ne = fmaf(-w, valsum[((size_t)u * C + j) * WI_D + d], Ne);
    }
    Ze = fmaxf(Ze, 0.f);
  }
  const float* p3 = part3 + uh * NS * WI_PART;
  float Mx = -INFINITY;
  for (int s = 0; s < NS; ++s) Mx = fmaxf(Mx, p3[(size_t)s * WI_PART]);
  float Zx = 0.f, Nx = 0.f;
  if (Mx > -INFINITY) {
    for (int s = 0; s < NS; ++s) {
      const float ms = p3[(size_t)s * WI_PART];
      if (ms == -INFINITY) continue;
      const float f = __expf(ms - Mx);
      Zx = fmaf(f, p3[(size_t)s * WI_PART + 1], Zx);
      Nx = fmaf(f, p3[(size_t)s * WI_PART + 4 + d], Nx);
    }
  }
  const float M = fmaxf(Mx, Me);
  const float fx = Mx > -INFINITY ? __expf(Mx - M) : 0.f;
  const float fe = (Me > -INFINITY && Ze > 0.f) ? __expf(Me - M) : 0.f;
  out[uh * WI_D + d] = (Nx * fx + Ne * fe) / (Zx * fx + Ze * fe);
}

// ---------------------------------------------------------------- D6 ----
__global__ void k_d6_append(const bf16* __restrict__ k_new, const bf16* __restrict__ v_new, bf16* __restrict__ appK,
                            bf16* __restrict__ appV, int* __restrict__ app_count, int t, int max_append) {
  const int u = blockIdx.x, lane = threadIdx.x;
  const size_t dst = ((size_t)u * max_append + t) * WI_D;
  reinterpret_cast<uint2*>(appK + dst)[lane] = ldg_u2(k_new + (size_t)u * WI_D + 4 * lane);
  reinterpret_cast<uint2*>(appV + dst)[lane] = ldg_u2(v_new + (size_t)u * WI_D + 4 * lane);
  if (u == 0 && lane == 0) *app_count = t + 1;
}

// Optional timing events: ev[0] before D1, ev[i] after the i-th kernel.
inline cudaError_t mark(const cudaEvent_t* ev, int i, cudaStream_t st) {
  return ev ? cudaEventRecordWithFlags(ev[i], st, cudaEventRecordExternal) : cudaSuccess;
}

template <int G>
cudaError_t launch_g(const WiGeom& g, const WiDecodeBufs& b, const void* qv, float* out, cudaStream_t st,
                     const cudaEvent_t* ev) {
  const bf16* q = static_cast<const bf16*>(qv);
  cudaError_t e0 = mark(ev, 0, st);
  if (e0 != cudaSuccess) return e0;
  const float lam = 1.0f / sqrtf((float)WI_D);
  const size_t smem1 = sizeof(float) * ((size_t)G * b.chunk + (size_t)(kD1Threads / 32) * G * WI_PART);
  static int smem1_set = 0;
  cudaError_t e = wi_ensure_smem(k_d1_score_estimate<G>, smem1, &smem1_set);
  if (e != cudaSuccess) return e;
  k_d1_score_estimate<G><<<dim3(b.nchunk, g.U), kD1Threads, smem1, st>>>(
      q, static_cast<const bf16*>(b.mu), b.valsum, b.cnt, b.scores, b.part1, g.C, b.chunk, b.nchunk, lam);
  if ((e = cudaGetLastError()) != cudaSuccess || (e = mark(ev, 1, st)) != cudaSuccess) return e;
  k_d2_topk<<<dim3(G, g.U), kTopkThreads, 0, st>>>(b.scores, b.cnt, b.nonempty, b.sel, b.selcnt, G, g.C, g.kmax,
                                                   b.err);
  if ((e = cudaGetLastError()) != cudaSuccess || (e = mark(ev, 2, st)) != cudaSuccess) return e;
  const size_t smemu = wi_union_smem_bytes(g);
  static int smemu_set = 0;
  e = wi_ensure_smem(k_d2_union, smemu, &smemu_set);
  if (e != cudaSuccess) return e;
  k_d2_union<<<g.U, kUnionThreads, smemu, st>>>(b.sel, b.selcnt, b.cnt, b.off, b.app_count, b.rows, b.rcount, b.rows_total, G,
                                                g.C, g.kmax, g.n, g.n_sink, g.W, b.rows_cap, b.err);
  if ((e = cudaGetLastError()) != cudaSuccess || (e = mark(ev, 3, st)) != cudaSuccess) return e;
  k_d3_exact<G><<<dim3(b.nsplit, g.U), kD3Threads, 0, st>>>(
      q, static_cast<const bf16*>(b.K), static_cast<const bf16*>(b.V), static_cast<const bf16*>(b.appK),
      static_cast<const bf16*>(b.appV), b.rows, b.rcount, b.part3, g.n, g.max_append > 0 ? g.max_append : 1,
      b.rows_cap, b.nsplit, lam, b.err);
  if ((e = cudaGetLastError()) != cudaSuccess || (e = mark(ev, 4, st)) != cudaSuccess) return e;
  k_d5_merge<<<dim3(G, g.U), WI_D, 0, st>>>(b.part1, b.part3, b.scores, b.sel, b.selcnt, b.nonempty, b.cnt,
                                            b.valsum, out, G, g.C, g.kmax, b.nchunk, b.nsplit, lam);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return mark(ev, 5, st);
}

}  // namespace

size_t wi_union_smem_bytes(const WiGeom& g) {
  const size_t words = (size_t)(g.C + 31) / 32;
  return sizeof(uint32_t) * ((size_t)g.G * words + 3 * (size_t)g.G * g.kmax + 1);
}

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
  k_d6_append<<<g.U, 32, 0, st>>>(static_cast<const bf16*>(k_new), static_cast<const bf16*>(v_new),
                                  static_cast<bf16*>(b.appK), static_cast<bf16*>(b.appV), b.app_count, t,
                                  g.max_append);
  return cudaGetLastError();
}
