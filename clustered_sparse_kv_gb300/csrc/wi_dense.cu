// wi_dense.cu -- full attention over every cached token: the dense comparator
// of the wave index (the attention that the tripartite approximation stands in
// for; RetroInfer summaries de/fr/zh section 2.A, speed-up over it in zh
// section 3).
//
// One decode step for all units.  Each unit's rows -- its n context rows in
// the index's cluster-contiguous order (attention does not depend on the row
// order) followed by its appended rows -- are cut into S row ranges, one CTA
// each.  A producer lane bulk-copies 64-row K and V stages into a 3-stage
// mbarrier ring; 8 consumer warps take 8 rows each per stage and compute the
// logits of all G query heads from that one copy (the group shares each row
// read), with an online softmax per head.  The last CTA of a unit (ticket)
// merges the S partials of every head by log-sum-exp.
#include "wi_internal.h"
#include "wi_pipe.cuh"

namespace {

constexpr int kDnRows = 64;
constexpr int kDnStages = 3;
constexpr int kDnWarps = 8;
constexpr int kDnThreads = 32 * (kDnWarps + 1);

struct DnStage {
  bf16 k[kDnRows * WI_D];
  bf16 v[kDnRows * WI_D];
};
constexpr size_t kDnSmem = sizeof(DnStage) * kDnStages + 2 * kDnStages * sizeof(uint64_t) +
                           sizeof(int) * (kDnStages + 4);

struct DenseArgs {
  const bf16* q;     // [U][G][128]
  const bf16* K;     // [U][n][128]
  const bf16* V;
  const bf16* appK;  // [U][max_append][128]
  const bf16* appV;
  const int* app_count;
  float* part;       // [U][G][S][WI_PART]: m, Z, -, -, N[128] of each row range
  unsigned* ticket;  // [U]
  float* out;        // [U][G][128]
  int* err;
  long long n;
  int S, max_append;
  float lam;
};

// Registers grow with G (query rows and accumulators of every head): two CTAs
// per SM up to 4 heads, one above.
template <int G>
__global__ void __launch_bounds__(kDnThreads, G <= 4 ? 2 : 1) k_dense_decode(DenseArgs a) {
  constexpr int HG = (G + 3) / 4;  // groups of 4 heads: 4 heads x 8 rows = one 32-value reduction
  extern __shared__ __align__(128) unsigned char dn_raw[];
  DnStage* st = reinterpret_cast<DnStage*>(dn_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(dn_raw + sizeof(DnStage) * kDnStages);
  uint64_t* empty = full + kDnStages;
  int* nrows = reinterpret_cast<int*>(empty + kDnStages);  // [stages]
  int* flags = nrows + kDnStages;                           // abort, last CTA
  const int split = blockIdx.x, u = blockIdx.y, S = a.S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kDnStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDnWarps);
    }
    flags[0] = 0;
    flags[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // context rows [r0, r1) of this range; the last range also takes the appended rows
  const long long per = (a.n + S - 1) / S;
  const long long r0 = min(a.n, (long long)split * per), r1 = min(a.n, r0 + per);
  float mo[HG], zo[HG], N[G][4];  // this lane's head (4 hg + lane / 8): running max and sum
#pragma unroll
  for (int hg = 0; hg < HG; ++hg) {
    mo[hg] = -INFINITY;
    zo[hg] = 0.f;
  }
#pragma unroll
  for (int h = 0; h < G; ++h) N[h][0] = N[h][1] = N[h][2] = N[h][3] = 0.f;

  if (warp == kDnWarps) {
    if (lane == 0) {
      const int amax = a.max_append > 0 ? a.max_append : 1;
      const int na = split == S - 1 ? min(max(*a.app_count, 0), a.max_append) : 0;
      int it = 0;
      // one stage: nr rows from kp / vp (nr = 0 ends the stream)
      auto put = [&](const bf16* kp, const bf16* vp, int nr) -> bool {
        const int s = it % kDnStages, ph = it / kDnStages;
        if (it >= kDnStages && !mbar_wait(&empty[s], (ph - 1) & 1, a.err)) return false;
        nrows[s] = nr;
        const uint32_t bytes = (uint32_t)nr * WI_D * 2;
        mbar_arrive_expect_tx(&full[s], 2 * bytes);
        if (nr > 0) {
          bulk_g2s(st[s].k, kp, bytes, &full[s]);
          bulk_g2s(st[s].v, vp, bytes, &full[s]);
        }
        ++it;
        return true;
      };
      const bf16* Ku = a.K + (size_t)u * a.n * WI_D;
      const bf16* Vu = a.V + (size_t)u * a.n * WI_D;
      const bf16* Ka = a.appK + (size_t)u * amax * WI_D;
      const bf16* Va = a.appV + (size_t)u * amax * WI_D;
      bool ok = true;
      for (long long r = r0; r < r1 && ok; r += kDnRows)
        ok = put(Ku + r * WI_D, Vu + r * WI_D, (int)min((long long)kDnRows, r1 - r));
      for (int r = 0; r < na && ok; r += kDnRows) ok = put(Ka + (size_t)r * WI_D, Va + (size_t)r * WI_D, min(kDnRows, na - r));
      if (ok) ok = put(nullptr, nullptr, 0);
      if (!ok) flags[0] = 1;  // the consumers' own bounded waits end their loop
    }
  } else {
    float qr[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) load_bf16x4(a.q + ((size_t)u * G + h) * WI_D + 4 * lane, qr[h]);
    const int ri = lane & 7;  // after the reduction: row (of the warp's 8) and head lane / 8 of the group
    for (int it = 0;; ++it) {
      const int s = it % kDnStages, ph = it / kDnStages;
      if (!mbar_wait(&full[s], ph & 1, a.err)) {
        flags[0] = 1;
        break;
      }
      const int nr = nrows[s];
      if (nr == 0) break;
      const int i0 = warp * 8;
      if (i0 < nr) {
        const DnStage& T = st[s];
#pragma unroll
        for (int hg = 0; hg < HG; ++hg) {
          // v[hh * 8 + i]: this lane's part of q_{4hg+hh} . K_{i0+i}
          float v[32];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float x[4] = {0.f, 0.f, 0.f, 0.f};
            if (i0 + i < nr) unpack_bf16x4(*reinterpret_cast<const uint2*>(&T.k[(i0 + i) * WI_D + 4 * lane]), x);
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
              const int h = 4 * hg + hh;
              float2 acc = make_float2(0.f, 0.f);
              if (h < G) {
                acc = __fmul2_rn(make_float2(qr[h < G ? h : 0][0], qr[h < G ? h : 0][1]), make_float2(x[0], x[1]));
                acc = __ffma2_rn(make_float2(qr[h < G ? h : 0][2], qr[h < G ? h : 0][3]), make_float2(x[2], x[3]), acc);
              }
              v[hh * 8 + i] = acc.x + acc.y;
            }
          }
          const float dot = transpose_reduce<32>(v);  // lane l: head 4hg + l/8, row l%8
          const bool valid = 4 * hg + (lane >> 3) < G && i0 + ri < nr;
          const float l = valid ? a.lam * dot : -INFINITY;
          float mx = fmaxf(l, __shfl_xor_sync(0xffffffffu, l, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          const float m_new = fmaxf(mo[hg], mx);
          const float sc = m_new == -INFINITY ? 1.f : __expf(mo[hg] - m_new);
          const float pr = valid ? __expf(l - m_new) : 0.f;
          float zs = pr + __shfl_xor_sync(0xffffffffu, pr, 1);
          zs += __shfl_xor_sync(0xffffffffu, zs, 2);
          zs += __shfl_xor_sync(0xffffffffu, zs, 4);
          zo[hg] = zo[hg] * sc + zs;
          mo[hg] = m_new;
#pragma unroll
          for (int hh = 0; hh < 4; ++hh) {
            const float f = __shfl_sync(0xffffffffu, sc, hh * 8);
            if (4 * hg + hh < G) {
              const int h = 4 * hg + hh < G ? 4 * hg + hh : 0;
              N[h][0] *= f; N[h][1] *= f; N[h][2] *= f; N[h][3] *= f;
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (i0 + i < nr) {  // warp-uniform
              float x[4];
              unpack_bf16x4(*reinterpret_cast<const uint2*>(&T.v[(i0 + i) * WI_D + 4 * lane]), x);
#pragma unroll
              for (int hh = 0; hh < 4; ++hh) {
                const float p = __shfl_sync(0xffffffffu, pr, hh * 8 + i);
                if (4 * hg + hh < G) {
                  const int h = 4 * hg + hh < G ? 4 * hg + hh : 0;
                  N[h][0] = fmaf(p, x[0], N[h][0]);
                  N[h][1] = fmaf(p, x[1], N[h][1]);
                  N[h][2] = fmaf(p, x[2], N[h][2]);
                  N[h][3] = fmaf(p, x[3], N[h][3]);
                }
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }
  __syncthreads();  // the stages are free: per-warp partials go there
  float* red = reinterpret_cast<float*>(dn_raw);  // [kDnWarps][G][WI_PART]
  if (warp < kDnWarps) {
#pragma unroll
    for (int hg = 0; hg < HG; ++hg)
      if ((lane & 7) == 0 && 4 * hg + (lane >> 3) < G) {
        float* r = red + ((size_t)warp * G + 4 * hg + (lane >> 3)) * WI_PART;
        r[0] = mo[hg];
        r[1] = zo[hg];
      }
#pragma unroll
    for (int h = 0; h < G; ++h)
      *reinterpret_cast<float4*>(red + ((size_t)warp * G + h) * WI_PART + 4 + 4 * lane) =
          make_float4(N[h][0], N[h][1], N[h][2], N[h][3]);
  }
  __syncthreads();
  if (flags[0]) return;  // uniform; the error is recorded
  // this range's partial of every head (column c of head h)
  float* pu = a.part + (size_t)u * G * S * WI_PART;
  for (int c = tid; c < G * WI_D; c += kDnThreads) {
    const int h = c / WI_D, d = c % WI_D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDnWarps; ++w) M = fmaxf(M, red[((size_t)w * G + h) * WI_PART]);
    float z = 0.f, acc = 0.f;
    if (M > -INFINITY)
#pragma unroll
      for (int w = 0; w < kDnWarps; ++w) {
        const float* r = red + ((size_t)w * G + h) * WI_PART;
        if (r[0] == -INFINITY) continue;
        const float f = __expf(r[0] - M);
        z = fmaf(f, r[1], z);
        acc = fmaf(f, r[4 + d], acc);
      }
    float* o = pu + ((size_t)h * S + split) * WI_PART;
    if (d == 0) {
      o[0] = M;
      o[1] = z;
    }
    o[4 + d] = acc;
  }
  // publish and take a ticket: the barrier orders the CTA's writes before thread 0's release;
  // the acquire side makes every earlier range's partial visible to the last CTA
  __syncthreads();
  if (tid == 0) flags[1] = ticket_acq_rel(&a.ticket[u]) == (unsigned)(S - 1);
  __syncthreads();
  if (!flags[1]) return;
  // ---- the last CTA of the unit: o_h = sum_s e^{m_s - M} N_s / sum_s e^{m_s - M} Z_s
  float* wt = reinterpret_cast<float*>(dn_raw);  // [G][S]: m_s, then the weights e^{m_s - M}
  float* zz = wt + (size_t)G * S;                // [G][S]: Z_s
  float* den = zz + (size_t)G * S;               // [G]
  for (int i = tid; i < G * S; i += kDnThreads) {
    const float2 mz = __ldcg(reinterpret_cast<const float2*>(pu + (size_t)i * WI_PART));
    wt[i] = mz.x;
    zz[i] = mz.y;
  }
  __syncthreads();
  if (warp < G) {
    const int h = warp;
    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, wt[h * S + s]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float Z = 0.f;
    for (int s = lane; s < S; s += 32) {
      const float m = wt[h * S + s];
      const float f = m == -INFINITY ? 0.f : __expf(m - M);
      wt[h * S + s] = f;
      Z = fmaf(f, zz[h * S + s], Z);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);
    if (lane == 0) den[h] = Z;
  }
  __syncthreads();
  for (int c = tid; c < G * WI_D; c += kDnThreads) {
    const int h = c / WI_D, d = c % WI_D;
    const float* col = pu + (size_t)h * S * WI_PART + 4 + d;
    float acc = 0.f;
#pragma unroll 8
    for (int s = 0; s < S; ++s) acc = fmaf(wt[h * S + s], __ldcg(col + (size_t)s * WI_PART), acc);
    a.out[((size_t)u * G + h) * WI_D + d] = acc / den[h];
  }
  if (tid == 0) a.ticket[u] = 0u;  // ready for the next call
}

template <int G>
cudaError_t launch_dense_g(const WiGeom& g, const WiDecodeBufs& b, const void* q, float* out, cudaStream_t st) {
  static int smem_set[kWiSmemDevices] = {};
  cudaError_t e = wi_ensure_smem(k_dense_decode<G>, kDnSmem, smem_set);
  if (e != cudaSuccess) return e;
  DenseArgs a;
  a.q = static_cast<const bf16*>(q);
  a.K = static_cast<const bf16*>(b.K);
  a.V = static_cast<const bf16*>(b.V);
  a.appK = static_cast<const bf16*>(b.appK);
  a.appV = static_cast<const bf16*>(b.appV);
  a.app_count = b.app_count;
  a.part = b.dpart;
  a.ticket = b.dticket;
  a.out = out;
  a.err = b.err;
  a.n = g.n;
  a.S = b.dsplits;
  a.max_append = g.max_append;
  a.lam = 1.0f / sqrtf((float)WI_D);
  k_dense_decode<G><<<dim3(b.dsplits, g.U), kDnThreads, kDnSmem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

int wi_dense_ctas_per_sm(int G) { return G <= 4 ? 2 : 1; }

cudaError_t wi_launch_dense(const WiGeom& g, const WiDecodeBufs& b, const void* q, float* out, cudaStream_t st) {
  switch (g.G) {
    case 1: return launch_dense_g<1>(g, b, q, out, st);
    case 2: return launch_dense_g<2>(g, b, q, out, st);
    case 3: return launch_dense_g<3>(g, b, q, out, st);
    case 4: return launch_dense_g<4>(g, b, q, out, st);
    case 5: return launch_dense_g<5>(g, b, q, out, st);
    case 6: return launch_dense_g<6>(g, b, q, out, st);
    case 7: return launch_dense_g<7>(g, b, q, out, st);
    case 8: return launch_dense_g<8>(g, b, q, out, st);
    default: return cudaErrorInvalidValue;
  }
}
