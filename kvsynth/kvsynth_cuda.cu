/*
 * kvsynth_cuda.cu -- the seeded synthetic generator of kvsynth.c, on the GPU.
 *
 * Input generation only, like kvsynth.c: no wave-index arithmetic.  It draws
 * the same counter-based SplitMix64 numbers, applies the same Box-Muller,
 * topic chain, rotate-half RoPE and sink scaling in double precision, and
 * rounds to bf16 the same way, so that caches too large to generate on the
 * host (a million tokens x 32 layers) come out with the host generator's
 * bytes.  It is compiled with -fmad=false so that every product and sum is
 * rounded separately, as the host build (-ffp-contract=off) does.  The
 * rotation frequencies theta^(-2i/d) are computed on the host with its libm
 * and passed in, so every rotation angle is the host's product exactly; the
 * remaining differences come from the device's double log, sin and cos
 * (within 1-2 ulp of the host's), which move a bf16 rounding only for values
 * within a few double ulps of a rounding boundary.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL
#define KVS_MAX_D 256

enum { TAG_TOPIC = 1, TAG_CHAIN = 2, TAG_KNOISE = 3, TAG_VALUE = 4, TAG_QTOPIC = 5, TAG_QNOISE = 6 };

typedef struct {
  uint64_t seed;
  int d, n_topics, n_sink;
  double p_stay, sigma_k, sink_scale, theta, q_scale, sigma_q;
} kvs_params;

struct InvFreq {
  double v[KVS_MAX_D / 2];
};

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t draw(uint64_t s, uint64_t i) { return mix64(s + (i + 1) * GOLDEN); }

__device__ __forceinline__ uint64_t stream_key(uint64_t seed, uint64_t a, uint64_t b, uint64_t c, uint64_t tag) {
  uint64_t s = draw(seed, 0);
  s = draw(s, a);
  s = draw(s, b);
  s = draw(s, c);
  return draw(s, tag);
}

__device__ __forceinline__ double uniform01(uint64_t key, uint64_t i) {
  return (double)((draw(key, i) >> 11) + 1) * 0x1p-53;
}

__device__ __forceinline__ void normal_pair(uint64_t key, uint64_t m, double* z0, double* z1) {
  const double u1 = uniform01(key, 2 * m), u2 = uniform01(key, 2 * m + 1);
  const double r = sqrt(-2.0 * log(u1));
  const double a = 6.283185307179586476925286766559 * u2;
  double s, c;
  sincos(a, &s, &c);
  *z0 = r * c;
  *z1 = r * s;
}

// double -> bf16 bits, round to nearest even, straight from double (as kvs_bf16 on the host)
__device__ __forceinline__ uint16_t to_bf16(double x) {
  if (x == 0.0) return signbit(x) ? 0x8000 : 0;
  int e;
  const double m = frexp(x, &e);
  const double r = rint(ldexp(m, 8));
  const float f = (float)ldexp(r, e - 8);
  return (uint16_t)(__float_as_uint(f) >> 16);
}

// topic centres of every unit: [units][T][d] doubles
__global__ void k_topics(kvs_params P, int L, int Hkv, int units, double* __restrict__ topics) {
  const long long per = (long long)P.n_topics * P.d / 2;  // normal pairs per unit
  const long long total = per * units;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int u = (int)(i / per);
    const long long m = i % per;
    const int b = u / (L * Hkv), l = (u / Hkv) % L, h = u % Hkv;
    const uint64_t key = stream_key(P.seed, b, l, h, TAG_TOPIC);
    double z0, z1;
    normal_pair(key, (uint64_t)m, &z0, &z1);
    topics[(size_t)u * P.n_topics * P.d + 2 * m] = z0;
    topics[(size_t)u * P.n_topics * P.d + 2 * m + 1] = z1;
  }
}

// One warp per (unit, position) row; lane l makes elements 2l, 2l+1 (normal pair l) and
// 2l+64, 2l+65 (pair l+32) for d = 128: the rotate-half pairs (i, i + 64) stay in one lane.
// Generic d: lane l takes normal pairs l, l + 32, ... < d/2, and the rotation is done through
// shared memory.
__global__ void __launch_bounds__(256) k_rows(kvs_params P, InvFreq inv, int L, int Hkv, int units, long p0,
                                              long p1, const double* __restrict__ topics,
                                              uint16_t* __restrict__ K, uint16_t* __restrict__ V) {
  __shared__ double xs[8][KVS_MAX_D];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int d = P.d, hd = d / 2, T = P.n_topics;
  const long rows_u = p1 - p0;
  const long long total = (long long)units * rows_u;
  double* x = xs[wib];
  for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + wib; r < total;
       r += (long long)gridDim.x * (blockDim.x >> 5)) {
    const int u = (int)(r / rows_u);
    const long p = p0 + (long)(r % rows_u);
    const int b = u / (L * Hkv), l = (u / Hkv) % L, h = u % Hkv;
    // topic of position p: the pick at the last position q <= p where the chain redrew
    // (q == 0, or its stay draw >= p_stay); the lanes test 32 positions at a time
    const uint64_t kc = stream_key(P.seed, b, l, h, TAG_CHAIN);
    long q = -1;
    for (long base = p; q < 0; base -= 32) {
      const long c = base - lane;
      const bool reset = c >= 0 && (c == 0 || uniform01(kc, 2 * (uint64_t)c) >= P.p_stay);
      const unsigned bal = __ballot_sync(0xffffffffu, reset);
      if (bal) q = base - (__ffs(bal) - 1);
    }
    const double u_pick = uniform01(kc, 2 * (uint64_t)q + 1);
    int t = (int)((1.0 - u_pick) * T);
    if (t >= T) t = T - 1;
    const double* cen = topics + ((size_t)u * T + t) * d;
    const uint64_t kk = stream_key(P.seed, b, l, h, TAG_KNOISE);
    const uint64_t kv = stream_key(P.seed, b, l, h, TAG_VALUE);
    uint16_t* ko = K + (size_t)r * d;
    uint16_t* vo = V + (size_t)r * d;
    for (int m = lane; m < hd; m += 32) {
      double z0, z1;
      normal_pair(kk, (uint64_t)p * hd + m, &z0, &z1);
      x[2 * m] = cen[2 * m] + P.sigma_k * z0;
      x[2 * m + 1] = cen[2 * m + 1] + P.sigma_k * z1;
    }
    __syncwarp();
    const double sc = (p < P.n_sink) ? P.sink_scale : 1.0;
    for (int i = lane; i < hd; i += 32) {
      const double ang = (double)p * inv.v[i];
      double s, c;
      sincos(ang, &s, &c);
      const double a = x[i], bb = x[i + hd];
      const double r0 = a * c - bb * s;
      const double r1 = bb * c + a * s;
      ko[i] = to_bf16(sc * r0);
      ko[i + hd] = to_bf16(sc * r1);
    }
    __syncwarp();
    for (int m = lane; m < hd; m += 32) {
      double z0, z1;
      normal_pair(kv, (uint64_t)p * hd + m, &z0, &z1);
      const uint32_t w = (uint32_t)to_bf16(z0) | ((uint32_t)to_bf16(z1) << 16);
      reinterpret_cast<uint32_t*>(vo)[m] = w;
    }
  }
}

// Queries of decode step `step` at position `pos`: one warp per query head.
__global__ void k_queries(kvs_params P, InvFreq inv, int B, int L, int Hq, int Hkv, long pos, int step,
                          const double* __restrict__ topics, uint16_t* __restrict__ Q) {
  __shared__ double xs[8][KVS_MAX_D];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int d = P.d, hd = d / 2, T = P.n_topics, g = Hq / Hkv;
  const int row = blockIdx.x * (blockDim.x >> 5) + wib;  // (b, l, h)
  if (row >= B * L * Hq) return;
  const int b = row / (L * Hq), l = (row / Hq) % L, h = row % Hq;
  const int hk = h / g;
  const int u = (b * L + l) * Hkv + hk;
  const uint64_t kt = stream_key(P.seed, b, l, (uint64_t)h * 1000003ULL + (uint64_t)step, TAG_QTOPIC);
  const uint64_t kn = stream_key(P.seed, b, l, (uint64_t)h * 1000003ULL + (uint64_t)step, TAG_QNOISE);
  int pick[3], got = 0;
  uint64_t i = 0;
  const int want = T >= 3 ? 3 : T;
  while (got < want) {  // every lane draws the same sequence
    int t = (int)((1.0 - uniform01(kt, i++)) * T);
    if (t >= T) t = T - 1;
    bool dup = false;
    for (int a = 0; a < got; ++a) dup |= (pick[a] == t);
    if (!dup) pick[got++] = t;
  }
  double* x = xs[wib];
  for (int m = lane; m < hd; m += 32) {
    double z0, z1;
    normal_pair(kn, (uint64_t)m, &z0, &z1);
    x[2 * m] = P.sigma_q * z0;
    x[2 * m + 1] = P.sigma_q * z1;
  }
  __syncwarp();
  for (int e = lane; e < d; e += 32)
    for (int a = 0; a < got; ++a) x[e] += P.q_scale * topics[((size_t)u * T + pick[a]) * d + e];
  __syncwarp();
  uint16_t* qo = Q + (size_t)row * d;
  for (int i2 = lane; i2 < hd; i2 += 32) {
    const double ang = (double)pos * inv.v[i2];
    double s, c;
    sincos(ang, &s, &c);
    const double a = x[i2], bb = x[i2 + hd];
    qo[i2] = to_bf16(a * c - bb * s);
    qo[i2 + hd] = to_bf16(bb * c + a * s);
  }
}

static InvFreq inv_freq(const kvs_params* P) {
  InvFreq f;
  for (int i = 0; i < KVS_MAX_D / 2; ++i) f.v[i] = i < P->d / 2 ? pow(P->theta, -2.0 * (double)i / (double)P->d) : 0.0;
  return f;
}

static int sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

extern "C" {

/* Topic centres of every unit, doubles [B*L*Hkv][n_topics][d] (device). 0, or a CUDA error code. */
int kvs_topics_dev(const kvs_params* P, int B, int L, int Hkv, double* topics, void* stream) {
  if (P->d > KVS_MAX_D || P->d % 2) return (int)cudaErrorInvalidValue;
  k_topics<<<sms() * 8, 256, 0, static_cast<cudaStream_t>(stream)>>>(*P, L, Hkv, B * L * Hkv, topics);
  return (int)cudaGetLastError();
}

/* Keys and values [B][L][Hkv][p1-p0][d] bf16 bits (device) for positions [p0, p1), from the
 * topic centres made by kvs_topics_dev with the same parameters. */
int kvs_cache_dev(const kvs_params* P, int B, int L, int Hkv, long p0, long p1, const double* topics, uint16_t* K,
                  uint16_t* V, void* stream) {
  if (P->d > KVS_MAX_D || P->d % 2 || p1 < p0 || p0 < 0) return (int)cudaErrorInvalidValue;
  if (p1 == p0) return 0;
  k_rows<<<sms() * 16, 256, 0, static_cast<cudaStream_t>(stream)>>>(*P, inv_freq(P), L, Hkv, B * L * Hkv, p0, p1,
                                                                     topics, K, V);
  return (int)cudaGetLastError();
}

/* Queries [B][L][Hq][d] bf16 bits (device) of decode step `step` at position `pos`. */
int kvs_queries_dev(const kvs_params* P, int B, int L, int Hq, int Hkv, long pos, int step, const double* topics,
                    uint16_t* Q, void* stream) {
  if (P->d > KVS_MAX_D || P->d % 2 || Hq % Hkv) return (int)cudaErrorInvalidValue;
  const int rows = B * L * Hq;
  k_queries<<<(rows + 7) / 8, 256, 0, static_cast<cudaStream_t>(stream)>>>(*P, inv_freq(P), B, L, Hq, Hkv, pos,
                                                                           step, topics, Q);
  return (int)cudaGetLastError();
}

}  // extern "C"
