/*
 * kvsynth.c -- seeded synthetic KV-cache and query generator.
 *
 * This is input generation only: it holds none of the wave-index arithmetic
 * (no clustering, scoring, selection or attention).  Both the CPU oracle and
 * the CUDA path consume its output bytes.
 *
 * Workload shape (RetroInfer summaries, "Problem" sections: Llama3/Qwen2.5 KV
 * caches at 128K..1M tokens; decode queries against that cache):
 *   - per unit (sequence, layer, kv head): T topic centres c_t ~ N(0, I_d);
 *   - token p picks a topic by a Markov chain: topic_0 uniform, then keep the
 *     previous topic with probability p_stay, else redraw uniformly over all T;
 *   - key_p = RoPE_p(c_topic + sigma_k * N(0, I_d)), scaled by sink_scale for
 *     p < n_sink (the scale commutes with the rotation);
 *   - value_p ~ N(0, I_d);
 *   - query of head h (kv head h / g) at decode position `pos`:
 *     RoPE_pos(q_scale * (c_a + c_b + c_c) + sigma_q * N(0, I_d)) with three
 *     distinct topics of that kv head drawn per (head, step).
 *   RoPE is the rotate-half form: pairs (i, i + d/2), frequency theta^(-2i/d).
 *   Every value is rounded once, from double, to bf16 (round to nearest even).
 *
 * Random numbers: a counter-based generator.  The i-th 64-bit draw of a
 * stream with key s is the SplitMix64 output function applied to
 * s + (i + 1) * 0x9E3779B97F4A7C15 (Steele, Lea, Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), so any draw can be computed
 * independently.  Normals come from the Box-Muller transform on pairs of
 * uniforms in (0, 1].
 */
#include <stdint.h>
#include <math.h>
#include <stddef.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

enum { TAG_TOPIC = 1, TAG_CHAIN = 2, TAG_KNOISE = 3, TAG_VALUE = 4, TAG_QTOPIC = 5, TAG_QNOISE = 6 };

uint64_t kvs_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* The i-th draw of the SplitMix64 sequence started from state s. */
uint64_t kvs_draw(uint64_t s, uint64_t i) { return kvs_mix64(s + (i + 1) * GOLDEN); }

/* Stream key for (seed, a, b, c, tag): a chain of SplitMix64 draws. */
uint64_t kvs_stream_key(uint64_t seed, uint64_t a, uint64_t b, uint64_t c, uint64_t tag) {
  uint64_t s = kvs_draw(seed, 0);
  s = kvs_draw(s, a);
  s = kvs_draw(s, b);
  s = kvs_draw(s, c);
  return kvs_draw(s, tag);
}

static inline double uniform01(uint64_t key, uint64_t i) {
  return (double)((kvs_draw(key, i) >> 11) + 1) * 0x1p-53; /* in (0, 1] */
}

/* Normals 2m and 2m+1 of a stream (Box-Muller on uniforms 2m, 2m+1). */
static inline void normal_pair(uint64_t key, uint64_t m, double* z0, double* z1) {
  const double u1 = uniform01(key, 2 * m), u2 = uniform01(key, 2 * m + 1);
  const double r = sqrt(-2.0 * log(u1));
  const double a = 6.283185307179586476925286766559 * u2;
  *z0 = r * cos(a);
  *z1 = r * sin(a);
}

double kvs_normal(uint64_t key, uint64_t i) {
  double z0, z1;
  normal_pair(key, i >> 1, &z0, &z1);
  return (i & 1) ? z1 : z0;
}

double kvs_uniform(uint64_t key, uint64_t i) { return uniform01(key, i); }

/* double -> bf16 bits, round to nearest even, straight from double. */
uint16_t kvs_bf16(double x) {
  if (x == 0.0) return signbit(x) ? 0x8000 : 0;
  int e;
  const double m = frexp(x, &e);               /* |m| in [0.5, 1) */
  const double r = nearbyint(ldexp(m, 8));     /* 8 significant bits, ties to even */
  const float f = (float)ldexp(r, e - 8);      /* exact: 8 significant bits */
  union { float f; uint32_t u; } cv;
  cv.f = f;
  return (uint16_t)(cv.u >> 16);
}

/* Rotate-half RoPE of one row in place: pairs (i, i + d/2). */
static void rope_row(double* x, int d, double theta, double pos) {
  const int h = d / 2;
  for (int i = 0; i < h; ++i) {
    const double inv = pow(theta, -2.0 * (double)i / (double)d);
    const double ang = pos * inv;
    const double c = cos(ang), s = sin(ang);
    const double a = x[i], b = x[i + h];
    x[i] = a * c - b * s;
    x[i + h] = b * c + a * s;
  }
}

typedef struct {
  uint64_t seed;
  int d, n_topics, n_sink;
  double p_stay, sigma_k, sink_scale, theta, q_scale, sigma_q;
} kvs_params;

static void unit_topics(const kvs_params* P, int seq, int layer, int kvh, double* topics) {
  const uint64_t key = kvs_stream_key(P->seed, seq, layer, kvh, TAG_TOPIC);
  const uint64_t total = (uint64_t)P->n_topics * P->d;
  for (uint64_t m = 0; m < total / 2; ++m) normal_pair(key, m, &topics[2 * m], &topics[2 * m + 1]);
}

/* Topic index of every position in [0, p1). */
static void unit_chain(const kvs_params* P, int seq, int layer, int kvh, long p1, int* topic) {
  const uint64_t key = kvs_stream_key(P->seed, seq, layer, kvh, TAG_CHAIN);
  const int T = P->n_topics;
  for (long p = 0; p < p1; ++p) {
    const double u_stay = uniform01(key, 2 * (uint64_t)p), u_pick = uniform01(key, 2 * (uint64_t)p + 1);
    int pick = (int)((1.0 - u_pick) * T); /* 1 - u in [0, 1) */
    if (pick >= T) pick = T - 1;
    if (p == 0 || u_stay >= P->p_stay) topic[p] = pick;
    else topic[p] = topic[p - 1];
  }
}

/*
 * Keys and values of one unit for positions [p0, p1), rows of d bf16.
 * work_topics: n_topics*d doubles; work_chain: p1 ints; work_row: d doubles.
 */
void kvs_unit_kv(const kvs_params* P, int seq, int layer, int kvh, long p0, long p1,
                 uint16_t* out_k, uint16_t* out_v, double* work_topics, int* work_chain, double* work_row) {
  const int d = P->d;
  unit_topics(P, seq, layer, kvh, work_topics);
  unit_chain(P, seq, layer, kvh, p1, work_chain);
  const uint64_t kk = kvs_stream_key(P->seed, seq, layer, kvh, TAG_KNOISE);
  const uint64_t kv = kvs_stream_key(P->seed, seq, layer, kvh, TAG_VALUE);
  for (long p = p0; p < p1; ++p) {
    const double* c = work_topics + (size_t)work_chain[p] * d;
    for (int m = 0; m < d / 2; ++m) {
      double z0, z1;
      normal_pair(kk, (uint64_t)p * (d / 2) + m, &z0, &z1);
      work_row[2 * m] = c[2 * m] + P->sigma_k * z0;
      work_row[2 * m + 1] = c[2 * m + 1] + P->sigma_k * z1;
    }
    rope_row(work_row, d, P->theta, (double)p);
    const double sc = (p < P->n_sink) ? P->sink_scale : 1.0;
    uint16_t* ko = out_k + (size_t)(p - p0) * d;
    for (int i = 0; i < d; ++i) ko[i] = kvs_bf16(sc * work_row[i]);
    uint16_t* vo = out_v + (size_t)(p - p0) * d;
    for (int m = 0; m < d / 2; ++m) {
      double z0, z1;
      normal_pair(kv, (uint64_t)p * (d / 2) + m, &z0, &z1);
      vo[2 * m] = kvs_bf16(z0);
      vo[2 * m + 1] = kvs_bf16(z1);
    }
  }
}

/*
 * Whole cache [B][L][Hkv][p1-p0][d] (bf16 bits) for positions [p0, p1),
 * parallel over units.  Returns 0, or -1 on allocation failure.
 */
#include <stdlib.h>
int kvs_cache(const kvs_params* P, int B, int L, int Hkv, long p0, long p1, uint16_t* K, uint16_t* V) {
  const int units = B * L * Hkv;
  const long rows = p1 - p0;
  int fail = 0;
#pragma omp parallel
  {
    double* wt = (double*)malloc(sizeof(double) * (size_t)P->n_topics * P->d);
    int* wc = (int*)malloc(sizeof(int) * (size_t)(p1 > 0 ? p1 : 1));
    double* wr = (double*)malloc(sizeof(double) * (size_t)P->d);
    if (!wt || !wc || !wr) {
#pragma omp atomic write
      fail = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int u = 0; u < units; ++u) {
        const int b = u / (L * Hkv), l = (u / Hkv) % L, h = u % Hkv;
        kvs_unit_kv(P, b, l, h, p0, p1, K + (size_t)u * rows * P->d, V + (size_t)u * rows * P->d, wt, wc, wr);
      }
    }
    free(wt);
    free(wc);
    free(wr);
  }
  return fail ? -1 : 0;
}

/*
 * Queries [B][L][Hq][d] (bf16 bits) for decode step `step` at position `pos`.
 * Query head h belongs to kv head h / (Hq / Hkv).
 */
int kvs_queries(const kvs_params* P, int B, int L, int Hq, int Hkv, long pos, int step, uint16_t* Q) {
  const int d = P->d, g = Hq / Hkv, T = P->n_topics;
  double* wt = (double*)malloc(sizeof(double) * (size_t)T * d);
  double* row = (double*)malloc(sizeof(double) * (size_t)d);
  if (!wt || !row) {
    free(wt);
    free(row);
    return -1;
  }
  for (int b = 0; b < B; ++b)
    for (int l = 0; l < L; ++l)
      for (int hk = 0; hk < Hkv; ++hk) {
        unit_topics(P, b, l, hk, wt);
        for (int j = 0; j < g; ++j) {
          const int h = hk * g + j;
          const uint64_t kt = kvs_stream_key(P->seed, b, l, (uint64_t)h * 1000003ULL + (uint64_t)step, TAG_QTOPIC);
          const uint64_t kn = kvs_stream_key(P->seed, b, l, (uint64_t)h * 1000003ULL + (uint64_t)step, TAG_QNOISE);
          int pick[3], got = 0;
          uint64_t i = 0;
          const int want = T >= 3 ? 3 : T;
          while (got < want) {
            int t = (int)((1.0 - uniform01(kt, i++)) * T);
            if (t >= T) t = T - 1;
            int dup = 0;
            for (int a = 0; a < got; ++a) dup |= (pick[a] == t);
            if (!dup) pick[got++] = t;
          }
          for (int m = 0; m < d / 2; ++m) {
            double z0, z1;
            normal_pair(kn, (uint64_t)m, &z0, &z1);
            row[2 * m] = P->sigma_q * z0;
            row[2 * m + 1] = P->sigma_q * z1;
          }
          for (int a = 0; a < got; ++a)
            for (int e = 0; e < d; ++e) row[e] += P->q_scale * wt[(size_t)pick[a] * d + e];
          rope_row(row, d, P->theta, (double)pos);
          uint16_t* qo = Q + (((size_t)b * L + l) * Hq + h) * d;
          for (int e = 0; e < d; ++e) qo[e] = kvs_bf16(row[e]);
        }
      }
  free(wt);
  free(row);
  return 0;
}
