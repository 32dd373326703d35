// wi_api.cu -- the C ABI (include/wave_index.h): argument checks, ownership,
// allocation and the order of the kernels of a build and of a decode step.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "wave_index.h"
#include "wi_internal.h"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

#define WI_CUDA(call)                                                                          \
  do {                                                                                         \
    cudaError_t e_ = (call);                                                                   \
    if (e_ != cudaSuccess) {                                                                   \
      cudaGetLastError(); /* clear a non-sticky error so later launch checks stay clean */    \
      return fail(WI_ECUDA, "%s: %s", #call, cudaGetErrorString(e_));                         \
    }                                                                                          \
  } while (0)

int env_int(const char* name, int dflt) {
  const char* s = getenv(name);
  if (!s || !*s) return dflt;
  return atoi(s);
}

}  // namespace

struct wi_index {
  wi_config cfg;
  WiGeom g;
  int device = 0;
  void* K = nullptr;
  void* V = nullptr;
  // index
  void* mu = nullptr;
  float* valsum = nullptr;
  void* valsum16 = nullptr;  // bf16 copy read by decode when the config asks for it
  int* cnt = nullptr;
  int* off = nullptr;
  int* perm = nullptr;
  int* nonempty = nullptr;
  void* appK = nullptr;
  void* appV = nullptr;
  int* app_count = nullptr;
  int appended = 0;
  // decode-time growth (only when max_append >= seg_len): the grown segments' rows and counters
  void* grownK = nullptr;
  void* grownV = nullptr;
  int* grown = nullptr;
  int* kcur = nullptr;
  int grown_host = 0;
  WiGrowBufs gw{};
  long long steps_run = 0;  // decode steps enqueued (host-side count)
  // decode scratch
  WiDecodeBufs b{};
  int* err = nullptr;
  // host-buffer variant staging
  void* q_dev = nullptr;
  void* kn_dev = nullptr;
  void* vn_dev = nullptr;
  float* out_dev = nullptr;
  // ... and, for steps without append from pinned host buffers, the copy-in, the decode chain and
  // the copy-out as one CUDA graph (captured on first use with those buffers)
  cudaStream_t cap_stream = nullptr;
  cudaGraph_t host_graph = nullptr;
  cudaGraphExec_t host_exec = nullptr;
  const void* host_q = nullptr;  // the mapped host buffers the graph reads and writes
  void* host_o = nullptr;
  int host_recaptures = 0;
  bool host_graph_off = false;  // capture failed, or the buffers keep changing: direct launches
  cudaStream_t last_stream = nullptr;
  std::vector<void*> allocs;
  // build timing: events around the whole build and around every assignment launch
  std::vector<cudaEvent_t> build_ev;  // [0] start, [1] end, then (before, after) per assignment
  // decode profiling
  std::vector<cudaEvent_t> prof_ev;  // WI_DECODE_EVENTS per slot
  int prof_slots = 0;
  long long prof_steps = 0;
  // host memory tier (wave buffer), once attached
  WiTierHost* tier = nullptr;
};

int wi_budget(const WiGeom& g, int C) {
  return g.budget_k > 0 ? g.budget_k : (int)std::ceil(g.budget_frac * (double)C);
}

int wi_geom_from_config(const wi_config* c, WiGeom* g, char* msg, size_t msglen) {
#define BAD(...)                          \
  do {                                    \
    snprintf(msg, msglen, __VA_ARGS__);   \
    return WI_EINVAL;                     \
  } while (0)
  if (!c) BAD("config is NULL");
  if (c->batch < 1 || c->layers < 1 || c->n_q_heads < 1 || c->n_kv_heads < 1)
    BAD("batch, layers, n_q_heads, n_kv_heads must be >= 1");
  if (c->n_q_heads % c->n_kv_heads) BAD("n_q_heads (%d) is not a multiple of n_kv_heads (%d)", c->n_q_heads,
                                        c->n_kv_heads);
  if (c->head_dim != 128) BAD("head_dim must be 128 (got %d)", c->head_dim);
  if (c->seg_len < 128 || c->seg_len % 128) BAD("seg_len must be a positive multiple of 128 (got %d)", c->seg_len);
  if (c->n_ctx < c->seg_len || c->n_ctx % c->seg_len) BAD("n_ctx (%lld) must be a positive multiple of seg_len",
                                                          c->n_ctx);
  if (c->clusters_per_seg < 16 || c->clusters_per_seg > 512 || c->clusters_per_seg % 16 ||
      c->seg_len % c->clusters_per_seg)
    BAD("clusters_per_seg must be a multiple of 16 in [16, 512] dividing seg_len (got %d)", c->clusters_per_seg);
  if (c->iters < 1) BAD("iters must be >= 1");
  if (c->n_sink < 0 || c->local_window < 0 || c->n_sink + c->local_window < 1 ||
      c->n_sink + c->local_window >= c->n_ctx)
    BAD("need 1 <= n_sink + local_window < n_ctx");
  if (c->max_append < 0) BAD("max_append must be >= 0");
  if (c->n_ctx + c->max_append >= (1LL << 24)) BAD("n_ctx + max_append must be < 2^24");
  if (c->valsum_bf16 != 0 && c->valsum_bf16 != 1) BAD("valsum_bf16 must be 0 or 1");
  if (c->group_topk != 0 && c->group_topk != 1) BAD("group_topk must be 0 or 1");
  if (c->reserved[0]) BAD("reserved fields must be zero");
  g->vs16 = c->valsum_bf16;
  g->grp = c->group_topk;
  g->U = c->batch * c->layers * c->n_kv_heads;
  g->G = c->n_q_heads / c->n_kv_heads;
  g->S = c->seg_len;
  g->Cs = c->clusters_per_seg;
  g->nseg = (int)(c->n_ctx / c->seg_len);
  // decode-time growth: one more segment per seg_len appended tokens
  g->Gmax = c->max_append / c->seg_len;
  if (((long long)g->nseg + g->Gmax) * g->Cs >= (1LL << 30)) BAD("too many clusters per unit");
  g->Cb = g->nseg * g->Cs;
  g->C = g->Cb + g->Gmax * g->Cs;
  g->n = c->n_ctx;
  g->n_sink = c->n_sink;
  g->W = c->local_window;
  g->n_idx = (int)(c->n_ctx - c->n_sink - c->local_window);
  g->perm_stride = g->n_idx + g->Gmax * g->S;
  g->iters = c->iters;
  g->max_append = c->max_append;
  g->budget_frac = c->budget_frac;
  g->budget_k = c->budget_k;
  const long long k = wi_budget(*g, g->Cb);
  if (k < 1 || k > g->Cb) BAD("retrieval budget k = %lld must be in [1, C = %d]", k, g->Cb);
  g->kbuild = (int)k;
  g->kmax = wi_budget(*g, g->C);
  if (g->G > 8) {
    snprintf(msg, msglen, "query heads per kv head must be <= 8 (got %d)", g->G);
    return WI_EUNSUPPORTED;
  }
  if (g->kmax > 4096) {
    snprintf(msg, msglen, "retrieval budget must be <= 4096 clusters (got %d)", g->kmax);
    return WI_EUNSUPPORTED;
  }
  if (g->C > 65536) {
    snprintf(msg, msglen, "at most 65536 clusters per kv head, grown segments included (got %d)", g->C);
    return WI_EUNSUPPORTED;
  }
  if (g->S > 16384) {
    snprintf(msg, msglen, "seg_len must be <= 16384 (got %d)", g->S);
    return WI_EUNSUPPORTED;
  }
  return WI_OK;
#undef BAD
}

namespace {

int alloc(wi_index* ix, void** p, size_t bytes) {
  if (bytes == 0) bytes = 16;
  // fault injection for the error path: WI_FAIL_ALLOC_AT=n makes the n-th device allocation of every
  // index report out-of-memory (nothing is allocated)
  const int fail_at = env_int("WI_FAIL_ALLOC_AT", 0);
  if (fail_at > 0 && ix->allocs.size() + 1 == (size_t)fail_at)
    return fail(WI_ENOMEM, "device allocation %d refused (WI_FAIL_ALLOC_AT)", fail_at);
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(WI_ENOMEM, "cudaMalloc(%zu bytes) failed: %s", bytes, cudaGetErrorString(e));
  }
  ix->allocs.push_back(*p);
  return WI_OK;
}

void destroy(wi_index* ix) {
  if (!ix) return;
  if (ix->tier) wi_tier_destroy(ix->tier);
  if (ix->host_exec) cudaGraphExecDestroy(ix->host_exec);
  if (ix->host_graph) cudaGraphDestroy(ix->host_graph);
  if (ix->cap_stream) cudaStreamDestroy(ix->cap_stream);
  for (cudaEvent_t e : ix->prof_ev) cudaEventDestroy(e);
  for (cudaEvent_t e : ix->build_ev) cudaEventDestroy(e);
  for (void* p : ix->allocs) cudaFree(p);
  delete ix;
}

// Index storage, decode scratch and staging.
int alloc_index(wi_index* ix, cudaStream_t st) {
  const WiGeom& g = ix->g;
  const size_t U = g.U, C = g.C, G = g.G;
  int rc;
#define A(ptr, bytes)                                                              \
  if ((rc = alloc(ix, reinterpret_cast<void**>(&(ptr)), (bytes))) != WI_OK) return rc
  A(ix->mu, U * C * 128 * 2);
  A(ix->valsum, U * C * 128 * 4);
  if (g.vs16) A(ix->valsum16, U * C * 128 * 2);
  A(ix->cnt, U * C * 4);
  A(ix->off, U * (C + 1) * 4);
  A(ix->perm, U * (size_t)g.perm_stride * 4);
  A(ix->nonempty, U * 4);
  const size_t app = (size_t)(g.max_append > 0 ? g.max_append : 1);
  A(ix->appK, U * app * 128 * 2);
  A(ix->appV, U * app * 128 * 2);
  A(ix->app_count, 4);
  A(ix->err, 4);
  A(ix->grown, 4);
  A(ix->kcur, 4);
  if (g.Gmax > 0) {
    // room for the segments that appends may add; their clusters stay empty until grown
    const size_t S = g.S, Cs = g.Cs, rows = (size_t)g.Gmax * U * S;
    A(ix->grownK, rows * 128 * 2);
    A(ix->grownV, rows * 128 * 2);
    WiGrowBufs& w = ix->gw;
    A(w.chat, U * Cs * 128 * 2);
    A(w.assign, U * S * 4);
    A(w.seg_counts, U * Cs * 4);
    A(w.seg_offsets, U * (Cs + 1) * 4);
    A(w.slots, U * S * 4);
    A(w.mu, U * Cs * 128 * 2);
    A(w.valsum, U * Cs * 128 * 4);
    A(w.cnt, U * Cs * 4);
    A(w.off, U * (Cs + 1) * 4);
    A(w.perm, U * S * 4);
    A(w.nonempty, U * 4);
    A(w.tK, U * S * 128 * 2);
    A(w.tV, U * S * 128 * 2);
    WI_CUDA(cudaMemsetAsync(ix->mu, 0, U * C * 128 * 2, st));
    WI_CUDA(cudaMemsetAsync(ix->valsum, 0, U * C * 128 * 4, st));
    WI_CUDA(cudaMemsetAsync(ix->cnt, 0, U * C * 4, st));
    WI_CUDA(cudaMemsetAsync(ix->off, 0, U * (C + 1) * 4, st));
    WI_CUDA(cudaMemsetAsync(ix->perm, 0xFF, U * (size_t)g.perm_stride * 4, st));
  }
  WiDecodeBufs& b = ix->b;
  int sms = 0;
  WI_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, ix->device));
  const int tiles = (int)((C + 15) / 16);  // score_estimate splits a unit's clusters on multiples of 16
  // scores: at most one wave of one CTA per SM (a partial second wave of a few CTAs would double
  // the kernel's time)
  int p1 = env_int("WI_D1_CTAS_PER_UNIT", 0);
  if (p1 <= 0) p1 = (int)(sms / U);
  if (p1 > tiles) p1 = tiles;
  if (p1 > 256) p1 = 256;
  if (p1 < 1) p1 = 1;
  b.p1 = p1;
  // the estimation CTAs share a launch with the U*G top-k CTAs (one CTA per SM each)
  int pe = env_int("WI_ESTIMATE_CTAS_PER_UNIT", 0);
  // with many heads the top-k CTAs fill the SMs beside the estimation CTAs, which need about 0.6 of
  // the SMs to keep HBM streaming: round(0.6 * SMs / U) per unit
  if (pe <= 0) pe = (size_t)U * G < (size_t)sms ? (int)((sms - U * G) / U) : (int)((6 * (size_t)sms + 5 * U) / (10 * U));
  if (pe > tiles) pe = tiles;
  if (pe > 256) pe = 256;
  if (pe < 1) pe = 1;
  b.p_es = pe;
  // estimation CTAs that fit in one wave go first, so their stream overlaps the top-k CTAs
  const int ef = env_int("WI_ESTIMATE_FIRST", -1);
  b.est_first = ef >= 0 ? (ef != 0) : ((size_t)U * pe < (size_t)sms);
  // when the top-k and estimation CTAs all fit in one wave, the top-k chain is the step's critical
  // path and its loads queue behind the estimation stream: two stages in flight per estimation CTA
  // (instead of three) still stream the value sums within the top-k's time
  const int esd = env_int("WI_ESTIMATE_DEPTH", 0);
  b.es_depth = esd == 2 || esd == 3 ? esd : ((size_t)U * (G + pe) <= (size_t)sms ? 2 : 3);
  // exact attention: (splits + 1 steady CTA) per head.  Few heads: fill two CTAs per SM in one wave
  // (the step is a latency chain); many heads: about two waves of split CTAs, so that the heads'
  // unequal row counts balance across the SMs
  int ns = env_int("WI_D3_SPLITS", 0);
  const size_t heads = U * G, slots = 2 * (size_t)sms;
  if (ns <= 0) ns = heads * 2 <= slots ? (int)(slots / heads) - 1 : (int)((2 * slots + heads - 1) / heads);
  if (ns > 64) ns = 64;
  if (ns < 1) ns = 1;
  b.nsplit = ns;
  // exact stages: 32 rows when every exact CTA is resident at once (two per SM), else 64 rows
  const int d3r = env_int("WI_D3_STAGE_ROWS", 0);
  b.d3_rows = d3r == 32 || d3r == 64 ? d3r : (heads * (size_t)(ns + 1) <= slots ? 32 : 64);
  // dense comparator: row ranges per unit such that the U * ranges CTAs come closest to whole waves
  // (a partial last wave idles SMs), at least 1024 rows each; the fewest ranges among equals
  int ds = 1;
  {
    const long long slots = (long long)wi_dense_ctas_per_sm(G) * sms;
    double best = -1.0;
    for (int d = 1; d <= 256; ++d) {
      if (d > 1 && g.n / d < 1024) break;
      const long long ctas = (long long)U * d, waves = (ctas + slots - 1) / slots;
      const double eff = (double)ctas / (double)(waves * slots);
      if (eff > best + 1e-9) { best = eff; ds = d; }
    }
  }
  b.dsplits = ds;
  A(b.dpart, U * G * (size_t)ds * WI_PART * 4);
  A(b.dticket, U * 4);
  const size_t GK = G + (size_t)g.grp;  // key rows per unit (the summed-score row, if any)
  A(b.scores, U * GK * C * 4);
  A(b.part1, U * G * (size_t)b.p_es * WI_PART * 4);
  A(b.sel, U * G * (size_t)g.kmax * 4);
  A(b.selcnt, U * G * 4);
  A(b.subpart, U * G * WI_PART * 4);
  A(b.runs, U * G * (size_t)g.kmax * 16);
  A(b.splits, U * G * (size_t)(b.nsplit + 2) * 16);
  A(b.sruns, U * G * (size_t)(b.nsplit + 1) * 32 * 16);
  A(b.part3, U * G * (size_t)(b.nsplit + 1) * WI_PART * 4);
  A(b.subn, U * G * (size_t)(b.nsplit + 1) * WI_PART * 4);
  A(b.ticket, U * G * 4);
  A(b.kmaxp, U * (size_t)b.p1 * GK * 4);
  A(b.rows_total, 8);
  A(ix->q_dev, U * G * 128 * 2);
  A(ix->out_dev, U * G * 128 * 4);
  A(ix->kn_dev, U * 128 * 2);
  A(ix->vn_dev, U * 128 * 2);
#undef A
  if (!wi_encode_rows_sw128(&b.map_mu, ix->mu, (unsigned long long)U * C, 128))
    return fail(WI_EUNSUPPORTED, "could not encode the tensor map of the centroid table");
  b.mu = ix->mu;
  b.valsum = ix->valsum;
  b.valsum16 = ix->valsum16;
  b.cnt = ix->cnt;
  b.off = ix->off;
  b.nonempty = ix->nonempty;
  b.K = ix->K;
  b.V = ix->V;
  b.appK = ix->appK;
  b.appV = ix->appV;
  b.app_count = ix->app_count;
  b.grownK = ix->grownK;
  b.grownV = ix->grownV;
  b.grown = ix->grown;
  b.kcur = ix->kcur;
  b.err = ix->err;
  WI_CUDA(cudaMemsetAsync(ix->app_count, 0, 4, st));
  WI_CUDA(cudaMemsetAsync(ix->grown, 0, 4, st));
  WI_CUDA(wi_launch_set_int(ix->kcur, g.kbuild, st));
  WI_CUDA(cudaMemsetAsync(ix->err, 0, 4, st));
  WI_CUDA(cudaMemsetAsync(b.selcnt, 0, U * G * 4, st));
  WI_CUDA(cudaMemsetAsync(b.ticket, 0, U * G * 4, st));
  WI_CUDA(cudaMemsetAsync(b.dticket, 0, U * 4, st));

  WI_CUDA(cudaMemsetAsync(b.rows_total, 0, 8, st));
  return WI_OK;
}

int new_index(const wi_config* cfg, void* k, void* v, wi_index** out, wi_index** ixp) {
  if (!out) return fail(WI_EINVAL, "out is NULL");
  *out = nullptr;
  WiGeom g;
  int rc = wi_geom_from_config(cfg, &g, g_err, sizeof(g_err));
  if (rc != WI_OK) return rc;
  if (!k || !v) return fail(WI_EINVAL, "k and v must be non-NULL device pointers");
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15)
    return fail(WI_EINVAL, "k and v must be 16-byte aligned");
  wi_index* ix = new (std::nothrow) wi_index();
  if (!ix) return fail(WI_ENOMEM, "host allocation failed");
  ix->cfg = *cfg;
  ix->g = g;
  ix->K = k;
  ix->V = v;
  cudaGetDevice(&ix->device);
  *ixp = ix;
  return WI_OK;
}

// Scratch rows of the in-place permutation: whole units, at most 1 GiB each for K and V.
int perm_scratch(const WiGeom& g, void** tK, void** tV, int* nb, cudaStream_t st) {
  const size_t per_unit = (size_t)(g.n_idx > 0 ? g.n_idx : 1) * 128 * 2;
  const size_t cap = (size_t)1 << 30;
  *nb = (int)(cap / per_unit);
  if (*nb < 1) *nb = 1;
  if (*nb > g.U) *nb = g.U;
  *tK = *tV = nullptr;
  if (cudaMallocAsync(tK, per_unit * *nb, st) != cudaSuccess || cudaMallocAsync(tV, per_unit * *nb, st) != cudaSuccess) {
    cudaGetLastError();
    if (*tK) cudaFreeAsync(*tK, st);
    *tK = nullptr;
    return fail(WI_ENOMEM, "permutation scratch (%zu bytes) allocation failed", 2 * per_unit * *nb);
  }
  return WI_OK;
}

// Permute the clustered rows of K, V by ix->perm, through bounded scratch.
int permute_kv(wi_index* ix, cudaStream_t st) {
  const WiGeom& g = ix->g;
  if (g.n_idx == 0) return WI_OK;
  void *tK = nullptr, *tV = nullptr;
  int nb = 0;
  int rc = perm_scratch(g, &tK, &tV, &nb, st);
  if (rc != WI_OK) return rc;
  cudaError_t e = cudaSuccess;
  for (int u0 = 0; u0 < g.U && e == cudaSuccess; u0 += nb) {
    const int nu = (g.U - u0) < nb ? (g.U - u0) : nb;
    e = wi_launch_permute(g, ix->K, ix->V, ix->perm, tK, tV, u0, nu, st);
  }
  cudaFreeAsync(tK, st);
  cudaFreeAsync(tV, st);
  if (e != cudaSuccess) return fail(WI_ECUDA, "permutation: %s", cudaGetErrorString(e));
  return WI_OK;
}

struct BuildScratch {
  void* chat = nullptr;
  int32_t* assign = nullptr;
  int* seg_counts = nullptr;
  int* seg_offsets = nullptr;
  int* slots = nullptr;
};

int scratch_alloc(const WiGeom& g, BuildScratch* s, cudaStream_t st) {
  const size_t SU = (size_t)g.U * g.nseg;
  const size_t rows = (size_t)g.U * g.n;
  cudaError_t e = cudaSuccess;
  e = cudaMallocAsync(&s->chat, SU * g.Cs * 128 * 2, st);
  if (e == cudaSuccess) e = cudaMallocAsync(reinterpret_cast<void**>(&s->assign), rows * 4, st);
  if (e == cudaSuccess) e = cudaMallocAsync(reinterpret_cast<void**>(&s->seg_counts), SU * g.Cs * 4, st);
  if (e == cudaSuccess) e = cudaMallocAsync(reinterpret_cast<void**>(&s->seg_offsets), SU * (g.Cs + 1) * 4, st);
  if (e == cudaSuccess) e = cudaMallocAsync(reinterpret_cast<void**>(&s->slots), SU * g.S * 4, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(WI_ENOMEM, "build scratch allocation failed: %s", cudaGetErrorString(e));
  }
  return WI_OK;
}

void scratch_free(BuildScratch* s, cudaStream_t st) {
  void* ps[] = {s->chat, s->assign, s->seg_counts, s->seg_offsets, s->slots};
  for (void* p : ps)
    if (p) cudaFreeAsync(p, st);
}

#define WI_LAUNCH(call)                                                                             \
  do {                                                                                              \
    cudaError_t e_ = (call);                                                                        \
    if (e_ != cudaSuccess) {                                                                        \
      cudaGetLastError();                                                                           \
      rc = fail(WI_ECUDA, "%s: %s", #call, cudaGetErrorString(e_));                                 \
      goto done;                                                                                    \
    }                                                                                               \
  } while (0)

}  // namespace

void wi_set_error(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }

extern "C" {

const char* wi_last_error(void) { return g_err; }

static int build_index_impl(const wi_config* cfg, void* k, void* v, const void* init_centroids, void* stream,
                            wi_index** out) {
  g_err[0] = 0;
  wi_index* ix = nullptr;
  int rc = new_index(cfg, k, v, out, &ix);
  if (rc != WI_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ix->last_stream = st;
  const WiGeom& g = ix->g;
  BuildScratch s;
  void *tK = nullptr, *tV = nullptr;
  int nb = 0;
  // every allocation of the build first: the build's kernels then run back to back
  if ((rc = alloc_index(ix, st)) != WI_OK || (rc = scratch_alloc(g, &s, st)) != WI_OK ||
      (rc = perm_scratch(g, &tK, &tV, &nb, st)) != WI_OK) {
    scratch_free(&s, st);
    destroy(ix);
    return rc;
  }
  for (int i = 0; i < 2 + 2 * g.iters; ++i) {
    cudaEvent_t e;
    WI_LAUNCH(cudaEventCreate(&e));
    ix->build_ev.push_back(e);
  }
  WI_LAUNCH(cudaEventRecord(ix->build_ev[0], st));
  if (init_centroids)
    WI_LAUNCH(cudaMemcpyAsync(s.chat, init_centroids, (size_t)g.U * g.nseg * g.Cs * 128 * 2, cudaMemcpyDefault, st));
  else
    WI_LAUNCH(wi_launch_init_centroids(g, k, s.chat, st));
  for (int t = 0; t < g.iters; ++t) {
    WI_LAUNCH(cudaEventRecord(ix->build_ev[2 + 2 * t], st));
    WI_LAUNCH(wi_launch_assign(g, k, s.chat, s.assign, ix->err, st));
    WI_LAUNCH(cudaEventRecord(ix->build_ev[3 + 2 * t], st));
    WI_LAUNCH(wi_launch_segment_sort(g, s.assign, s.seg_counts, s.seg_offsets, s.slots, ix->err, st));
    if (t + 1 < g.iters)
      WI_LAUNCH(wi_launch_centroid_update(g, k, s.seg_counts, s.seg_offsets, s.slots, s.chat, st));
  }
  // the final index and the in-place permutation, one pass over K and V for both
  WI_LAUNCH(wi_launch_reduce_permute(g, k, v, s.seg_counts, s.seg_offsets, s.slots, ix->mu, ix->valsum, ix->cnt,
                                     ix->off, ix->perm, ix->nonempty, tK, tV, nb, st));
  if (g.vs16) WI_LAUNCH(wi_launch_to_bf16(ix->valsum, ix->valsum16, (long long)g.U * g.C * 128, st));
  cudaFreeAsync(tK, st);
  cudaFreeAsync(tV, st);
  tK = tV = nullptr;
  scratch_free(&s, st);
  s = BuildScratch();
  WI_LAUNCH(cudaEventRecord(ix->build_ev[1], st));
  *out = ix;
  return WI_OK;
done:
  if (tK) cudaFreeAsync(tK, st);
  if (tV) cudaFreeAsync(tV, st);
  scratch_free(&s, st);
  cudaStreamSynchronize(st);
  destroy(ix);
  return rc;
}

static int index_import_impl(const wi_config* cfg, void* k, void* v, const int32_t* counts, const int32_t* perm,
                    const uint16_t* mu, const float* valsum, void* stream, wi_index** out) {
  g_err[0] = 0;
  wi_index* ix = nullptr;
  int rc = new_index(cfg, k, v, out, &ix);
  if (rc != WI_OK) return rc;
  if (!counts || !perm || !mu || !valsum) {
    destroy(ix);
    return fail(WI_EINVAL, "counts, perm, mu and valsum must be non-NULL");
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ix->last_stream = st;
  const WiGeom& g = ix->g;
  // the caller's arrays hold the build's Cb clusters; the index's rows have room for C (grown segments)
  const size_t U = g.U, Cb = g.Cb, C = g.C, PS = g.perm_stride;
  std::vector<int32_t> hc(U * Cb), hp(U * (size_t)g.n_idx), hoff(U * (C + 1), (int)(g.n - g.W)), hne(U, 0);
  std::vector<int32_t> hcC(U * C, 0), hpP(U * PS, -1);
  std::vector<unsigned char> seen;
  if (cudaMemcpy(hc.data(), counts, hc.size() * 4, cudaMemcpyDefault) != cudaSuccess ||
      cudaMemcpy(hp.data(), perm, hp.size() * 4, cudaMemcpyDefault) != cudaSuccess) {
    cudaGetLastError();
    destroy(ix);
    return fail(WI_EINVAL, "counts / perm are not readable (host or device memory expected)");
  }
  for (size_t u = 0; u < U; ++u) {
    long long run = g.n_sink;
    seen.assign((size_t)g.n, 0);
    for (size_t c = 0; c < Cb; ++c) {
      const int m = hc[u * Cb + c];
      if (m < 0) { destroy(ix); return fail(WI_EINVAL, "negative count (unit %zu, cluster %zu)", u, c); }
      hcC[u * C + c] = m;
      hoff[u * (C + 1) + c] = (int)run;
      const int s = (int)(c / g.Cs);
      for (int t = 0; t < m; ++t) {
        const long long slot = run + t - g.n_sink;
        if (slot >= g.n_idx) { destroy(ix); return fail(WI_EINVAL, "counts exceed the clustered tokens (unit %zu)", u); }
        const long long p = hp[u * g.n_idx + slot];
        if (p < g.n_sink || p >= g.n - g.W || p / g.S != s || seen[p]) {
          destroy(ix);
          return fail(WI_EINVAL, "perm is not a bijection on the clustered positions of each segment (unit %zu)", u);
        }
        seen[p] = 1;
      }
      run += m;
      if (m > 0) hne[u]++;
    }
    if (run != g.n - g.W) { destroy(ix); return fail(WI_EINVAL, "counts of unit %zu do not cover the clustered tokens", u); }
    std::copy(hp.begin() + u * g.n_idx, hp.begin() + (u + 1) * g.n_idx, hpP.begin() + u * PS);
  }
  if ((rc = alloc_index(ix, st)) != WI_OK) { destroy(ix); return rc; }
  WI_LAUNCH(cudaMemcpyAsync(ix->cnt, hcC.data(), hcC.size() * 4, cudaMemcpyHostToDevice, st));
  WI_LAUNCH(cudaMemcpyAsync(ix->perm, hpP.data(), hpP.size() * 4, cudaMemcpyHostToDevice, st));
  WI_LAUNCH(cudaMemcpyAsync(ix->off, hoff.data(), hoff.size() * 4, cudaMemcpyHostToDevice, st));
  WI_LAUNCH(cudaMemcpyAsync(ix->nonempty, hne.data(), hne.size() * 4, cudaMemcpyHostToDevice, st));
  WI_LAUNCH(cudaMemcpy2DAsync(ix->mu, C * 128 * 2, mu, Cb * 128 * 2, Cb * 128 * 2, U, cudaMemcpyDefault, st));
  WI_LAUNCH(cudaMemcpy2DAsync(ix->valsum, C * 128 * 4, valsum, Cb * 128 * 4, Cb * 128 * 4, U, cudaMemcpyDefault,
                              st));
  if (g.vs16) WI_LAUNCH(wi_launch_to_bf16(ix->valsum, ix->valsum16, (long long)U * C * 128, st));
  if ((rc = permute_kv(ix, st)) != WI_OK) goto done;
  // the host vectors above are pageable: finish the copies before they go away
  WI_LAUNCH(cudaStreamSynchronize(st));
  *out = ix;
  return WI_OK;
done:
  cudaStreamSynchronize(st);
  destroy(ix);
  return rc;
}

int wi_index_export(const wi_index* ix, int32_t* counts, int32_t* offsets, int32_t* perm, uint16_t* mu,
                    float* valsum, void* stream) {
  g_err[0] = 0;
  if (!ix) return fail(WI_EINVAL, "index is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WiGeom& g = ix->g;
  const size_t U = g.U, C = g.C;
  if (counts) WI_CUDA(cudaMemcpyAsync(counts, ix->cnt, U * C * 4, cudaMemcpyDefault, st));
  if (offsets) WI_CUDA(cudaMemcpyAsync(offsets, ix->off, U * (C + 1) * 4, cudaMemcpyDefault, st));
  if (perm) WI_CUDA(cudaMemcpyAsync(perm, ix->perm, U * (size_t)g.perm_stride * 4, cudaMemcpyDefault, st));
  if (mu) WI_CUDA(cudaMemcpyAsync(mu, ix->mu, U * C * 128 * 2, cudaMemcpyDefault, st));
  if (valsum) WI_CUDA(cudaMemcpyAsync(valsum, ix->valsum, U * C * 128 * 4, cudaMemcpyDefault, st));
  return WI_OK;
}

int wi_decode_step(wi_index* ix, const void* q, const void* k_new, const void* v_new, float* out, void* stream) {
  g_err[0] = 0;
  if (!ix || !q || !out) return fail(WI_EINVAL, "index, q and out must be non-NULL");
  if ((k_new == nullptr) != (v_new == nullptr)) return fail(WI_EINVAL, "k_new and v_new must both be set or both NULL");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
    return fail(WI_EINVAL, "q, k_new and v_new must be 16-byte aligned");
  if (k_new && ix->appended >= ix->g.max_append)
    return fail(WI_EFULL, "append buffer full (%d tokens)", ix->g.max_append);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (ix->tier) {  // the tier's replacement rounds enqueue work of their own between steps
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    WI_CUDA(cudaStreamIsCapturing(st, &cs));
    if (cs != cudaStreamCaptureStatusNone)
      return fail(WI_EUNSUPPORTED, "an index with a host memory tier cannot be captured in a graph");
    ix->b.tier.step = (int)ix->steps_run;
  }
  ix->last_stream = st;
  const cudaEvent_t* ev = nullptr;
  if (ix->prof_slots > 0) {
    ev = ix->prof_ev.data() + (size_t)(ix->prof_steps % ix->prof_slots) * WI_DECODE_EVENTS;
    ix->prof_steps++;
  }
  cudaError_t e = wi_launch_decode(ix->g, ix->b, q, out, st, ev);
  if (e != cudaSuccess) return fail(WI_ECUDA, "decode launch: %s", cudaGetErrorString(e));
  if (ix->tier) {
    char msg[320];
    const int rc = wi_tier_after_step(ix->tier, ix->steps_run, st, msg, sizeof(msg));
    if (rc != WI_OK) return fail(rc, "%s", msg);
  }
  ix->steps_run++;
  if (k_new) {
    const WiGeom& g = ix->g;
    e = wi_launch_append(g, ix->b, k_new, v_new, ix->appended, st);
    if (e != cudaSuccess) return fail(WI_ECUDA, "append launch: %s", cudaGetErrorString(e));
    ix->appended++;
    // decode-time index maintenance: once the local window holds W + seg_len rows, its oldest
    // seg_len rows become one more segment (every seg_len appended tokens)
    if (ix->grown_host < g.Gmax && ix->appended == (ix->grown_host + 1) * g.S) {
      const int gi = ix->grown_host;
      e = wi_launch_grow(g, ix->b, ix->gw, ix->mu, ix->valsum, ix->valsum16, ix->cnt, ix->off, ix->perm,
                         ix->nonempty, gi, wi_budget(g, g.Cb + (gi + 1) * g.Cs), ix->err, st);
      if (e != cudaSuccess) return fail(WI_ECUDA, "index growth launch: %s", cudaGetErrorString(e));
      ix->grown_host++;
    }
  }
  return WI_OK;
}

int wi_decode_kernel(wi_index* ix, int kernel, const void* q, float* out, void* stream) {
  g_err[0] = 0;
  if (!ix || !q || !out) return fail(WI_EINVAL, "index, q and out must be non-NULL");
  if (kernel < 0 || kernel >= WI_DECODE_KERNELS) return fail(WI_EINVAL, "kernel must be in [0, %d)", WI_DECODE_KERNELS);
  if (reinterpret_cast<uintptr_t>(q) & 15) return fail(WI_EINVAL, "q must be 16-byte aligned");
  if (ix->steps_run == 0)
    return fail(WI_EINVAL, "run one whole decode step on this index first");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ix->last_stream = st;
  cudaError_t e = wi_launch_decode(ix->g, ix->b, q, out, st, nullptr, 1u << kernel);
  if (e != cudaSuccess) return fail(WI_ECUDA, "decode kernel launch: %s", cudaGetErrorString(e));
  return WI_OK;
}

int wi_dense_decode(wi_index* ix, const void* q, float* out, void* stream) {
  g_err[0] = 0;
  if (!ix || !q || !out) return fail(WI_EINVAL, "index, q and out must be non-NULL");
  if (ix->tier) return fail(WI_EUNSUPPORTED, "full attention reads the caller's K and V, which a host memory tier releases");
  if (reinterpret_cast<uintptr_t>(q) & 15) return fail(WI_EINVAL, "q must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ix->last_stream = st;
  cudaError_t e = wi_launch_dense(ix->g, ix->b, q, out, st);
  if (e != cudaSuccess) return fail(WI_ECUDA, "dense decode launch: %s", cudaGetErrorString(e));
  return WI_OK;
}

// The device address of page-locked host memory mapped into the device's address space, or null.
static void* mapped_host(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

static void drop_host_graph(wi_index* ix) {
  if (ix->host_exec) cudaGraphExecDestroy(ix->host_exec);
  if (ix->host_graph) cudaGraphDestroy(ix->host_graph);
  ix->host_exec = nullptr;
  ix->host_graph = nullptr;
}

// Capture the host-buffer step as a graph: a copy kernel reads the query from mapped host memory,
// the decode chain runs and its merge writes the output straight into mapped host memory (no DMA
// setup per step).  False if the runtime refuses (the caller then launches directly).
static bool capture_host_graph(wi_index* ix, const void* qd, void* od, size_t qb, size_t ob) {
  if (!ix->cap_stream && cudaStreamCreateWithFlags(&ix->cap_stream, cudaStreamNonBlocking) != cudaSuccess)
    return false;
  cudaStream_t cs = ix->cap_stream;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) return false;
  (void)ob;
  bool ok = wi_launch_copy16(qd, ix->q_dev, qb, cs) == cudaSuccess &&
            wi_launch_decode(ix->g, ix->b, ix->q_dev, static_cast<float*>(od), cs, nullptr) == cudaSuccess;
  cudaGraph_t graph = nullptr;
  ok = cudaStreamEndCapture(cs, &graph) == cudaSuccess && ok && graph;
  cudaGraphExec_t exec = nullptr;
  if (!ok || cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    return false;
  }
  ix->host_graph = graph;
  ix->host_exec = exec;
  ix->host_q = qd;
  ix->host_o = od;
  return true;
}

int wi_decode_step_host(wi_index* ix, const void* q_host, const void* k_new_host, const void* v_new_host,
                        float* out_host, void* stream) {
  g_err[0] = 0;
  if (!ix || !q_host || !out_host) return fail(WI_EINVAL, "index, q and out must be non-NULL");
  if ((k_new_host == nullptr) != (v_new_host == nullptr))
    return fail(WI_EINVAL, "k_new and v_new must both be set or both NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WiGeom& g = ix->g;
  const size_t qb = (size_t)g.U * g.G * 128 * 2, kb = (size_t)g.U * 128 * 2, ob = (size_t)g.U * g.G * 128 * 4;
  void* qd = nullptr;
  void* od = nullptr;
  if (!k_new_host && ix->prof_slots == 0 && !ix->host_graph_off && !ix->tier && (qd = mapped_host(q_host)) &&
      (od = mapped_host(out_host)) && ((reinterpret_cast<uintptr_t>(qd) | reinterpret_cast<uintptr_t>(od)) & 15) == 0) {
    if (ix->host_exec && (ix->host_q != qd || ix->host_o != od)) {  // other buffers: capture again
      drop_host_graph(ix);
      if (++ix->host_recaptures > 4) ix->host_graph_off = true;  // buffers keep changing: stop capturing
    }
    if (!ix->host_graph_off && !ix->host_exec && !capture_host_graph(ix, qd, od, qb, ob)) {
      cudaGetLastError();
      ix->host_graph_off = true;
    }
    if (ix->host_exec && !ix->host_graph_off) {
      ix->last_stream = st;
      WI_CUDA(cudaGraphLaunch(ix->host_exec, st));
      WI_CUDA(cudaStreamSynchronize(st));
      return WI_OK;
    }
  }
  WI_CUDA(cudaMemcpyAsync(ix->q_dev, q_host, qb, cudaMemcpyHostToDevice, st));
  if (k_new_host) {
    WI_CUDA(cudaMemcpyAsync(ix->kn_dev, k_new_host, kb, cudaMemcpyHostToDevice, st));
    WI_CUDA(cudaMemcpyAsync(ix->vn_dev, v_new_host, kb, cudaMemcpyHostToDevice, st));
  }
  int rc = wi_decode_step(ix, ix->q_dev, k_new_host ? ix->kn_dev : nullptr, k_new_host ? ix->vn_dev : nullptr,
                          ix->out_dev, stream);
  if (rc != WI_OK) return rc;
  WI_CUDA(cudaMemcpyAsync(out_host, ix->out_dev, ob, cudaMemcpyDeviceToHost, st));
  WI_CUDA(cudaStreamSynchronize(st));
  return WI_OK;
}

int wi_last_selection(const wi_index* ix, int32_t* ids, int32_t* counts, void* stream) {
  g_err[0] = 0;
  if (!ix || !ids) return fail(WI_EINVAL, "index and ids must be non-NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WiGeom& g = ix->g;
  WI_CUDA(cudaMemcpyAsync(ids, ix->b.sel, (size_t)g.U * g.G * g.kmax * 4, cudaMemcpyDefault, st));
  if (counts) WI_CUDA(cudaMemcpyAsync(counts, ix->b.selcnt, (size_t)g.U * g.G * 4, cudaMemcpyDefault, st));
  return WI_OK;
}

int wi_index_shape(const wi_index* ix, int* units, int* clusters, int* k_max, int* group, int* appended) {
  g_err[0] = 0;
  if (!ix) return fail(WI_EINVAL, "index is NULL");
  if (units) *units = ix->g.U;
  if (clusters) *clusters = ix->g.C;
  if (k_max) *k_max = ix->g.kmax;
  if (group) *group = ix->g.G;
  if (appended) *appended = ix->appended;
  return WI_OK;
}

int wi_decode_layout(const wi_index* ix, int* score_ctas, int* estimate_ctas, int* exact_splits) {
  g_err[0] = 0;
  if (!ix) return fail(WI_EINVAL, "index is NULL");
  if (score_ctas) *score_ctas = ix->b.p1;
  if (estimate_ctas) *estimate_ctas = ix->b.p_es;
  if (exact_splits) *exact_splits = ix->b.nsplit;
  return WI_OK;
}

int wi_kmeans_step(const wi_config* cfg, const void* k, const void* centroids, int32_t* assign, void* new_centroids,
                   void* stream) {
  g_err[0] = 0;
  WiGeom g;
  int rc = wi_geom_from_config(cfg, &g, g_err, sizeof(g_err));
  if (rc != WI_OK) return rc;
  if (!k || !centroids || !assign || !new_centroids)
    return fail(WI_EINVAL, "k, centroids, assign and new_centroids must be non-NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  BuildScratch s;
  int* err = nullptr;
  if ((rc = scratch_alloc(g, &s, st)) != WI_OK) {
    scratch_free(&s, st);
    return rc;
  }
  if (cudaMallocAsync(reinterpret_cast<void**>(&err), 4, st) != cudaSuccess) {
    cudaGetLastError();
    scratch_free(&s, st);
    return fail(WI_ENOMEM, "allocation failed");
  }
  const size_t cb = (size_t)g.U * g.nseg * g.Cs * 128 * 2;
  WI_LAUNCH(cudaMemsetAsync(err, 0, 4, st));
  WI_LAUNCH(cudaMemcpyAsync(s.chat, centroids, cb, cudaMemcpyDeviceToDevice, st));
  WI_LAUNCH(wi_launch_assign(g, k, s.chat, assign, err, st));
  WI_LAUNCH(wi_launch_segment_sort(g, assign, s.seg_counts, s.seg_offsets, s.slots, err, st));
  WI_LAUNCH(wi_launch_centroid_update(g, k, s.seg_counts, s.seg_offsets, s.slots, s.chat, st));
  WI_LAUNCH(cudaMemcpyAsync(new_centroids, s.chat, cb, cudaMemcpyDeviceToDevice, st));
  {
    int herr = 0;
    WI_LAUNCH(cudaMemcpyAsync(&herr, err, 4, cudaMemcpyDeviceToHost, st));
    WI_LAUNCH(cudaStreamSynchronize(st));
    if (herr) rc = fail(WI_EDEVICE, "device invariant violated (flags 0x%x)", herr);
  }
done:
  scratch_free(&s, st);
  if (err) cudaFreeAsync(err, st);
  return rc;
}

int wi_init_centroids(const wi_config* cfg, const void* k, void* centroids, void* stream) {
  g_err[0] = 0;
  WiGeom g;
  int rc = wi_geom_from_config(cfg, &g, g_err, sizeof(g_err));
  if (rc != WI_OK) return rc;
  if (!k || !centroids) return fail(WI_EINVAL, "k and centroids must be non-NULL");
  WI_CUDA(wi_launch_init_centroids(g, k, centroids, static_cast<cudaStream_t>(stream)));
  return WI_OK;
}

static int profile_begin_impl(wi_index* ix, int max_steps) {
  g_err[0] = 0;
  if (!ix || max_steps < 0) return fail(WI_EINVAL, "index is NULL or max_steps < 0");
  for (cudaEvent_t e : ix->prof_ev) cudaEventDestroy(e);
  ix->prof_ev.clear();
  ix->prof_slots = 0;
  ix->prof_steps = 0;
  const size_t n = (size_t)max_steps * WI_DECODE_EVENTS;
  for (size_t i = 0; i < n; ++i) {
    cudaEvent_t e;
    WI_CUDA(cudaEventCreate(&e));
    ix->prof_ev.push_back(e);
  }
  ix->prof_slots = max_steps;
  return WI_OK;
}

int wi_profile_read(wi_index* ix, double* kernel_ms, int* steps, unsigned long long* exact_rows) {
  g_err[0] = 0;
  if (!ix) return fail(WI_EINVAL, "index is NULL");
  WI_CUDA(cudaDeviceSynchronize());
  const int filled = (int)(ix->prof_steps < ix->prof_slots ? ix->prof_steps : ix->prof_slots);
  if (kernel_ms) {
    for (int k = 0; k < WI_DECODE_KERNELS; ++k) kernel_ms[k] = 0.0;
    for (int sl = 0; sl < filled; ++sl) {
      const cudaEvent_t* ev = ix->prof_ev.data() + (size_t)sl * WI_DECODE_EVENTS;
      for (int k = 0; k < WI_DECODE_KERNELS; ++k) {
        float ms = 0.f;
        WI_CUDA(cudaEventElapsedTime(&ms, ev[k], ev[k + 1]));
        kernel_ms[k] += ms;
      }
    }
  }
  if (steps) *steps = filled;
  if (exact_rows) WI_CUDA(cudaMemcpy(exact_rows, ix->b.rows_total, 8, cudaMemcpyDeviceToHost));
  return WI_OK;
}

int wi_index_build_stats(wi_index* ix, double* build_ms, double* assign_ms, int* assign_launches) {
  g_err[0] = 0;
  if (!ix) return fail(WI_EINVAL, "index is NULL");
  if (ix->build_ev.size() < 2) return fail(WI_EUNSUPPORTED, "the index was not built by wi_build_index");
  WI_CUDA(cudaEventSynchronize(ix->build_ev[1]));
  float ms = 0.f;
  if (build_ms) {
    WI_CUDA(cudaEventElapsedTime(&ms, ix->build_ev[0], ix->build_ev[1]));
    *build_ms = ms;
  }
  const int n = (int)(ix->build_ev.size() - 2) / 2;
  if (assign_ms) {
    double acc = 0.0;
    for (int t = 0; t < n; ++t) {
      WI_CUDA(cudaEventElapsedTime(&ms, ix->build_ev[2 + 2 * t], ix->build_ev[3 + 2 * t]));
      acc += ms;
    }
    *assign_ms = acc;
  }
  if (assign_launches) *assign_launches = n;
  return WI_OK;
}

int wi_check_device(wi_index* ix) {
  g_err[0] = 0;
  if (!ix) return fail(WI_EINVAL, "index is NULL");
  WI_CUDA(cudaStreamSynchronize(ix->last_stream));
  int herr = 0;
  WI_CUDA(cudaMemcpy(&herr, ix->err, 4, cudaMemcpyDeviceToHost));
  if (herr) {
    WI_CUDA(cudaMemset(ix->err, 0, 4));
    return fail(WI_EDEVICE, "device invariant violated (flags 0x%x)", herr);
  }
  return WI_OK;
}

int wi_tier_attach(wi_index* ix, int slots_per_unit, int admit_per_round, int async, void* stream) {
  g_err[0] = 0;
  if (!ix) return fail(WI_EINVAL, "index is NULL");
  if (ix->tier) return fail(WI_EINVAL, "the index already has a host memory tier");
  const WiGeom& g = ix->g;
  if (g.Gmax > 0) return fail(WI_EUNSUPPORTED, "a host memory tier needs an index that does not grow (max_append < seg_len)");
  if (g.vs16) return fail(WI_EUNSUPPORTED, "a host memory tier needs fp32 value sums");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char msg[320];
  WiTierDev dev{};
  const int rc = wi_tier_create(g, ix->K, ix->V, slots_per_unit, admit_per_round, async, ix->device, st, &ix->tier,
                                &dev, msg, sizeof(msg));
  if (rc != WI_OK) return fail(rc, "%s", msg);
  ix->b.tier = dev;
  ix->last_stream = st;
  return WI_OK;
}

int wi_tier_round(wi_index* ix, void* stream) {
  g_err[0] = 0;
  if (!ix || !ix->tier) return fail(WI_EINVAL, "index has no host memory tier");
  if (ix->steps_run == 0) return WI_OK;
  char msg[320];
  const int rc = wi_tier_round_now(ix->tier, ix->steps_run - 1, static_cast<cudaStream_t>(stream), msg, sizeof(msg));
  if (rc != WI_OK) return fail(rc, "%s", msg);
  return WI_OK;
}

int wi_tier_stats(wi_index* ix, long long* counters, unsigned long long* rows, int* slots, int* pages) {
  g_err[0] = 0;
  if (!ix || !ix->tier) return fail(WI_EINVAL, "index has no host memory tier");
  wi_tier_idle(ix->tier);
  WI_CUDA(cudaStreamSynchronize(ix->last_stream));
  if (counters) wi_tier_counters(ix->tier, counters);
  if (rows) WI_CUDA(cudaMemcpy(rows, wi_tier_row_counters(ix->tier), 16, cudaMemcpyDeviceToHost));
  int s = 0, p = 0;
  wi_tier_geometry(ix->tier, &s, &p);
  if (slots) *slots = s;
  if (pages) *pages = p;
  return WI_OK;
}

int wi_tier_tables(wi_index* ix, int32_t* slot_of, int32_t* use) {
  g_err[0] = 0;
  if (!ix || !ix->tier) return fail(WI_EINVAL, "index has no host memory tier");
  wi_tier_idle(ix->tier);
  WI_CUDA(cudaStreamSynchronize(ix->last_stream));
  int s = 0, p = 0;
  wi_tier_geometry(ix->tier, &s, &p);
  const size_t bytes = (size_t)ix->g.U * p * 4;
  if (slot_of) WI_CUDA(cudaMemcpy(slot_of, wi_tier_slot_table(ix->tier), bytes, cudaMemcpyDeviceToHost));
  if (use) WI_CUDA(cudaMemcpy(use, wi_tier_use_table(ix->tier), bytes, cudaMemcpyDeviceToHost));
  return WI_OK;
}

// The entry points that allocate host memory (std::vector, the index object's lists): an allocation
// failure is reported as WI_ENOMEM, never thrown across the C ABI.
int wi_build_index(const wi_config* cfg, void* k, void* v, const void* init_centroids, void* stream,
                   wi_index** out) {
  try {
    return build_index_impl(cfg, k, v, init_centroids, stream, out);
  } catch (...) {
    if (out) *out = nullptr;
    return fail(WI_ENOMEM, "host allocation failed");
  }
}

int wi_index_import(const wi_config* cfg, void* k, void* v, const int32_t* counts, const int32_t* perm,
                    const uint16_t* mu, const float* valsum, void* stream, wi_index** out) {
  try {
    return index_import_impl(cfg, k, v, counts, perm, mu, valsum, stream, out);
  } catch (...) {
    if (out) *out = nullptr;
    return fail(WI_ENOMEM, "host allocation failed");
  }
}

int wi_profile_begin(wi_index* ix, int max_steps) {
  try {
    return profile_begin_impl(ix, max_steps);
  } catch (...) {
    return fail(WI_ENOMEM, "host allocation failed");
  }
}

void wi_free(wi_index* ix) {
  if (!ix) return;
  cudaDeviceSynchronize();
  destroy(ix);
}

}  // extern "C"
