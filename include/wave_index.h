/*
 * wave_index.h -- C ABI of the GB300 wave-index hot path.
 *
 * RetroInfer treats the KV cache as a vector store that each decode step
 * queries (RetroInfer abstract; summaries de/fr/zh section 2.A).  This library
 * builds that store's index at prefill -- segmented spherical k-means over
 * the keys of every (sequence, layer, kv head), with per-cluster counts, mean
 * keys and value sums -- and runs the decode-time tripartite attention:
 * steady zone (sinks + local window) and the top-k retrieved clusters exactly,
 * every other cluster estimated from its mean key, count and value sum, the
 * zones merged by log-sum-exp.
 *
 * Conventions for every entry point:
 *   - All tensors are row-major and contiguous.  bf16 tensors are passed as
 *     raw 16-bit patterns (uint16_t / void*).
 *   - "device" pointers must be CUDA device memory of the current device
 *     (cudaMalloc / torch); "host" pointers plain host memory; "any" pointers
 *     either (copied with cudaMemcpyDefault, so they must be UVA-addressable).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *     enqueued on it; outputs are valid once the stream has been synchronised,
 *     unless stated otherwise.
 *   - Every call returns WI_OK (0) or a negative WI_E* code and then leaves a
 *     thread-local message readable with wi_last_error().  No call aborts,
 *     exits, throws across the ABI or traps on the device.  On error an
 *     output handle is set to NULL.
 *   - Head size d must be 128.  Query head h attends with kv head h / g,
 *     g = n_q_heads / n_kv_heads.  A "unit" is one (sequence b, layer l,
 *     kv head h), numbered u = (b * layers + l) * n_kv_heads + h.
 */
#ifndef WAVE_INDEX_H
#define WAVE_INDEX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  WI_OK = 0,
  WI_EINVAL = -1,       /* bad argument: shape, null pointer, d != 128, k > C, ... */
  WI_ENOMEM = -2,       /* a device or host allocation failed */
  WI_ECUDA = -3,        /* a CUDA runtime call failed (message names it) */
  WI_EUNSUPPORTED = -4, /* valid but not supported by this build */
  WI_EDEVICE = -5,      /* a kernel reported a violated invariant */
  WI_EFULL = -6         /* the append buffer is full */
};

typedef struct wi_index wi_index; /* opaque, library-owned */

/*
 * Shapes and method parameters.  Zones (summaries de/fr/zh 2.A): the steady
 * zone is positions [0, n_sink) and [n_ctx - local_window, n_ctx) plus every
 * token appended during decode; all other positions are clustered.
 * Segmented clustering (same sections): each run of seg_len positions is
 * clustered on its own into clusters_per_seg clusters (global id =
 * segment * clusters_per_seg + local id) by `iters` rounds of spherical
 * k-means (summary fr 2.A.2).  Retrieval budget (summary zh section 3):
 * k = budget_k if > 0, else ceil(budget_frac * C), C = all clusters of a unit;
 * capped at the unit's non-empty clusters at decode time.
 * Decode-time growth (an extension: the pages describe the index at prefill):
 * the index holds room for C = (n_ctx / seg_len + max_append / seg_len) *
 * clusters_per_seg clusters per unit; those of segments not grown yet are
 * empty, and the budget k counts only the clusters held so far.
 * Limits of this build (WI_EUNSUPPORTED beyond them): n_q_heads / n_kv_heads
 * <= 8, k <= 4096, seg_len <= 16384, C <= 65536 (room for growth included).
 */
typedef struct {
  int batch, layers, n_q_heads, n_kv_heads, head_dim; /* head_dim == 128 */
  long long n_ctx;        /* tokens per unit at build; a multiple of seg_len */
  int seg_len;            /* a multiple of 128, >= 128 */
  int clusters_per_seg;   /* multiple of 16 in [16, 512] dividing seg_len */
  int iters;              /* k-means rounds (assignments), >= 1 */
  int n_sink, local_window;
  int max_append;         /* capacity of the decode-time append buffer, >= 0; with max_append >=
                             seg_len the index also grows during decode (wi_decode_step) */
  double budget_frac;
  int budget_k;
  int valsum_bf16;        /* 0: decode reads the fp32 value sums; 1: it reads a bf16 copy made at
                             build / import (round to nearest even; half the estimation bytes) */
  int group_topk;         /* 0: each query head takes its own top-k; 1: the query heads of a kv head
                             share the top-k of their summed scores (each head keeps its own logits,
                             estimate and retrieved-term weights) */
  int reserved[1];        /* must be zero */
} wi_config;

/*
 * Build the index (prefill): segmented spherical k-means and the per-cluster
 * count, mean key and value sum of every unit (summaries de/fr/zh 2.A
 * "segmented clustering", fr 2.A.2 "spherical k-means", zh 2.A "precomputed
 * value sum").  k, v: device bf16 [batch][layers][n_kv_heads]
 * [n_ctx][128], caller-owned.  The library permutes their clustered rows IN
 * PLACE into cluster-contiguous order (cluster by cluster, by position inside
 * a cluster; steady rows stay where they are) and keeps pointing at them: the
 * caller keeps both alive and unmodified until wi_free.
 * init_centroids: NULL for the default seeding (the normalised key at the
 * start of each stride-(seg_len/clusters_per_seg) block of a segment), or
 * device bf16 [units][n_ctx/seg_len][clusters_per_seg][128] used as the
 * centroids of the first round (rows should be unit-norm).
 * Enqueues the build on `stream` and returns; *out is usable on that stream.
 */
int wi_build_index(const wi_config* cfg, void* k, void* v, const void* init_centroids, void* stream,
                   wi_index** out);

/*
 * Adopt an index computed elsewhere instead of clustering (e.g. by a CPU
 * reference).  counts: [units][Cb] int32, Cb = (n_ctx / seg_len) *
 * clusters_per_seg (the build's clusters); perm: [units][n_ctx - n_sink -
 * local_window] int32, the original position of every clustered slot in
 * cluster-contiguous order (slots of cluster j follow those of cluster j-1;
 * slot numbering starts at row n_sink); mu: bf16 [units][Cb][128] mean keys;
 * valsum: fp32 [units][Cb][128] value sums.  All four are "any" pointers and
 * are copied.  k, v as in wi_build_index (permuted in place by perm).
 * Returns WI_EINVAL if perm is not a bijection on the clustered positions
 * consistent with counts and segments (checked on the host).
 */
int wi_index_import(const wi_config* cfg, void* k, void* v, const int32_t* counts, const int32_t* perm,
                    const uint16_t* mu, const float* valsum, void* stream, wi_index** out);

/*
 * Copy the index out ("any" pointers; any of them may be NULL to skip it),
 * C = the clusters per unit from wi_index_shape (room for growth included).
 * counts [units][C], offsets [units][C+1] (row of the first slot of each
 * cluster; offsets[Cb] = n_ctx - local_window; a grown segment g's slots are
 * rows n_ctx + g*seg_len + slot), perm [units][n_ctx - n_sink - local_window
 * + (max_append / seg_len) * seg_len] (as in wi_index_import, then every grown
 * segment's seg_len slots; -1 where nothing has grown yet), mu bf16
 * [units][C][128], valsum fp32 [units][C][128].  Clusters not grown yet have
 * count 0 and zero mean key and value sum.  Asynchronous.
 */
int wi_index_export(const wi_index* ix, int32_t* counts, int32_t* offsets, int32_t* perm, uint16_t* mu,
                    float* valsum, void* stream);

/*
 * One decode step of the tripartite attention approximation (summaries
 * de/fr/zh 2.A: steady and retrieval zones exact, estimation zone from each
 * cluster's mean key, count and value sum, merged by log-sum-exp; zh section 3
 * for the ~1.8% retrieval budget).  q: device bf16 [batch][layers][n_q_heads][128], the
 * queries of the step (already rotated), 16-byte aligned; out: device fp32 [batch][layers]
 * [n_q_heads][128], attention output per query head.  Attention runs over
 * the current context: the n_ctx built tokens plus every token appended so
 * far.  If k_new and v_new (device bf16 [batch][layers][n_kv_heads][128]) are
 * non-NULL, that token is appended AFTER this step's attention; returns
 * WI_EFULL (nothing enqueued) when max_append tokens are already appended.
 * Appended tokens join the local window.  When an append leaves the window
 * holding local_window + seg_len rows (every seg_len appended tokens), the
 * step also grows the index: the window's oldest seg_len rows become one more
 * segment, clustered like a build segment (same seeds rule, iters rounds,
 * counts / mean keys / value sums; its rows copied, cluster-contiguous, into
 * library memory), its clusters take the next free ids and the budget is
 * recomputed for the clusters held.
 * Uses only library-owned scratch: no allocation and no host synchronisation.
 * Steps without append replay correctly from a captured CUDA graph (a graph
 * captured before a growth keeps attending over the grown index correctly:
 * the growth state lives in device memory).
 */
int wi_decode_step(wi_index* ix, const void* q, const void* k_new, const void* v_new, float* out, void* stream);

/*
 * wi_decode_step with HOST q / k_new / v_new / out: copies the inputs to the
 * device, runs the step, copies the output back and synchronises `stream`
 * before returning (out is valid on return).  Pinned host memory makes the
 * copies asynchronous DMA; pageable memory works but is slower.  A step with
 * pinned (device-mapped, 16-byte aligned) q and out, no append and decode
 * profiling off runs as one CUDA graph that the index captures for that pair
 * of buffers: a copy kernel reads q from host memory, the decode kernels run
 * and the final merge writes out straight to host memory.  The index owns a
 * stream and the graph until wi_free; a call with other buffers captures
 * again, and after a few such changes the index launches directly, as it
 * does for every other step.  Results are identical either way.
 */
int wi_decode_step_host(wi_index* ix, const void* q_host, const void* k_new_host, const void* v_new_host,
                        float* out_host, void* stream);

/*
 * Clusters retrieved by the last decode step: ids [units][g][k_max] int32
 * ("any"), ascending within each head, padded with -1; counts [units][g]
 * int32 ("any", may be NULL).  k_max is reported by wi_index_shape.
 */
int wi_last_selection(const wi_index* ix, int32_t* ids, int32_t* counts, void* stream);

/*
 * Full attention over every token the index holds: the dense comparator that
 * the wave index approximates (RetroInfer summaries de/fr/zh section 2.A; the
 * speed-up over it in zh section 3).  For every unit and query head,
 * out = softmax(q K^T / sqrt(128)) V over the unit's n_ctx context rows and
 * the tokens appended so far, with no index involved (the context rows are
 * read in the index's cluster-contiguous order; attention does not depend on
 * the order).  q: device bf16 [batch][layers][n_q_heads][128]; out: device
 * fp32, same layout (both caller-owned, q 16-byte aligned).  Uses the index's
 * own scratch: calls on one index must be ordered (one stream).  Stream-
 * ordered, asynchronous, no allocation, graph-capturable.  Fp32 accumulation.
 */
int wi_dense_decode(wi_index* ix, const void* q, float* out, void* stream);

/*
 * One kernel of the decode step alone (benchmarking aid: the duration of one
 * kernel in isolation, without events between kernels).  kernel 0: centroid
 * scores; 1: top-k with the estimation over all clusters; 2: exact attention
 * with the final merge.  Each kernel reads what the previous one wrote in the
 * last decode step of this index, so it repeats that step's work for its
 * part; q and out as in wi_decode_step (kernel 2 rewrites out).  Returns
 * WI_EINVAL before the index's first wi_decode_step.  Stream-ordered, no
 * allocation, graph-capturable.
 */
int wi_decode_kernel(wi_index* ix, int kernel, const void* q, float* out, void* stream);

/* Sizes of an index: units, clusters per unit C (room for decode-time growth
 * included), k_max (the budget for C clusters, the largest it can grow to),
 * group g, tokens appended so far (host-side count).  Any output pointer may
 * be NULL. */
int wi_index_shape(const wi_index* ix, int* units, int* clusters, int* k_max, int* group, int* appended);

/*
 * Launch layout of this index's decode kernels, fixed when the index is made
 * from the device's SM count: scores CTAs per unit, estimation CTAs per unit,
 * and exact-attention splits per head over the selected rows (one more CTA
 * takes the steady rows).  The environment variables WI_D1_CTAS_PER_UNIT,
 * WI_ESTIMATE_CTAS_PER_UNIT and WI_D3_SPLITS (positive integers), and
 * WI_ESTIMATE_FIRST (0 or 1: the estimation CTAs before the top-k CTAs in
 * their shared launch; default: when they fit in one wave), WI_D3_STAGE_ROWS
 * (32 or 64: rows per shared-memory stage of the exact-attention CTAs;
 * default 32 when all of them are resident at once, else 64) and
 * WI_ESTIMATE_DEPTH (2 or 3: value-sum tiles in flight per estimation CTA;
 * default 2 when the top-k and estimation CTAs fit in one wave, else 3),
 * read when the index is made, override the defaults.  Results do not depend on the
 * layout beyond float rounding order.  Any output pointer may be NULL.
 */
int wi_decode_layout(const wi_index* ix, int* score_ctas, int* estimate_ctas, int* exact_splits);

/*
 * One spherical k-means round on every segment, for per-round checking:
 * assignment of each clustered token against `centroids` (device bf16
 * [units][n_segments][clusters_per_seg][128]) written to assign (device int32
 * [units][n_ctx], global cluster id, -1 for steady positions), then the
 * updated centroids bf16(normalise(sum of normalised member keys)), empty
 * clusters unchanged, to new_centroids (device, same shape; may alias
 * centroids).  k: device bf16 keys as in wi_build_index (not modified).
 * Allocates and frees its own scratch on `stream`.
 */
int wi_kmeans_step(const wi_config* cfg, const void* k, const void* centroids, int32_t* assign,
                   void* new_centroids, void* stream);

/*
 * The default first-round centroids of every segment, for per-step checking
 * of the k-means initialisation (segmented spherical k-means: summaries
 * de/fr/zh 2.A, fr 2.A.2; seeding is not stated there, and this build takes
 * the first key of each stride-(seg_len/clusters_per_seg) block of the
 * segment, steady positions included): centroids[u][s][j] =
 * bf16(K[u][s*seg_len + j*stride] / |K[u][s*seg_len + j*stride]|), the
 * centroids that wi_build_index uses when init_centroids is NULL.
 * k: device bf16 keys as in wi_build_index (not modified); centroids: device
 * bf16 [units][n_segments][clusters_per_seg][128].  Asynchronous on `stream`.
 */
int wi_init_centroids(const wi_config* cfg, const void* k, void* centroids, void* stream);

/*
 * Per-kernel timing of decode steps (benchmarking aid).  After
 * wi_profile_begin(ix, max_steps), every decode step on this index records
 * CUDA events around each of its WI_NUM_DECODE_KERNELS kernels (centroid
 * scores; top-k with the retrieved clusters' estimation terms, sharing one
 * launch with the estimation over all clusters; exact attention with the
 * final merge) into slot
 * (step number % max_steps); steps captured into a CUDA graph record them on
 * every replay.  wi_profile_read synchronises the device and returns, per
 * kernel, the summed duration in milliseconds over the filled slots
 * (kernel_ms[WI_NUM_DECODE_KERNELS], may be NULL), the number of filled
 * slots, and the exact-zone rows processed by all decode steps since the
 * index was created, counted per query head (the bytes the exact-attention
 * kernel loads are rows * 512).
 * wi_profile_begin with max_steps = 0 turns recording off.
 */
#define WI_NUM_DECODE_KERNELS 3
int wi_profile_begin(wi_index* ix, int max_steps);
int wi_profile_read(wi_index* ix, double* kernel_ms, int* steps, unsigned long long* exact_rows);

/*
 * wi_kmeans_step without any device allocation (the paper has no
 * counterpart; this is an interface for callers that may not allocate).
 * A serving process usually gives nearly all GPU memory to its KV-cache
 * pool, and some hosts allow device memory only through their own arena;
 * such callers cannot let a clustering round call cudaMalloc.  Same
 * arguments, same results as wi_kmeans_step; its scratch is a fixed 8 MiB
 * device array that every GPU loading this library holds until the process
 * exits.  Problems that need more scratch (about 400K tokens in total at 512
 * clusters per 8192-token segment) return WI_EINVAL with a message.
 * All calls share the array: calls whose work overlaps on the GPU race on it
 * (order them on one stream).  Every call looks up the array's device
 * address with the caller's device current (no allocation), so a device
 * reset between calls is harmless.  Synchronises `stream` before returning.
 */
int wi_kmeans_step_noalloc(const wi_config* cfg, const void* k, const void* centroids, int32_t* assign,
                           void* new_centroids, void* stream);

/*
 * Timing of the build that made this index (CUDA events recorded on its
 * stream): whole build in ms, summed duration of its `iters` assignment
 * launches in ms, and their number.  Waits for the build to finish.  Returns
 * WI_EUNSUPPORTED for an index made by wi_index_import.  Any output may be NULL.
 */
int wi_index_build_stats(wi_index* ix, double* build_ms, double* assign_ms, int* assign_launches);

/* Synchronise the index's last stream and report a device-side invariant
 * violation recorded by any kernel since the last call (WI_EDEVICE). */
int wi_check_device(wi_index* ix);

/* Test hook: the failure path of the kernels' bounded waits, run on purpose.
 * Launches, on the current device, one kernel whose thread waits on a
 * shared-memory mbarrier that nothing ever completes, through the same
 * bounded wait the library's kernels use (it gives up after about 2^31 SM
 * cycles, ~1 s, records the timeout bit 16 in the kernel's error word and
 * returns), and synchronises the device.  On WI_OK, *device_error is the
 * kernel's error word (16 when the wait gave up) and *wait_returned 1 when the
 * wait returned without completion (2 if it had completed).  No fault, trap
 * or endless loop; the context stays usable.  Host outputs; errors:
 * WI_EINVAL (null pointer), WI_ENOMEM, WI_ECUDA. */
int wi_selftest_wait_timeout(int* device_error, int* wait_returned);

/*
 * Host memory tier: the wave buffer (summaries de/fr/zh section 2.B: a GPU
 * block cache of the KV blocks retrieval keeps returning to, LRU replacement
 * run by the CPU asynchronously, an execution buffer that feeds attention the
 * tokens from the steady zone, the cache and CPU memory).
 *
 * wi_tier_attach copies the index's permuted K and V (the caller's k / v,
 * device) to page-locked host memory owned by the library and the sink and
 * window rows to a device copy, and waits for `stream`; from then on no call
 * reads the caller's k / v, which the caller may free or reuse.  The host
 * rows are split into pages of 16 consecutive rows of a unit; each unit gets
 * `slots_per_unit` (0 .. pages per unit) page slots in device memory, empty at
 * first.  The exact-attention kernel of every later decode step copies each
 * retrieved row from its cached page or, if the page is not cached, straight
 * from host memory over the CPU-GPU link, and stamps the page with the step.
 * A replacement round takes the pages read since the previous round, in
 * increasing page order per unit: a cached page becomes the most recently
 * used; a page not cached is admitted (at most `admit_per_round` per unit and
 * round) into the lowest free slot, else into the slot of the least recently
 * used page unless that page was read in this same round, in which case the
 * round admits nothing more.  A round unmaps its victims on the decode stream,
 * fills their slots from host memory on a stream of its own and maps the new
 * pages on the decode stream once the fill has landed: decode never waits for
 * a round and never reads a slot being refilled.  With async != 0 a library
 * thread runs a round whenever it is idle after a decode step (on the newest
 * stamps); with async == 0 rounds run only in wi_tier_round.  Outputs do not
 * depend on where rows were read from: they equal the same index's outputs
 * without the tier bit for bit.
 * Needs an index that does not grow (max_append < seg_len) and fp32 value
 * sums (WI_EUNSUPPORTED otherwise).  Afterwards wi_dense_decode returns
 * WI_EUNSUPPORTED, and wi_decode_step refuses a stream being captured into a
 * graph.  Host memory: 2 * units * n_ctx * 256 bytes; device: 2 * units *
 * slots_per_unit * 4096 bytes plus 8 bytes per page for the tables.
 */
int wi_tier_attach(wi_index* ix, int slots_per_unit, int admit_per_round, int async, void* stream);

/* One replacement round now, on the calling thread, over the pages read by
 * every decode step enqueued so far; waits for a running round first and for
 * the round's own work before returning. */
int wi_tier_round(wi_index* ix, void* stream);

/* Counters of the tier since attach, after waiting for any running round and
 * the index's last stream: counters[6] = rounds, pages read (as the rounds saw
 * them), of which cached, of which not, pages admitted, pages evicted;
 * rows[2] = rows the exact-attention kernels copied from cached pages, from
 * host memory.  slots / pages: slots and pages per unit.  Outputs may be NULL. */
int wi_tier_stats(wi_index* ix, long long* counters, unsigned long long* rows, int* slots, int* pages);

/* Test hook: the tier's tables, host int32 [units][pages] each: the slot
 * holding each page (-1: not cached) and the last step that read it (-1:
 * none).  Waits like wi_tier_stats.  Either output may be NULL. */
int wi_tier_tables(wi_index* ix, int32_t* slot_of, int32_t* use);

/* The tier's replacement policy alone, on the host (no device involved), for
 * checking: a cache of `slots` pages out of `pages` for one unit.  wi_lru_round
 * runs one round for the pages in `touched` (any order, repeats ignored) at
 * round number t and writes the evictions and admissions, in the order it made
 * them, as (page, slot) pairs; each output array needs room for n entries (any
 * may be NULL).  wi_lru_new returns NULL for bad sizes. */
void* wi_lru_new(int pages, int slots, int admit_max);
int wi_lru_round(void* policy, const int32_t* touched, int n, long long t, int32_t* ev_pages, int32_t* ev_slots,
                 int* n_ev, int32_t* ad_pages, int32_t* ad_slots, int* n_ad);
void wi_lru_free(void* policy);

/* Error-path testing: with the environment variable WI_FAIL_ALLOC_AT=n (n >= 1),
 * the n-th device allocation made for any index fails as out-of-memory; the
 * call returns WI_ENOMEM having released what it had allocated.  Likewise
 * WI_FAIL_TIER_ALLOC_AT=n for the n-th allocation (device or page-locked
 * host) of wi_tier_attach, which then leaves the index as it was. */

/* Release the index and everything it owns (not k / v).  NULL is a no-op.
 * Synchronises the device first. */
void wi_free(wi_index* ix);

/* Message of the last failed call on this thread ("" if none). */
const char* wi_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* WAVE_INDEX_H */
