// wi_internal.h -- host-side declarations shared by the wave-index sources.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "wave_index.h"

// Geometry of one build / index, derived from wi_config.
struct WiGeom {
  int U;          // units = batch * layers * n_kv_heads
  int G;          // query heads per kv head
  int S, Cs;      // segment length, clusters per segment
  int nseg;       // segments per unit at build
  int Cb;         // clusters per unit of the build's segments = nseg * Cs
  int Gmax;       // segments that decode-time growth may add: max_append / S
  int C;          // clusters per unit the index holds room for = Cb + Gmax * Cs (row stride of every
                  // per-cluster array; clusters of segments not grown yet are empty)
  long long n;    // built tokens per unit
  int n_sink, W;  // steady zone
  int n_idx;      // clustered tokens per unit at build = n - n_sink - W
  int perm_stride;  // slots per unit in perm = n_idx + Gmax * S
  int iters;
  int kbuild;     // retrieval budget over the build's clusters
  int kmax;       // retrieval budget over all C clusters (the largest it can grow to)
  int max_append;
  int vs16;       // decode reads the bf16 copy of the value sums
  int grp;        // group-shared retrieval: one top-k per kv head from the heads' summed scores
  double budget_frac;
  int budget_k;
};

// Retrieval budget for C clusters: budget_k if set, else ceil(budget_frac * C).
int wi_budget(const WiGeom& g, int C);

int wi_geom_from_config(const wi_config* cfg, WiGeom* g, char* msg, size_t msglen);
void wi_set_error(const char* msg);  // sets the thread-local message of wi_last_error()

// ---- build kernels (wi_build.cu); all enqueue on `st` and return the launch status
// out[i] = bf16(in[i]), round to nearest even.
cudaError_t wi_launch_to_bf16(const float* in, void* out, long long n, cudaStream_t st);
cudaError_t wi_launch_init_centroids(const WiGeom& g, const void* K, void* chat, cudaStream_t st);
cudaError_t wi_launch_assign(const WiGeom& g, const void* K, const void* chat, int32_t* assign, int* err,
                             cudaStream_t st);
cudaError_t wi_launch_segment_sort(const WiGeom& g, const int32_t* assign, int* seg_counts, int* seg_offsets,
                                   int* slots, int* err, cudaStream_t st);
cudaError_t wi_launch_centroid_update(const WiGeom& g, const void* K, const int* seg_counts, const int* seg_offsets,
                                      const int* slots, void* chat, cudaStream_t st);
// B4 + B5: the final index of the g.Cb build clusters of every unit (arrays of row stride g.C, offsets
// g.C + 1, perm g.perm_stride; nonempty cleared first) and the in-place cluster-contiguous permutation
// of K and V, batch_units units at a time through the scratch rows tmpK / tmpV (batch_units * n_idx
// rows each).
cudaError_t wi_launch_reduce_permute(const WiGeom& g, void* K, void* V, const int* seg_counts, const int* seg_offsets,
                                     const int* slots, void* mu, float* valsum, int* cnt, int* off, int* perm,
                                     int* nonempty, void* tmpK, void* tmpV, int batch_units, cudaStream_t st);
cudaError_t wi_launch_permute(const WiGeom& g, void* K, void* V, const int* perm, void* tmpK, void* tmpV,
                              int u0, int nu, cudaStream_t st);
size_t wi_assign_smem_bytes(const WiGeom& g);

bool wi_encode_rows_sw128(CUtensorMap* map, const void* base, unsigned long long rows, unsigned box_rows);

// ---- tensor-core assignment (wi_assign_tc.cu)
bool wi_assign_tc_supported(const WiGeom& g);
cudaError_t wi_launch_assign_tc(const WiGeom& g, const void* K, const void* chat, int32_t* assign, int* err,
                                cudaStream_t st);

// ---- host memory tier (wi_tier.cu): the build's clustered K/V rows held in page-locked host memory,
// pages of kWiPageRows rows cached in device memory (the wave buffer).
constexpr int kWiPageRows = 16;
struct WiTierDev {
  int on;                 // the exact kernel reads clustered rows through the tier
  int slots;              // cache slots (pages) per unit
  int pages;              // pages per unit: ceil(n / kWiPageRows) over the unit's row space [0, n)
  int step;               // decode step number written into `use` (set per launch)
  const int* slot_of;     // [U][pages] device: cache slot holding each page, or -1
  const void* poolK;      // [U][slots][kWiPageRows][128] bf16, device
  const void* poolV;
  const void* hostK;      // [U][n][128] bf16 page-locked host memory (its device address)
  const void* hostV;
  const void* steadyK;    // [U][n_sink + W][128] bf16 device: the build's sink and window rows
  const void* steadyV;
  int* use;               // [U][pages] device: last step whose exact kernel read each page
  unsigned long long* rows_src;  // [2] device: exact rows read from the cache, from host memory
};

struct WiTierHost;  // the tier's host side: replacement policy, thread, buffers (wi_tier.cu)
// Copies the index's permuted K/V rows (device, [U][n][128] each) to page-locked host memory and the
// sinks and window to a device copy, then waits for st: K and V are not read afterwards.
int wi_tier_create(const WiGeom& g, const void* K, const void* V, int slots, int admit, int async, int device,
                   cudaStream_t st, WiTierHost** out, WiTierDev* dev, char* msg, size_t len);
void wi_tier_destroy(WiTierHost* T);
int wi_tier_after_step(WiTierHost* T, long long step, cudaStream_t st, char* msg, size_t len);
int wi_tier_round_now(WiTierHost* T, long long step, cudaStream_t st, char* msg, size_t len);
void wi_tier_idle(WiTierHost* T);
void wi_tier_counters(WiTierHost* T, long long out[6]);
int wi_tier_geometry(const WiTierHost* T, int* slots, int* pages);
const int* wi_tier_slot_table(const WiTierHost* T);
const int* wi_tier_use_table(const WiTierHost* T);
const unsigned long long* wi_tier_row_counters(const WiTierHost* T);

// ---- decode kernels (wi_decode.cu)
struct WiDecodeBufs {
  CUtensorMap map_mu;     // mu as rows of 128 bf16, 128-row boxes, 128-byte swizzle (tensor-core scores)
  const void* mu;
  const float* valsum;
  const void* valsum16;   // [U][C][128] bf16 copy, when the config asks decode to read it (else null)
  const int* cnt;
  const int* off;
  const int* nonempty;
  const void* K;
  const void* V;
  void* appK;
  void* appV;
  int* app_count;
  const void* grownK;     // [Gmax][U][S][128] rows of the segments grown during decode, cluster-contiguous
  const void* grownV;
  int* grown;             // segments grown so far (device)
  int* kcur;              // retrieval budget of the clusters held so far (device)
  float* scores;          // [U][G][C] order-preserving score keys (uint32; 0 = empty cluster)
  float* part1;           // [U][G][p_es][WI_PART]  estimation partials
  int* sel;               // [U][G][kmax]
  int* selcnt;            // [U][G]
  float* subpart;         // [U][G][WI_PART]      estimation terms of the selected clusters
  int4* runs;             // [U][G][kmax]  (first row, rows, weight bits, id) of each selected cluster
  int4* splits;           // [U][G][nsplit+2]  starts of the nsplit+1 row-balanced splits (steady + selected rows)
  int4* sruns;            // [U][G][nsplit+1][32] the first 32 runs of each split (copies)
  float* part3;           // [U][G][nsplit+1][WI_PART]  exact partials (the last split: steady rows)
  float* subn;            // [U][G][nsplit+1][WI_PART]  retrieved clusters' value-sum terms per split
  unsigned int* ticket;   // [U][G]  CTAs of exact_merge finished, per head
  unsigned int* kmaxp;    // [U][p1][G] largest score key over the non-empty clusters of each k_scores CTA
  unsigned long long* rows_total;  // running sum of exact rows loaded over all steps
  int* err;
  int p1;                 // k_scores CTAs per unit
  int p_es;               // estimation CTAs per unit (= estimation partials per head)
  int est_first;          // the select/estimate launch starts its estimation CTAs first
  int es_depth;           // estimation stages in flight per CTA (2 or 3)
  int nsplit;             // exact_merge CTAs per head over the selected rows (plus one for steady rows)
  int d3_rows;            // exact_merge stage height: 32 (one wave of CTAs) or 64 rows
  WiTierDev tier;         // host memory tier (tier.on == 0: none)
  // dense comparator (full attention)
  float* dpart;           // [U][G][dsplits][WI_PART]  row-range partials
  unsigned int* dticket;  // [U]
  int dsplits;            // row ranges (CTAs) per unit
};
#define WI_PART 132  // floats per zone partial: m, Z, 2 pad, N[128]

#define WI_DECODE_KERNELS 3  // scores, select_estimate (top-k + estimation CTAs), exact_merge
#define WI_DECODE_EVENTS 4   // per profiled step: before the first kernel, then after each kernel
// Full attention over every cached and appended token (the dense comparator).
cudaError_t wi_launch_dense(const WiGeom& g, const WiDecodeBufs& b, const void* q, float* out, cudaStream_t st);
int wi_dense_ctas_per_sm(int G);
// mask: bit i launches decode kernel i (1 scores, 2 select/estimate, 4 exact/merge); 7 = a whole step
cudaError_t wi_launch_decode(const WiGeom& g, const WiDecodeBufs& b, const void* q, float* out, cudaStream_t st,
                             const cudaEvent_t* ev, unsigned mask = 7u);
// bytes (a multiple of 16) from src to dst, 16-byte aligned; either may be mapped host memory.
cudaError_t wi_launch_copy16(const void* src, void* dst, size_t bytes, cudaStream_t st);
cudaError_t wi_launch_append(const WiGeom& g, const WiDecodeBufs& b, const void* k_new, const void* v_new, int t,
                             cudaStream_t st);

// ---- decode-time index maintenance (wi_grow.cu): the oldest S rows of the local window become
// segment `gi` of the grown part (B1-B5 on that one segment), merged into the index.
struct WiGrowBufs {
  // one segment of every unit: [U][S] tokens, [U][Cs] clusters
  void* chat;
  int32_t* assign;
  int* seg_counts;
  int* seg_offsets;
  int* slots;
  void* mu;
  float* valsum;
  int* cnt;
  int* off;
  int* perm;
  int* nonempty;
  void* tK;   // permutation scratch [U][S][128]
  void* tV;
};
cudaError_t wi_launch_set_int(int* p, int v, cudaStream_t st);
cudaError_t wi_launch_grow(const WiGeom& g, const WiDecodeBufs& b, const WiGrowBufs& w, void* mu, float* valsum,
                           void* valsum16, int* cnt, int* off, int* perm, int* nonempty, int gi, int k_after,
                           int* err, cudaStream_t st);

