// wi_tier.cu -- the wave buffer: the build's clustered K/V rows in host memory,
// a cache of their pages in device memory, replacement run by a host thread.
//
// RetroInfer's wave buffer (summaries de/fr/zh section 2.B) keeps the KV cache
// in CPU memory, caches the blocks attention keeps retrieving in a GPU block
// cache (retrieved tokens recur from one decode step to the next), and lets the
// CPU run the LRU replacement and the data movement asynchronously while the
// GPU computes; an execution buffer feeds the attention kernel the tokens from
// the steady zone, the cache and the CPU.  Here:
//   * a page is kWiPageRows consecutive rows of a unit's K and V in the index's
//     cluster-contiguous order (a retrieved cluster covers one page or a few);
//   * the rows live in page-locked host memory mapped into the device's address
//     space; on a Grace-Blackwell node the GPU reads it over NVLink-C2C;
//   * every unit has `slots` cache pages in device memory; slot_of[u][p] names
//     the slot holding page p, or -1;
//   * the exact-attention kernel is the execution buffer: its producer warp
//     copies every retrieved row into the shared-memory stages from the cached
//     page or straight from host memory, and stamps each page it read with the
//     step number (use[u][p]);
//   * a replacement round (LruPages) takes the pages read since the previous
//     round: hits become most recently used, misses are admitted into free or
//     least-recently-used slots.  The round unmaps the victims on the decode
//     stream, fills their slots from host memory on a side stream, and maps the
//     new pages on the decode stream once the fill has landed, so a decode step
//     never waits for the host and never reads a slot being refilled;
//   * the rounds run on a host thread, one at a time, each on the newest
//     snapshot of the stamps (taken on the decode stream when the thread is
//     idle), or synchronously on request.
// Where a row is read from does not change any result: the stages hold the
// same rows in the same order either way.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <condition_variable>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <mutex>
#include <new>
#include <queue>
#include <thread>
#include <utility>
#include <vector>

#include "wave_index.h"
#include "wi_common.cuh"
#include "wi_internal.h"

namespace {

// Replacement rounds of one unit's page cache.  In one round the pages read since the previous
// round are taken in increasing order: a cached page becomes the most recently used; a page not
// cached is admitted (at most admit_max per round) into the lowest free slot, else into the slot of
// the least recently used page unless that page was read in this same round (then every cached page
// was, and the round admits nothing more); an admitted page is the most recently used.
class LruPages {
 public:
  LruPages(int pages, int slots, int admit_max)
      : slots_(slots), admit_(admit_max), slot_of_(pages, -1), page_of_(slots, -1), prev_(slots, -1),
        next_(slots, -1), stamp_(slots, -1) {
    for (int s = 0; s < slots; ++s) free_.push(s);
  }

  int slot_of(int p) const { return slot_of_[p]; }
  int pages() const { return (int)slot_of_.size(); }

  // touched: ascending, distinct, in [0, pages)
  void round(const int* touched, int n, long long t, std::vector<std::pair<int, int>>* ev,
             std::vector<std::pair<int, int>>* ad) {
    int admitted = 0;
    for (int i = 0; i < n; ++i) {
      const int p = touched[i];
      int s = slot_of_[p];
      if (s >= 0) {  // hit
        unlink(s);
        append(s);
        stamp_[s] = t;
        continue;
      }
      if (admitted >= admit_) continue;
      if (!free_.empty()) {
        s = free_.top();
        free_.pop();
      } else {
        s = head_;
        if (s < 0 || stamp_[s] == t) continue;  // no slots, or every cached page was read this round
        unlink(s);
        const int victim = page_of_[s];
        slot_of_[victim] = -1;
        ev->emplace_back(victim, s);
      }
      page_of_[s] = p;
      slot_of_[p] = s;
      stamp_[s] = t;
      append(s);
      ad->emplace_back(p, s);
      ++admitted;
    }
  }

 private:
  int slots_, admit_;
  std::vector<int> slot_of_, page_of_, prev_, next_;
  std::vector<long long> stamp_;
  int head_ = -1, tail_ = -1;  // recency list of the used slots: head = least recently used
  std::priority_queue<int, std::vector<int>, std::greater<int>> free_;

  void unlink(int s) {
    if (prev_[s] >= 0) next_[prev_[s]] = next_[s]; else head_ = next_[s];
    if (next_[s] >= 0) prev_[next_[s]] = prev_[s]; else tail_ = prev_[s];
    prev_[s] = next_[s] = -1;
  }
  void append(int s) {
    prev_[s] = tail_;
    next_[s] = -1;
    if (tail_ >= 0) next_[tail_] = s; else head_ = s;
    tail_ = s;
  }
};

// table[patch[i].x] = patch[i].y.
__global__ void k_tier_patch(int* __restrict__ table, const int2* __restrict__ patch, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const int2 e = patch[i];
    table[e.x] = e.y;
  }
}

// One CTA per entry (unit, page, slot): the page's kWiPageRows K and V rows from host memory into
// the slot (16-byte words, all of the CTA's threads).
__global__ void k_tier_fill(const uint4* __restrict__ hostK, const uint4* __restrict__ hostV, uint4* __restrict__ poolK,
                            uint4* __restrict__ poolV, const int4* __restrict__ list, long long n_rows, int slots) {
  const int4 e = list[blockIdx.x];  // (unit, page, slot, 0)
  constexpr int kW = kWiPageRows * WI_D * 2 / 16;  // 16-byte words of one page of K (or V)
  const size_t src = ((size_t)e.x * n_rows + (size_t)e.y * kWiPageRows) * WI_D * 2 / 16;
  const size_t dst = ((size_t)e.x * slots + e.z) * kW;
  for (int i = threadIdx.x; i < 2 * kW; i += blockDim.x) {
    if (i < kW) poolK[dst + i] = hostK[src + i];
    else poolV[dst + i - kW] = hostV[src + i - kW];
  }
}

}  // namespace

struct WiTierHost {
  WiGeom g{};
  int slots = 0, pages = 0, admit = 0;
  bool async = false;
  int device = 0;
  std::vector<LruPages> pol;
  // device
  int* slot_of = nullptr;
  int* use = nullptr;
  void* poolK = nullptr;
  void* poolV = nullptr;
  void* steadyK = nullptr;
  void* steadyV = nullptr;
  unsigned long long* rows_src = nullptr;
  // page-locked host memory
  void* hostK = nullptr;
  void* hostV = nullptr;
  void* hostK_d = nullptr;  // their device addresses
  void* hostV_d = nullptr;
  int* use_h = nullptr;     // snapshot of `use`
  int2* patch_h = nullptr;  // [2][cap] unmap, map
  int4* fill_h = nullptr;   // [cap]
  int2* patch_d = nullptr;
  int4* fill_d = nullptr;
  size_t cap = 0;           // entries per patch (U * admit)
  cudaStream_t side = nullptr;
  cudaEvent_t ev_snap = nullptr, ev_unmap = nullptr, ev_fill = nullptr, ev_map = nullptr;
  long long last_round = -1;
  // counters (rounds, pages touched, hits, misses, admitted, evicted)
  std::atomic<long long> stat[6];
  // worker
  std::thread th;
  std::mutex mu;
  std::condition_variable cv;
  bool stop = false, busy = false, pending = false;
  long long pend_step = 0;
  cudaStream_t pend_stream = nullptr;
  std::atomic<int> werr{0};
  char wmsg[256] = {0};

  WiTierHost() {
    for (auto& s : stat) s = 0;
  }
};

namespace {

int tier_fail(char* msg, size_t len, int code, const char* what, cudaError_t e) {
  snprintf(msg, len, "%s: %s", what, cudaGetErrorString(e));
  return code;
}

// One replacement round over the snapshot in use_h, taken after step t was enqueued.
int run_round(WiTierHost* T, long long t, cudaStream_t st, char* msg, size_t len) {
  const int U = T->g.U, P = T->pages;
  std::vector<int> touched;
  std::vector<std::pair<int, int>> ev, ad;
  size_t n_un = 0, n_map = 0;
  int2* unmap = T->patch_h;
  int2* map = T->patch_h + T->cap;
  for (int u = 0; u < U; ++u) {
    touched.clear();
    const int* us = T->use_h + (size_t)u * P;
    for (int p = 0; p < P; ++p)
      if (us[p] > T->last_round && us[p] <= t) touched.push_back(p);
    long long hits = 0;
    for (int p : touched) hits += T->pol[u].slot_of(p) >= 0;
    ev.clear();
    ad.clear();
    T->pol[u].round(touched.data(), (int)touched.size(), t, &ev, &ad);
    T->stat[1] += (long long)touched.size();
    T->stat[2] += hits;
    T->stat[3] += (long long)touched.size() - hits;
    T->stat[4] += (long long)ad.size();
    T->stat[5] += (long long)ev.size();
    for (auto& e : ev) unmap[n_un++] = make_int2(u * P + e.first, -1);
    for (auto& a : ad) {
      T->fill_h[n_map] = make_int4(u, a.first, a.second, 0);
      map[n_map++] = make_int2(u * P + a.first, a.second);
    }
  }
  T->stat[0] += 1;
  T->last_round = t;
  if (n_map == 0) return WI_OK;
  cudaError_t e;
  // the lists go to device buffers by stream-ordered copies from page-locked memory; the host side is
  // rewritten only by the next round, after this one has waited for all of its work
  if (n_un > 0) {
    if ((e = cudaMemcpyAsync(T->patch_d, unmap, n_un * sizeof(int2), cudaMemcpyHostToDevice, st)) != cudaSuccess)
      return tier_fail(msg, len, WI_ECUDA, "tier unmap copy", e);
    k_tier_patch<<<(unsigned)((n_un + 255) / 256), 256, 0, st>>>(T->slot_of, T->patch_d, (int)n_un);
    if ((e = cudaGetLastError()) != cudaSuccess) return tier_fail(msg, len, WI_ECUDA, "tier unmap", e);
  }
  // the victims' slots are refilled only after every step enqueued before the unmap
  if ((e = cudaEventRecord(T->ev_unmap, st)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(T->side, T->ev_unmap, 0)) != cudaSuccess)
    return tier_fail(msg, len, WI_ECUDA, "tier ordering", e);
  if ((e = cudaMemcpyAsync(T->fill_d, T->fill_h, n_map * sizeof(int4), cudaMemcpyHostToDevice, T->side)) !=
      cudaSuccess)
    return tier_fail(msg, len, WI_ECUDA, "tier fill list copy", e);
  k_tier_fill<<<(unsigned)n_map, 256, 0, T->side>>>(
      static_cast<const uint4*>(T->hostK_d), static_cast<const uint4*>(T->hostV_d), static_cast<uint4*>(T->poolK),
      static_cast<uint4*>(T->poolV), T->fill_d, T->g.n, T->slots);
  if ((e = cudaGetLastError()) != cudaSuccess) return tier_fail(msg, len, WI_ECUDA, "tier fill", e);
  if ((e = cudaEventRecord(T->ev_fill, T->side)) != cudaSuccess ||
      (e = cudaEventSynchronize(T->ev_fill)) != cudaSuccess)
    return tier_fail(msg, len, WI_ECUDA, "tier fill wait", e);
  // the fill has landed: later steps may read the new pages from their slots
  if ((e = cudaMemcpyAsync(T->patch_d + T->cap, map, n_map * sizeof(int2), cudaMemcpyHostToDevice, st)) !=
      cudaSuccess)
    return tier_fail(msg, len, WI_ECUDA, "tier map copy", e);
  k_tier_patch<<<(unsigned)((n_map + 255) / 256), 256, 0, st>>>(T->slot_of, T->patch_d + T->cap, (int)n_map);
  if ((e = cudaGetLastError()) != cudaSuccess) return tier_fail(msg, len, WI_ECUDA, "tier map", e);
  if ((e = cudaEventRecord(T->ev_map, st)) != cudaSuccess || (e = cudaEventSynchronize(T->ev_map)) != cudaSuccess)
    return tier_fail(msg, len, WI_ECUDA, "tier map wait", e);
  return WI_OK;
}

int snapshot(WiTierHost* T, cudaStream_t st, char* msg, size_t len) {
  cudaError_t e;
  if ((e = cudaMemcpyAsync(T->use_h, T->use, (size_t)T->g.U * T->pages * 4, cudaMemcpyDeviceToHost, st)) !=
          cudaSuccess ||
      (e = cudaEventRecord(T->ev_snap, st)) != cudaSuccess)
    return tier_fail(msg, len, WI_ECUDA, "tier snapshot", e);
  return WI_OK;
}

void worker(WiTierHost* T) {
  cudaSetDevice(T->device);
  std::unique_lock<std::mutex> lk(T->mu);
  for (;;) {
    T->cv.wait(lk, [T] { return T->stop || T->pending; });
    if (T->stop) return;
    T->pending = false;
    T->busy = true;
    const long long t = T->pend_step;
    cudaStream_t st = T->pend_stream;
    lk.unlock();
    int rc = WI_OK;
    char msg[256] = {0};
    cudaError_t e = cudaEventSynchronize(T->ev_snap);
    if (e != cudaSuccess) rc = tier_fail(msg, sizeof(msg), WI_ECUDA, "tier snapshot wait", e);
    if (rc == WI_OK) {
      try {
        rc = run_round(T, t, st, msg, sizeof(msg));
      } catch (...) {  // host memory for the round's lists ran out: the thread stops its rounds
        snprintf(msg, sizeof(msg), "tier round: host allocation failed");
        rc = WI_ENOMEM;
      }
    }
    lk.lock();
    if (rc != WI_OK && T->werr.load() == 0) {
      snprintf(T->wmsg, sizeof(T->wmsg), "%s", msg);
      T->werr = rc;
    }
    T->busy = false;
    T->cv.notify_all();
  }
}

}  // namespace

int wi_tier_create(const WiGeom& g, const void* K, const void* V, int slots, int admit, int async, int device,
                   cudaStream_t st, WiTierHost** out, WiTierDev* dev, char* msg, size_t len) {
  *out = nullptr;
  const int pages = (int)((g.n + kWiPageRows - 1) / kWiPageRows);
  if (slots < 0 || slots > pages) {
    snprintf(msg, len, "slots per unit must be in [0, %d] (got %d)", pages, slots);
    return WI_EINVAL;
  }
  if (admit < 0) {
    snprintf(msg, len, "admit_per_round must be >= 0");
    return WI_EINVAL;
  }
  WiTierHost* T = new (std::nothrow) WiTierHost();
  if (!T) {
    snprintf(msg, len, "tier: host allocation failed");
    return WI_ENOMEM;
  }
  T->g = g;
  T->slots = slots;
  T->pages = pages;
  T->admit = std::min(admit, pages);  // a round reads at most `pages` distinct pages of a unit
  T->async = async != 0;
  T->device = device;
  T->cap = std::max<size_t>(1, (size_t)g.U * (size_t)T->admit);
  const size_t U = g.U, rows = (size_t)g.U * g.n, ns = (size_t)g.n_sink + g.W;
  cudaError_t e = cudaSuccess;
  // fault injection for the error path: WI_FAIL_TIER_ALLOC_AT=n makes the n-th allocation (device or
  // page-locked host) of the tier report out-of-memory, nothing allocated
  const char* fenv = getenv("WI_FAIL_TIER_ALLOC_AT");
  const int fail_at = fenv ? atoi(fenv) : 0;
  int n_alloc = 0;
  auto refused = [&]() { return ++n_alloc == fail_at; };
  auto A = [&](void** p, size_t bytes) {
    if (e == cudaSuccess) e = refused() ? cudaErrorMemoryAllocation : cudaMalloc(p, std::max<size_t>(bytes, 16));
  };
  auto H = [&](void** p, size_t bytes, unsigned flags) {
    if (e == cudaSuccess) e = refused() ? cudaErrorMemoryAllocation : cudaHostAlloc(p, std::max<size_t>(bytes, 16), flags);
  };
  A(reinterpret_cast<void**>(&T->slot_of), U * pages * 4);
  A(reinterpret_cast<void**>(&T->use), U * pages * 4);
  A(&T->poolK, U * (size_t)slots * kWiPageRows * WI_D * 2);
  A(&T->poolV, U * (size_t)slots * kWiPageRows * WI_D * 2);
  A(&T->steadyK, U * ns * WI_D * 2);
  A(&T->steadyV, U * ns * WI_D * 2);
  A(reinterpret_cast<void**>(&T->rows_src), 16);
  A(reinterpret_cast<void**>(&T->patch_d), 2 * T->cap * sizeof(int2));
  A(reinterpret_cast<void**>(&T->fill_d), T->cap * sizeof(int4));
  H(&T->hostK, rows * WI_D * 2, cudaHostAllocMapped);
  H(&T->hostV, rows * WI_D * 2, cudaHostAllocMapped);
  H(reinterpret_cast<void**>(&T->use_h), U * pages * 4, cudaHostAllocDefault);
  H(reinterpret_cast<void**>(&T->patch_h), 2 * T->cap * sizeof(int2), cudaHostAllocDefault);
  H(reinterpret_cast<void**>(&T->fill_h), T->cap * sizeof(int4), cudaHostAllocDefault);
  if (e == cudaSuccess) e = cudaHostGetDevicePointer(&T->hostK_d, T->hostK, 0);
  if (e == cudaSuccess) e = cudaHostGetDevicePointer(&T->hostV_d, T->hostV, 0);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&T->side, cudaStreamNonBlocking);
  for (cudaEvent_t* ev : {&T->ev_snap, &T->ev_unmap, &T->ev_fill, &T->ev_map})
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    const int code = (e == cudaErrorMemoryAllocation) ? WI_ENOMEM : WI_ECUDA;
    if (n_alloc == fail_at) snprintf(msg, len, "tier allocation %d refused (WI_FAIL_TIER_ALLOC_AT)", fail_at);
    else tier_fail(msg, len, code, "tier allocation", e);
    wi_tier_destroy(T);
    return code;
  }
  // the index's permuted rows to host memory; the sinks and the window to the steady copy
  const size_t rb = WI_D * 2, pitch = (size_t)g.n * rb;
  if (e == cudaSuccess) e = cudaMemcpyAsync(T->hostK, K, rows * rb, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(T->hostV, V, rows * rb, cudaMemcpyDeviceToHost, st);
  for (int kv = 0; kv < 2 && e == cudaSuccess; ++kv) {
    const char* src = static_cast<const char*>(kv ? V : K);
    char* dst = static_cast<char*>(kv ? T->steadyV : T->steadyK);
    if (g.n_sink > 0)
      e = cudaMemcpy2DAsync(dst, ns * rb, src, pitch, (size_t)g.n_sink * rb, U, cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess && g.W > 0)
      e = cudaMemcpy2DAsync(dst + (size_t)g.n_sink * rb, ns * rb, src + (size_t)(g.n - g.W) * rb, pitch,
                            (size_t)g.W * rb, U, cudaMemcpyDeviceToDevice, st);
  }
  if (e == cudaSuccess) e = cudaMemsetAsync(T->slot_of, 0xFF, U * pages * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(T->use, 0xFF, U * pages * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(T->rows_src, 0, 16, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);  // the caller's K and V are no longer read after this
  if (e != cudaSuccess) {
    tier_fail(msg, len, WI_ECUDA, "tier copy-out", e);
    wi_tier_destroy(T);
    return WI_ECUDA;
  }
  try {
    T->pol.reserve(U);
    for (size_t u = 0; u < U; ++u) T->pol.emplace_back(pages, slots, T->admit);
    if (T->async) T->th = std::thread(worker, T);
  } catch (...) {  // host memory for the policy, or the replacement thread, could not be had
    snprintf(msg, len, "tier: the replacement policy or its thread could not be set up");
    wi_tier_destroy(T);
    return WI_ENOMEM;
  }
  dev->on = 1;
  dev->slots = slots;
  dev->pages = pages;
  dev->step = 0;
  dev->slot_of = T->slot_of;
  dev->poolK = T->poolK;
  dev->poolV = T->poolV;
  dev->hostK = T->hostK_d;
  dev->hostV = T->hostV_d;
  dev->steadyK = T->steadyK;
  dev->steadyV = T->steadyV;
  dev->use = T->use;
  dev->rows_src = T->rows_src;
  *out = T;
  return WI_OK;
}

void wi_tier_destroy(WiTierHost* T) {
  if (!T) return;
  if (T->th.joinable()) {
    {
      std::lock_guard<std::mutex> lk(T->mu);
      T->stop = true;
    }
    T->cv.notify_all();
    T->th.join();
  }
  if (T->side) cudaStreamSynchronize(T->side);
  for (void* p : {(void*)T->slot_of, (void*)T->use, T->poolK, T->poolV, T->steadyK, T->steadyV, (void*)T->rows_src,
                  (void*)T->patch_d, (void*)T->fill_d})
    if (p) cudaFree(p);
  for (void* p : {T->hostK, T->hostV, (void*)T->use_h, (void*)T->patch_h, (void*)T->fill_h})
    if (p) cudaFreeHost(p);
  for (cudaEvent_t ev : {T->ev_snap, T->ev_unmap, T->ev_fill, T->ev_map})
    if (ev) cudaEventDestroy(ev);
  if (T->side) cudaStreamDestroy(T->side);
  delete T;
}

// After decode step `step` was enqueued on st: if the replacement thread is idle, snapshot the page
// stamps behind the step and hand the round to the thread.
int wi_tier_after_step(WiTierHost* T, long long step, cudaStream_t st, char* msg, size_t len) {
  if (!T->async) return WI_OK;
  std::lock_guard<std::mutex> lk(T->mu);
  if (T->werr.load() != 0) {
    snprintf(msg, len, "tier replacement thread: %s", T->wmsg);
    return T->werr.load();
  }
  if (T->busy || T->pending) return WI_OK;
  const int rc = snapshot(T, st, msg, len);
  if (rc != WI_OK) return rc;
  T->pend_step = step;
  T->pend_stream = st;
  T->pending = true;
  T->cv.notify_all();
  return WI_OK;
}

// One round now, on this thread, over the stamps of every step enqueued so far (last = step).
int wi_tier_round_now(WiTierHost* T, long long step, cudaStream_t st, char* msg, size_t len) {
  std::unique_lock<std::mutex> lk(T->mu);
  T->cv.wait(lk, [T] { return !T->busy && !T->pending; });
  if (T->werr.load() != 0) {
    snprintf(msg, len, "tier replacement thread: %s", T->wmsg);
    return T->werr.load();
  }
  T->busy = true;
  lk.unlock();
  int rc = snapshot(T, st, msg, len);
  if (rc == WI_OK) {
    const cudaError_t e = cudaEventSynchronize(T->ev_snap);
    if (e != cudaSuccess) rc = tier_fail(msg, len, WI_ECUDA, "tier snapshot wait", e);
  }
  if (rc == WI_OK) {
    try {
      rc = run_round(T, step, st, msg, len);
    } catch (...) {
      snprintf(msg, len, "tier round: host allocation failed");
      rc = WI_ENOMEM;
    }
  }
  lk.lock();
  T->busy = false;
  T->cv.notify_all();
  return rc;
}

// Waits until no round is running or pending.
void wi_tier_idle(WiTierHost* T) {
  std::unique_lock<std::mutex> lk(T->mu);
  T->cv.wait(lk, [T] { return !T->busy && !T->pending; });
}

void wi_tier_counters(WiTierHost* T, long long out[6]) {
  for (int i = 0; i < 6; ++i) out[i] = T->stat[i].load();
}

int wi_tier_geometry(const WiTierHost* T, int* slots, int* pages) {
  *slots = T->slots;
  *pages = T->pages;
  return WI_OK;
}

const int* wi_tier_slot_table(const WiTierHost* T) { return T->slot_of; }
const int* wi_tier_use_table(const WiTierHost* T) { return T->use; }
const unsigned long long* wi_tier_row_counters(const WiTierHost* T) { return T->rows_src; }

// ---- the replacement policy alone, for checking on the host (no device involved)
static int lru_round_impl(LruPages* L, const int32_t* touched, int n, long long t, int32_t* ev_pages,
                          int32_t* ev_slots, int* n_ev, int32_t* ad_pages, int32_t* ad_slots, int* n_ad);

extern "C" {

void* wi_lru_new(int pages, int slots, int admit_max) {
  if (pages < 1 || slots < 0 || admit_max < 0) return nullptr;
  try {
    return new LruPages(pages, slots, admit_max);
  } catch (...) {
    return nullptr;
  }
}

int wi_lru_round(void* h, const int32_t* touched, int n, long long t, int32_t* ev_pages, int32_t* ev_slots,
                 int* n_ev, int32_t* ad_pages, int32_t* ad_slots, int* n_ad) {
  if (!h || n < 0 || (n > 0 && !touched) || !n_ev || !n_ad) return WI_EINVAL;
  LruPages* L = static_cast<LruPages*>(h);
  try {
    return lru_round_impl(L, touched, n, t, ev_pages, ev_slots, n_ev, ad_pages, ad_slots, n_ad);
  } catch (...) {
    return WI_ENOMEM;
  }
}

}  // extern "C"

static int lru_round_impl(LruPages* L, const int32_t* touched, int n, long long t, int32_t* ev_pages,
                          int32_t* ev_slots, int* n_ev, int32_t* ad_pages, int32_t* ad_slots, int* n_ad) {
  std::vector<int> tp(touched, touched + n);
  std::sort(tp.begin(), tp.end());
  tp.erase(std::unique(tp.begin(), tp.end()), tp.end());
  for (int p : tp)
    if (p < 0 || p >= L->pages()) return WI_EINVAL;
  std::vector<std::pair<int, int>> ev, ad;
  L->round(tp.data(), (int)tp.size(), t, &ev, &ad);
  *n_ev = (int)ev.size();
  *n_ad = (int)ad.size();
  for (size_t i = 0; i < ev.size(); ++i) {
    if (ev_pages) ev_pages[i] = ev[i].first;
    if (ev_slots) ev_slots[i] = ev[i].second;
  }
  for (size_t i = 0; i < ad.size(); ++i) {
    if (ad_pages) ad_pages[i] = ad[i].first;
    if (ad_slots) ad_slots[i] = ad[i].second;
  }
  return WI_OK;
}

extern "C" void wi_lru_free(void* h) { delete static_cast<LruPages*>(h); }
