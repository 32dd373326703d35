// wi_assign_tc.cu -- spherical k-means assignment on the 5th-generation
// tensor cores: a_i = argmax_j K_i . c_j over a segment's centroids.
//
// Spherical k-means (RetroInfer summary fr 2.A.2) inside segmented
// clustering (summaries de/fr/zh 2.A): every segment of S tokens is assigned
// to its own Cs centroids.  Per segment this is the dense contraction
// [S x 128] . [128 x Cs] (bf16 operands, fp32 accumulation) followed by a row
// argmax, ties to the lowest centroid id.
//
// Kernel structure (one persistent CTA per SM, 1 CTA / SM):
//   warp 0       TMA producer: the segment's centroids (B, Cs x 128, K-major,
//                128-byte swizzle) once per segment, token tiles (A, 128 x 128)
//                through a 2-stage ring;
//   warp 1       allocates the 512 TMEM columns and issues tcgen05.mma
//                (M = 128, N = min(Cs, 256), K = 16 per instruction) into one
//                of two accumulator halves, so that the argmax of one half
//                overlaps the products of the other;
//   warps 2..17  epilogue: tcgen05.ld of the accumulator rows (warp w reads
//                TMEM lanes 32*(w%4)..+31), running argmax over its column
//                share (four column groups), combine through shared memory,
//                store.
// Every mbarrier wait is bounded (wi_pipe.cuh); on a timeout the kernel
// records WI_DEVERR_MBAR_TIMEOUT, waits for its own copies and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <mutex>

#include "wi_common.cuh"
#include "wi_internal.h"
#include "wi_pipe.cuh"
#include "wi_tc.cuh"

namespace {

constexpr int kTM = 128;                 // tokens per tile (MMA M)
constexpr int kStagesA = 3;
constexpr int kEpiWarps = 16;                  // four column groups of four warps (one per TMEM lane quarter)
constexpr int kGroups = kEpiWarps / 4;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kATileBytes = kTM * WI_D * 2;  // 32 KB: two 16 KB halves of 64 columns
constexpr int kMaxCs = 512;
constexpr int kBBytes = kMaxCs * WI_D * 2;   // 128 KB

struct TcSmem {
  // small state first (3 KB), then the 1024-byte aligned tiles for the 128-byte swizzle
  float best_v[kGroups - 1][kTM];           // epilogue combine: column groups 1.. x row
  uint16_t best_j[kGroups - 1][kTM];
  uint64_t full_a[kStagesA], empty_a[kStagesA];
  uint64_t full_b, b_free;
  uint64_t tmem_full[2], tmem_empty[2];
  uint32_t tmem_base;
  int abort_flag;
  unsigned char pad[3072 - (kGroups - 1) * kTM * 6 - (2 * kStagesA + 6) * 8 - 8];
  unsigned char b[kBBytes];                 // [k half][Cs rows][128 B]
  unsigned char a[kStagesA][kATileBytes];   // [k half][128 rows][128 B]
};
static_assert(offsetof(TcSmem, b) == 3072, "tile region must start 1024-byte aligned");

struct TcParams {
  int32_t* assign;
  int* err;
  long long n;      // tokens per unit
  int S, Cs, nseg;  // segment length, centroids per segment, segments per unit
  int n_sink, W;
  int total_tiles;  // (units * nseg) * (S / 128)
  int N, halves;    // MMA N and number of accumulator halves (Cs = N * halves)
};

__global__ void __launch_bounds__(kThreads, 1) k_assign_tc(const __grid_constant__ CUtensorMap map_k,
                                                          const __grid_constant__ CUtensorMap map_c,
                                                          TcParams P) {
  extern __shared__ __align__(1024) unsigned char tc_raw[];
  TcSmem& sm = *reinterpret_cast<TcSmem*>(tc_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (smem_addr(sm.b) & 1023u) {  // the swizzled tiles need 1024-byte alignment; never run misaligned
    if (tid == 0) atomicOr(P.err, WI_DEVERR_BAD_ROW);
    return;
  }
  const int tiles_per_seg = P.S / kTM;
  const int t0 = (int)((long long)P.total_tiles * blockIdx.x / gridDim.x);
  const int t1 = (int)((long long)P.total_tiles * (blockIdx.x + 1) / gridDim.x);
  const uint32_t idesc = make_idesc(kTM, P.N);
  if (tid == 0) {
    for (int s = 0; s < kStagesA; ++s) {
      mbar_init(&sm.full_a[s], 1);
      mbar_init(&sm.empty_a[s], 1);
    }
    mbar_init(&sm.full_b, 1);
    mbar_init(&sm.b_free, 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(&sm.tmem_full[h], 1);
      mbar_init(&sm.tmem_empty[h], kEpiWarps);
    }
    sm.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {  // the whole warp allocates all 512 columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_addr(&sm.tmem_base))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_k)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_c)) : "memory");
      int cur_su = -1, bloads = 0, issued = 0;
      bool ok = true;
      const uint32_t bbytes = (uint32_t)P.Cs * WI_D * 2;
      for (int t = t0; t < t1 && ok; ++t) {
        const int su = t / tiles_per_seg, mt = t % tiles_per_seg;
        if (su != cur_su) {
          if (bloads > 0 && !mbar_wait(&sm.b_free, (bloads - 1) & 1, P.err)) { ok = false; break; }
          mbar_arrive_expect_tx(&sm.full_b, bbytes);
          for (int r0 = 0; r0 < P.Cs; r0 += 256) {
            const int rows = P.Cs - r0 < 256 ? P.Cs - r0 : 256;
            (void)rows;
            // k half 0 region: rows at r0 * 128 B; k half 1 region after all Cs rows
            tma_load_2d(sm.b + r0 * 128, &map_c, 0, su * P.Cs + r0, &sm.full_b);
            tma_load_2d(sm.b + P.Cs * 128 + r0 * 128, &map_c, 64, su * P.Cs + r0, &sm.full_b);
          }
          cur_su = su;
          ++bloads;
        }
        const int it = t - t0, s = it % kStagesA, r = it / kStagesA;
        if (r > 0 && !mbar_wait(&sm.empty_a[s], (r - 1) & 1, P.err)) { ok = false; break; }
        mbar_arrive_expect_tx(&sm.full_a[s], kATileBytes);
        const long long row0 = (long long)(su / P.nseg) * P.n + (long long)(su % P.nseg) * P.S + (long long)mt * kTM;
        tma_load_2d(sm.a[s], &map_k, 0, (int)row0, &sm.full_a[s]);
        tma_load_2d(sm.a[s] + kATileBytes / 2, &map_k, 64, (int)row0, &sm.full_a[s]);
        issued = it + 1;
      }
      if (!ok) {
        sm.abort_flag = 1;
        for (int s = 0; s < kStagesA && s < issued; ++s) {
          const int last = ((issued - 1 - s) / kStagesA) * kStagesA + s;
          mbar_wait(&sm.full_a[s], (last / kStagesA) & 1, P.err);
        }
        if (bloads > 0) mbar_wait(&sm.full_b, (bloads - 1) & 1, P.err);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (one lane)
    if (lane == 0) {
      int cur_su = -1, bloads = 0;
      bool ok = true;
      for (int t = t0; t < t1 && ok; ++t) {
        const int su = t / tiles_per_seg;
        if (su != cur_su) {
          if (!mbar_wait(&sm.full_b, bloads & 1, P.err)) { ok = false; break; }
          cur_su = su;
          ++bloads;
          tc_fence_after();
        }
        const int it = t - t0, s = it % kStagesA, r = it / kStagesA;
        if (!mbar_wait(&sm.full_a[s], r & 1, P.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a0 = smem_addr(sm.a[s]);
        const uint32_t b0 = smem_addr(sm.b);
        for (int h = 0; h < P.halves; ++h) {
          if (it > 0 && !mbar_wait(&sm.tmem_empty[h], (it - 1) & 1, P.err)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < WI_D / 16; ++kk) {
            // k step kk: 16 columns = 32 bytes inside the 128-byte swizzle row of k half kk / 4
            const uint32_t aoff = (uint32_t)(kk >> 2) * (kATileBytes / 2) + (uint32_t)(kk & 3) * 32;
            const uint32_t boff = (uint32_t)(kk >> 2) * (uint32_t)(P.Cs * 128) + (uint32_t)h * (uint32_t)(P.N * 128) +
                                  (uint32_t)(kk & 3) * 32;
            mma_bf16(tmem + (uint32_t)(h * P.N), make_desc_sw128(a0 + aoff), make_desc_sw128(b0 + boff), idesc,
                     kk > 0 ? 1u : 0u);
          }
          mma_commit(&sm.tmem_full[h]);
        }
        if (!ok) break;
        mma_commit(&sm.empty_a[s]);  // the A stage is free once these products are done
        const bool last_of_seg = (t + 1 == t1) || ((t + 1) / tiles_per_seg != su);
        if (last_of_seg) mma_commit(&sm.b_free);
      }
      if (!ok) sm.abort_flag = 1;
    }
  } else {
    // ---------------- epilogue: warps 2..2+kEpiWarps-1
    const int ew = warp - 2;
    const int quarter = warp & 3;       // TMEM lane quarter this warp may access
    const int cgroup = ew >> 2;         // column group g takes columns [g*cols, (g+1)*cols) of each N block
    const int row = quarter * 32 + lane;
    const int groups = min(kGroups, P.N / 32);     // groups with columns (N = 64: two)
    const int cols = P.N / groups;                 // columns per group per half (multiple of 32)
    const int my_cols = cgroup < groups ? cols : 0;  // a group without columns still meets every barrier
    bool ok = true;                     // after one timed-out wait the warp stops waiting but keeps
                                        // meeting the epilogue barriers, so no warp is left behind
    // the row's running argmax as kChains independent chains over interleaved columns (column i goes
    // to chain i % kChains, each chain keeps its first maximum), so that the compares do not form one
    // dependent chain; combined at the end with ties to the lowest column
    constexpr int kChains = 8;
    for (int t = t0; t < t1; ++t) {
      const int it = t - t0;
      const int su = t / tiles_per_seg, mt = t % tiles_per_seg;
      float cv[kChains];
      int cj[kChains];
#pragma unroll
      for (int c = 0; c < kChains; ++c) { cv[c] = -INFINITY; cj[c] = 0x7fffffff; }
      for (int h = 0; h < P.halves && ok; ++h) {
        if (!mbar_wait(&sm.tmem_full[h], it & 1, P.err)) { ok = false; sm.abort_flag = 1; break; }
        tc_fence_after();
        for (int c0 = 0; c0 < my_cols; c0 += 32) {  // 32 columns per load (the other warps hide its wait)
          const int col = h * P.N + cgroup * cols + c0;
          const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)col;
          uint32_t r0[32];
          tmem_ld32_nowait(ta, r0);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float v = __uint_as_float(r0[i]);
            if (v > cv[i % kChains]) { cv[i % kChains] = v; cj[i % kChains] = col + i; }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.tmem_empty[h]);
      }
      float bv = cv[0];
      int bj = cj[0];
#pragma unroll
      for (int c = 1; c < kChains; ++c)
        if (cv[c] > bv || (cv[c] == bv && cj[c] < bj)) { bv = cv[c]; bj = cj[c]; }
      if (cgroup > 0) {
        sm.best_v[cgroup - 1][row] = bv;
        sm.best_j[cgroup - 1][row] = (uint16_t)min(bj, 0xFFFF);
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
      if (cgroup == 0) {
        for (int g2 = 1; g2 < groups; ++g2) {
          const float ov = sm.best_v[g2 - 1][row];
          const int oj = sm.best_j[g2 - 1][row];
          if (ov > bv || (ov == bv && oj < bj)) { bv = ov; bj = oj; }
        }
        const int u = su / P.nseg, sg = su % P.nseg;
        const long long p = (long long)sg * P.S + (long long)mt * kTM + row;
        int a = -1;
        if (!(p < P.n_sink || p >= P.n - P.W)) {
          if (bj < 0 || bj >= P.Cs) { atomicOr(P.err, WI_DEVERR_BAD_CLUSTER); bj = 0; }
          a = sg * P.Cs + bj;
        }
        if (ok) P.assign[(long long)u * P.n + p] = a;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

}  // namespace


namespace {
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// 2-D bf16 tensor map over rows of 128 elements (256 B), box = 64 columns x box_rows rows, 128-byte swizzle.
bool encode_rows_impl(CUtensorMap* map, const void* base, unsigned long long rows, unsigned box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)WI_D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)WI_D * 2};
  const cuuint32_t box[2] = {64u, box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool wi_encode_rows_sw128(CUtensorMap* map, const void* base, unsigned long long rows, unsigned box_rows) {
  return encode_rows_impl(map, base, rows, box_rows);
}

bool wi_tensor_maps_available() { return get_encode() != nullptr; }

bool wi_assign_tc_supported(const WiGeom& g) {
  if (!(g.Cs == 64 || g.Cs == 128 || g.Cs == 256 || g.Cs == 512)) return false;
  if (g.S % kTM) return false;
  if ((long long)g.U * g.n >= (1LL << 31)) return false;  // TMA row coordinates are 32-bit
  return wi_tensor_maps_available();
}

cudaError_t wi_launch_assign_tc(const WiGeom& g, const void* K, const void* chat, int32_t* assign, int* err,
                                cudaStream_t st) {
  CUtensorMap map_k, map_c;
  const int box_c = g.Cs < 256 ? g.Cs : 256;
  if (!wi_encode_rows_sw128(&map_k, K, (unsigned long long)g.U * g.n, kTM) ||
      !wi_encode_rows_sw128(&map_c, chat, (unsigned long long)g.U * g.nseg * g.Cs, (unsigned)box_c))
    return cudaErrorInvalidValue;
  TcParams P;
  P.assign = assign;
  P.err = err;
  P.n = g.n;
  P.S = g.S;
  P.Cs = g.Cs;
  P.nseg = g.nseg;
  P.n_sink = g.n_sink;
  P.W = g.W;
  P.total_tiles = g.U * g.nseg * (g.S / kTM);
  P.N = g.Cs < 256 ? g.Cs : 256;
  P.halves = g.Cs / P.N;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = P.total_tiles < sms ? P.total_tiles : sms;
  const size_t smem = sizeof(TcSmem);
  static int smem_set[kWiSmemDevices] = {};
  cudaError_t e = wi_ensure_smem(k_assign_tc, smem, smem_set);
  if (e != cudaSuccess) return e;
  k_assign_tc<<<grid, kThreads, smem, st>>>(map_k, map_c, P);
  return cudaGetLastError();
}
