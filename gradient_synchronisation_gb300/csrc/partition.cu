// The push-side h0 partition (zr_partition, zr_partition_static) and Zen's
// index sets (zr_hash_index_sets), one cooperative launch each.
//
// What is computed (Zen page, Problem 1, requirement 1, and section 3.3.2):
// a stable split of one COO list into n_parts partitions by the consistent
// first-level hash h0, partition-major, input order kept inside a partition;
// with the identity input (position i holds index i) the split of [0, M)
// that gives the index sets I_p.
//
// GB300 design.  All CTAs are co-resident (cooperative launch) and wait for
// one another once:
//   1. count   CTA c takes a contiguous slice of the list and counts it per
//              partition (each thread its 16 consecutive entries of a
//              8192-entry tile, in per-thread 16-bit counters, 32 partitions
//              per pass); the CTA's counts go to the workspace.
//   -- grid-wide wait: a CTA that has waited about a second sets
//      ZR_ERR_TIMEOUT and returns, so the wait always ends.
//   2. bases   each CTA sums, per partition, the counts of the CTAs before
//              it and of all CTAs: its first output position in every
//              partition.  CTA 0 writes the offsets.
//   3. place   per tile, a block scan of the per-thread counters gives each
//              thread its slots, the entries go partition-major into a
//              shared staging array, and each partition's run leaves with
//              coalesced stores at the partition's running position.  A
//              slice of one tile stays in shared memory across the wait.
// Every output position is checked against the list length, so nothing is
// written outside the outputs.

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "zr.h"
#include "zr_device.cuh"
#include "zr_internal.h"

namespace zr {
namespace {

constexpr int kT = 512;                  // threads per CTA
constexpr int kW = kT / 32;              // warps per CTA
constexpr int kSlab = 32;                // partitions per counting pass
constexpr int kCntWords = kSlab / 2 * kT;  // packed 16-bit counters: 2 per word
constexpr int kMaxCtas = 1024;           // bound of the grid (sizes the workspace)
constexpr int kHeader = 256;             // status word + barrier counter, cleared per call
constexpr unsigned long long kWaitNs = 1000000000ull;  // grid wait limit, ~1 s
constexpr unsigned kSpinLimit = 1u << 23;              // and an iteration backstop

constexpr int kPTile = 8192;             // entries per tile, 16 per thread
constexpr int kPPer = kPTile / kT;

// The test hook: the CTA with this index skips its arrival at the grid wait.
std::atomic<int> g_barrier_skip{-1};

__device__ __forceinline__ void flag(int32_t* status, int code) { atomicCAS(status, 0, code); }

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int warp_excl_scan(int v, int* total) {
  const int lane = threadIdx.x & 31;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  *total = __shfl_sync(0xffffffffu, x, 31);
  return x - v;
}

template <typename V>
__device__ __forceinline__ V warp_sum(V v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Grid-wide wait of a cooperative launch.  Every CTA arrives once (a release
// by fence, then an atomic add) and thread 0 polls the counter with acquire
// loads.  The wait is bounded: after kWaitNs of the global timer (or
// kSpinLimit polls) it sets ZR_ERR_TIMEOUT and reports failure, and the
// caller returns without writing anything that depends on the other CTAs.
__device__ bool grid_wait(unsigned* counter, unsigned expected, int skip_cta, int32_t* status) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    __threadfence();
    if ((int)blockIdx.x != skip_cta) atomicAdd(counter, 1u);
    const unsigned long long t0 = globaltimer();
    for (unsigned it = 0;; ++it) {
      if (ld_acquire(counter) >= expected) break;
      if (it >= kSpinLimit || globaltimer() - t0 > kWaitNs) {
        flag(status, ZR_ERR_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(128);
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// ---------------------------------------------------------------- counters
// Per-thread partition counters for one slab of kSlab partitions, 16 bits
// each, two per 32-bit word: word (q >> 1) * kT + t holds thread t's counter
// of slab partitions q & ~1 (low half) and q | 1 (high half).  Scanning a
// row of words as integers scans both halves at once (every total here stays
// below 2^16, so the low half never carries into the high one).
__device__ __forceinline__ void counter_add(uint32_t* cw, int q) {
  uint32_t* w = cw + (q >> 1) * kT + threadIdx.x;
  *w += 1u << ((q & 1) * 16);
}

__device__ __forceinline__ int counter_take(uint32_t* cw, int q) {
  uint32_t* w = cw + (q >> 1) * kT + threadIdx.x;
  const uint32_t v = *w;
  *w = v + (1u << ((q & 1) * 16));
  return (int)((v >> ((q & 1) * 16)) & 0xffffu);
}

__device__ __forceinline__ void counters_clear(uint32_t* cw) {
#pragma unroll
  for (int i = 0; i < kSlab / 2; ++i) cw[i * kT + threadIdx.x] = 0;
}

// Exclusive scan over the threads of each counter row (warp w scans row w;
// lane l owns columns 16l .. 16l + 15), then the slab's partition totals
// wtot[s0 .. s0 + 31] and their exclusive prefix wofs[] starting at *run
// (advanced by the slab's total).  Ends with __syncthreads.
__device__ void counters_scan(uint32_t* cw, int s0, int parts, int* wtot, int* wofs, int* run) {
  __shared__ uint32_t row_tot[kSlab / 2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  static_assert(kW == kSlab / 2, "one warp per counter row");
  {
    uint4* p = reinterpret_cast<uint4*>(cw + warp * kT + lane * 16);
    uint4 a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = p[i];
    uint32_t v[16] = {a[0].x, a[0].y, a[0].z, a[0].w, a[1].x, a[1].y, a[1].z, a[1].w,
                      a[2].x, a[2].y, a[2].z, a[2].w, a[3].x, a[3].y, a[3].z, a[3].w};
    uint32_t s = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t x = v[i];
      v[i] = s;
      s += x;
    }
    uint32_t x = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    const uint32_t excl = x - s;
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] += excl;
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    if (lane == 31) row_tot[warp] = x;
  }
  __syncthreads();
  if (warp == 0) {
    const int q = lane;
    const int p = s0 + q;
    const int t = (p < parts) ? (int)((row_tot[q >> 1] >> ((q & 1) * 16)) & 0xffffu) : 0;
    int tot;
    const int ex = warp_excl_scan(t, &tot);
    const int r0 = *run;
    if (p < parts) {
      wtot[p] = t;
      wofs[p] = r0 + ex;
    }
    __syncwarp();
    if (lane == 0) *run = r0 + tot;
  }
  __syncthreads();
}

// Per-CTA partition bases after the grid wait: base[p] = offset of partition
// p + the counts of CTAs c' < c in p.  CTA 0 writes the offsets (when
// requested) and, when d_total is given, the total.  Ends with __syncthreads.
__device__ void partition_bases(const int32_t* cnt_g, int G, int parts, long long* base,
                                long long* d_offsets, long long* d_total) {
  __shared__ long long s_tot[ZR_MAX_PARTS];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x;
  for (int p = warp; p < parts; p += (int)(blockDim.x >> 5)) {
    long long before = 0, all = 0;
    for (int j = lane; j < G; j += 32) {
      const long long v = __ldcg(cnt_g + (size_t)p * G + j);
      all += v;
      if (j < c) before += v;
    }
    before = warp_sum(before);
    all = warp_sum(all);
    if (lane == 0) {
      base[p] = before;
      s_tot[p] = all;
    }
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive prefix of the totals over the partitions, 8 per lane
    long long v[8], s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int p = lane * 8 + i;
      v[i] = p < parts ? s_tot[p] : 0;
      const long long x = v[i];
      v[i] = s;
      s += x;
    }
    long long x = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    const long long excl = x - s;
    const long long total = __shfl_sync(0xffffffffu, x, 31);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int p = lane * 8 + i;
      if (p < parts) {
        const long long off = v[i] + excl;
        base[p] += off;
        if (c == 0 && d_offsets) d_offsets[p] = off;
      }
    }
    if (c == 0 && lane == 0) {
      if (d_offsets) d_offsets[parts] = total;
      if (d_total) *d_total = total;
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------- partition
struct PartArgs {
  const int32_t* idx;  // null: the identity input (position i holds index i)
  const float* val;
  long long nnz;
  int parts;
  H0 h;
  int32_t* out_idx;
  float* out_val;      // null with the identity input
  long long* d_offsets;
  int32_t* status;
  unsigned* barrier;
  int32_t* cnt;        // [parts][G]
  int skip_cta;
};

struct PartShared {
  long long base[ZR_MAX_PARTS];
  int wtot[ZR_MAX_PARTS], wofs[ZR_MAX_PARTS];
  int tot[ZR_MAX_PARTS];
  int run;
  alignas(16) uint32_t cw[kCntWords];
  int32_t key[kPTile];
  float val[kPTile];
  uint8_t part[kPTile];
  int32_t okey[kPTile];
  float oval[kPTile];
  uint8_t opart[kPTile];
};
constexpr size_t kPartSmem = sizeof(PartShared);

// Loads tile [t0, t0 + len) of the list into shared memory and hashes it;
// the values only when with_val (the count pass of a slice that does not
// stay in shared memory across the wait needs the keys alone).
__device__ void part_load(const PartArgs& A, PartShared& S, long long t0, int len,
                          bool with_val) {
  for (int i = threadIdx.x; i < len; i += kT) {
    const long long pos = t0 + i;
    const int32_t k = A.idx ? __ldcs(A.idx + pos) : (int32_t)pos;
    S.key[i] = k;
    if (A.val && with_val) S.val[i] = __ldcs(A.val + pos);
    S.part[i] = (uint8_t)A.h((uint32_t)k);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kT, 1) partition_kernel(const __grid_constant__ PartArgs A) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  PartShared& S = *reinterpret_cast<PartShared*>(smem_raw);
  const int tid = threadIdx.x;
  const int G = gridDim.x, c = blockIdx.x;
  // CTA c's slice [lo, hi): equal slices, multiples of 4 entries
  const long long per = ((A.nnz + G - 1) / G + 3) & ~3ll;
  const long long lo = min((long long)c * per, A.nnz);
  const long long hi = min(lo + per, A.nnz);
  const long long len = hi - lo;
  const bool resident = len <= kPTile;
  for (int p = tid; p < A.parts; p += kT) S.tot[p] = 0;
  __syncthreads();
  // count: per tile, thread t counts its entries [kPPer t, kPPer (t + 1))
  // in its own counters; a warp per counter row adds the row up
  const int lane = tid & 31, warp = tid >> 5;
  for (long long t0 = lo; t0 < hi; t0 += kPTile) {
    const int tl = (int)min((long long)kPTile, hi - t0);
    part_load(A, S, t0, tl, resident);
    const int i0 = tid * kPPer, i1 = min(i0 + kPPer, tl);
    for (int s0 = 0; s0 < A.parts; s0 += kSlab) {
      counters_clear(S.cw);
      for (int i = i0; i < i1; ++i) {
        const int q = (int)S.part[i] - s0;
        if ((unsigned)q < (unsigned)kSlab) counter_add(S.cw, q);
      }
      __syncthreads();
      int s_lo = 0, s_hi = 0;
      for (int j = lane; j < kT; j += 32) {
        const uint32_t v = S.cw[warp * kT + j];
        s_lo += (int)(v & 0xffffu);
        s_hi += (int)(v >> 16);
      }
      s_lo = warp_sum(s_lo);
      s_hi = warp_sum(s_hi);
      if (lane == 0) {
        const int p0 = s0 + 2 * warp;
        if (p0 < A.parts) S.tot[p0] += s_lo;
        if (p0 + 1 < A.parts) S.tot[p0 + 1] += s_hi;
      }
      __syncthreads();
    }
  }
  for (int p = tid; p < A.parts; p += kT) A.cnt[(size_t)p * G + c] = S.tot[p];
  if (!grid_wait(A.barrier, (unsigned)G, A.skip_cta, A.status)) return;
  partition_bases(A.cnt, G, A.parts, S.base, A.d_offsets, nullptr);
  // place: per tile, thread t owns entries [kPPer t, kPPer (t + 1)) (input order)
  for (long long t0 = lo; t0 < hi; t0 += kPTile) {
    const int tl = (int)min((long long)kPTile, hi - t0);
    if (!resident) part_load(A, S, t0, tl, true);
    const int i0 = tid * kPPer, i1 = min(i0 + kPPer, tl);
    if (tid == 0) S.run = 0;
    for (int s0 = 0; s0 < A.parts; s0 += kSlab) {
      counters_clear(S.cw);
      for (int i = i0; i < i1; ++i) {
        const int q = (int)S.part[i] - s0;
        if ((unsigned)q < (unsigned)kSlab) counter_add(S.cw, q);
      }
      __syncthreads();
      counters_scan(S.cw, s0, A.parts, S.wtot, S.wofs, &S.run);
      for (int i = i0; i < i1; ++i) {
        const int p = S.part[i];
        const int q = p - s0;
        if ((unsigned)q >= (unsigned)kSlab) continue;
        const int slot = S.wofs[p] + counter_take(S.cw, q);
        S.okey[slot] = S.key[i];
        if (A.val) S.oval[slot] = S.val[i];
        S.opart[slot] = (uint8_t)p;
      }
      __syncthreads();
    }
    for (int s = tid; s < tl; s += kT) {
      const int p = S.opart[s];
      const long long dst = S.base[p] + (s - S.wofs[p]);
      if (dst >= 0 && dst < A.nnz) {
        A.out_idx[dst] = S.okey[s];
        if (A.val) A.out_val[dst] = S.oval[s];
      } else {
        flag(A.status, ZR_ERR_INTERNAL);
      }
    }
    __syncthreads();
    for (int p = tid; p < A.parts; p += kT) S.base[p] += S.wtot[p];
    __syncthreads();
  }
}

// ---------------------------------------------------------------- host side
// Per-device grid sizes of the two cooperative kernels (CTAs that fit at
// once), filled once per device under a lock.
struct CoopInfo {
  std::atomic<int> ready{0};
  int part_grid = 0;
};

CoopInfo* coop_info() {
  static CoopInfo info[64];
  static std::mutex lock;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  CoopInfo& d = info[dev];
  if (d.ready.load(std::memory_order_acquire)) return &d;
  std::lock_guard<std::mutex> guard(lock);
  if (!d.ready.load(std::memory_order_relaxed)) {
    int coop = 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop)
      return nullptr;
    if (cudaFuncSetAttribute((const void*)partition_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kPartSmem) != cudaSuccess)
      return nullptr;
    int bp = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bp, partition_kernel, kT, kPartSmem) !=
            cudaSuccess ||
        bp < 1)
      return nullptr;
    d.part_grid = min(sm_count() * bp, kMaxCtas);
    d.ready.store(1, std::memory_order_release);
  }
  return &d;
}

zr_status launch_coop(const void* fn, int grid, int threads, size_t smem, void* arg,
                      cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {arg};
  if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) return ZR_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
}

size_t coo_workspace(int parts) {
  return (size_t)kHeader + (size_t)parts * kMaxCtas * sizeof(int32_t);
}

}  // namespace

size_t partition_workspace_bytes(int64_t nnz, int n_parts) {
  (void)nnz;
  return coo_workspace(n_parts);
}

namespace {
zr_status partition_run(const int32_t* idx, const float* val, int64_t nnz, int n_parts,
                        uint64_t part_seed, int32_t* out_idx, float* out_val, int64_t* d_offsets,
                        void* ws, cudaStream_t stream) {
  if (nnz == 0) {
    unsigned char* w = static_cast<unsigned char*>(ws);
    if (cudaMemsetAsync(w, 0, kHeader, stream) != cudaSuccess) return ZR_ERR_CUDA;
    if (cudaMemsetAsync(d_offsets, 0, (size_t)(n_parts + 1) * 8, stream) != cudaSuccess)
      return ZR_ERR_CUDA;
    return ZR_OK;
  }
  CoopInfo* info = coop_info();
  if (!info) return ZR_ERR_CUDA;
  PartArgs A;
  A.idx = idx;
  A.val = val;
  A.nnz = nnz;
  A.parts = n_parts;
  A.h = make_h0(part_seed, (uint32_t)n_parts);
  A.out_idx = out_idx;
  A.out_val = out_val;
  A.d_offsets = reinterpret_cast<long long*>(d_offsets);
  unsigned char* w = static_cast<unsigned char*>(ws);
  A.status = reinterpret_cast<int32_t*>(w);
  A.barrier = reinterpret_cast<unsigned*>(w + 4);
  A.cnt = reinterpret_cast<int32_t*>(w + kHeader);
  A.skip_cta = g_barrier_skip.load(std::memory_order_relaxed);
  // no more CTAs than 4-entry groups, so no CTA's slice is empty by rounding
  int grid = info->part_grid;
  const long long groups = (nnz + 3) / 4;
  if (grid > groups) grid = (int)groups;
  if (cudaMemsetAsync(w, 0, kHeader, stream) != cudaSuccess) return ZR_ERR_CUDA;
  return launch_coop((const void*)partition_kernel, grid, kT, kPartSmem, &A, stream);
}
}  // namespace

zr_status partition_launch(const int32_t* idx, const float* val, int64_t nnz, int n_parts,
                           uint64_t part_seed, int32_t* out_idx, float* out_val,
                           int64_t* d_offsets, void* ws, cudaStream_t stream) {
  return partition_run(idx, val, nnz, n_parts, part_seed, out_idx, out_val, d_offsets, ws, stream);
}

zr_status index_sets_launch(int64_t m, int n_parts, uint64_t part_seed, int32_t* out_sets,
                            int64_t* d_offsets, void* ws, cudaStream_t stream) {
  return partition_run(nullptr, nullptr, m, n_parts, part_seed, out_sets, nullptr, d_offsets, ws,
                       stream);
}

}  // namespace zr

extern "C" void zr_test_barrier_skip(int32_t cta) {
  zr::g_barrier_skip.store(cta, std::memory_order_relaxed);
}
