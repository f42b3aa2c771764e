// Sparse (COO) gradient aggregation and the h0 partition.
//
// What is computed (Zen page, section 2.1 "COO", Problem 1, section 3.2
// Technique #3 and Algorithm 1's first-level hash): the union of N sorted
// index lists, each union index carrying the rank-ordered sum of the values
// that hold it, split into n_parts partitions by the consistent hash h0 and
// written partition-major, ascending index inside a partition.
//
// GB300 design.  The key range [0, M) is cut into bins of W = 8192 keys.
// Every bin is an independent unit of work small enough for one CTA's shared
// memory, which makes the merge of N lists a dense-window problem instead of
// a comparison merge:
//   1. bin_starts:  one streaming pass over every list finds, for each rank
//      and bin, where the bin's entries start (sorted lists: a bin boundary is
//      where consecutive keys fall in different bins).  It also checks that
//      the lists are strictly ascending and in range.
//   2. bin_count:   per bin, OR every rank's keys into a W-bit presence map in
//      shared memory, hash the union's members and count them per partition.
//   3. scan:        one CTA turns the (bin, partition) counts into output
//      positions: partition-major, bins in key order inside a partition.
//   4. bin_write:   per bin, fold the values into a W-float window in shared
//      memory rank by rank (ascending rank order, a barrier between ranks: the
//      exact left fold of the oracle, since the window starts at -0.0 and
//      -0.0 + x == x for every x), then emit the members in key order with a
//      warp-level stable multi-split on the partition id.
// Bins are handed to CTAs round-robin, so the skewed hot region of an
// embedding gradient spreads over the whole grid.
//
// Every index taken from the inputs is range-checked before it addresses
// shared memory, and segment bounds read from the workspace are clamped to
// the list lengths, so malformed input can only produce wrong output and a
// status word, never an out-of-bounds access.

#include <cuda_runtime.h>
#include <stdint.h>

#include "zr.h"
#include "zr_device.cuh"
#include "zr_internal.h"

namespace zr {
namespace {

constexpr int kLogW = 13;
constexpr int kW = 1 << kLogW;          // keys per bin
constexpr int kWords = kW / 32;         // presence words per bin
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kWordsPerWarp = kWords / kWarps;
constexpr int kScanThreads = 512;
constexpr int kScanGroup = 8;           // partitions scanned together
constexpr int kPartTile = 4096;         // zr_partition: entries per tile
constexpr int kPartThreads = 512;

struct Lists {
  const int32_t* idx[ZR_MAX_RANKS];
  const float* val[ZR_MAX_RANKS];
  int64_t nnz[ZR_MAX_RANKS];
};

__device__ __forceinline__ void flag(int32_t* status, int code) {
  atomicCAS(status, 0, code);
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct SparseLayout {
  size_t status, starts, counts, pos, total;
};

SparseLayout sparse_layout(int n, int64_t bins, int parts) {
  SparseLayout L;
  L.status = 0;
  L.starts = 256;
  L.counts = L.starts + align256((size_t)n * (size_t)(bins + 1) * sizeof(int32_t));
  L.pos = L.counts + align256((size_t)bins * parts * sizeof(int32_t));
  L.total = L.pos + align256((size_t)bins * parts * sizeof(int64_t));
  return L;
}

// ---------------------------------------------------------------- 1. starts
// Grid: x over list positions (one thread per position plus the end), y = rank.
__global__ void bin_starts_kernel(const __grid_constant__ Lists lists, int64_t dense_size,
                                  int64_t bins, int32_t* starts, int32_t* status) {
  const int r = blockIdx.y;
  const int64_t nnz = lists.nnz[r];
  const int32_t* idx = lists.idx[r];
  int32_t* row = starts + (size_t)r * (bins + 1);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i <= nnz;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t b_here;
    if (i < nnz) {
      const int64_t key = idx[i];
      bool ok = key >= 0 && key < dense_size;
      if (i > 0 && key <= (int64_t)idx[i - 1]) ok = false;
      if (!ok) flag(status, ZR_ERR_INPUT_UNSORTED);
      b_here = key < 0 ? -1 : min(key >> kLogW, bins);
    } else {
      b_here = bins;
    }
    int64_t b_prev = -1;
    if (i > 0) {
      const int64_t pk = idx[i - 1];
      b_prev = pk < 0 ? -1 : min(pk >> kLogW, bins);
    }
    for (int64_t b = b_prev + 1; b <= b_here; ++b) row[b] = (int32_t)i;
  }
}

__device__ __forceinline__ void segment(const int32_t* starts, int64_t bins, int r, int64_t b,
                                        int64_t nnz, int64_t& s, int64_t& e) {
  const int32_t* row = starts + (size_t)r * (bins + 1);
  s = min(max((int64_t)row[b], (int64_t)0), nnz);
  e = min(max((int64_t)row[b + 1], s), nnz);
}

// ---------------------------------------------------------------- 2. count
__global__ void __launch_bounds__(kThreads)
bin_count_kernel(const __grid_constant__ Lists lists, int n, int64_t bins, const int32_t* starts,
                 H0 h, int parts, int32_t* counts, int32_t* status) {
  __shared__ uint32_t bits[kWords];
  __shared__ int32_t cnt[ZR_MAX_PARTS];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t b = blockIdx.x; b < bins; b += gridDim.x) {
    const int64_t base = b << kLogW;
    for (int t = threadIdx.x; t < kWords; t += kThreads) bits[t] = 0;
    for (int t = threadIdx.x; t < parts; t += kThreads) cnt[t] = 0;
    __syncthreads();
    for (int r = 0; r < n; ++r) {
      int64_t s, e;
      segment(starts, bins, r, b, lists.nnz[r], s, e);
      const int32_t* idx = lists.idx[r];
      for (int64_t i = s + threadIdx.x; i < e; i += kThreads) {
        const int64_t slot = (int64_t)idx[i] - base;
        if (slot >= 0 && slot < kW) atomicOr(&bits[slot >> 5], 1u << (slot & 31));
        else flag(status, ZR_ERR_INPUT_UNSORTED);
      }
    }
    __syncthreads();
    for (int j = 0; j < kWordsPerWarp; ++j) {
      const int word = warp * kWordsPerWarp + j;
      const bool present = (bits[word] >> lane) & 1u;
      const uint32_t key = (uint32_t)(base + word * 32 + lane);
      const int p = present ? (parts > 1 ? (int)h(key) : 0) : parts;
      const unsigned peers = __match_any_sync(0xffffffffu, p);
      if (present && (peers & lanemask_lt()) == 0) atomicAdd(&cnt[p], __popc(peers));
    }
    __syncthreads();
    for (int t = threadIdx.x; t < parts; t += kThreads) counts[b * parts + t] = cnt[t];
    __syncthreads();
  }
}

// ---------------------------------------------------------------- 3. scan
// One CTA.  pos[b][p] = offsets[p] + sum_{b' < b} counts[b'][p], where
// offsets[p] = sum_{p' < p} total[p'].  Writes offsets[0..parts] and the total
// when the caller asked for them.
__global__ void __launch_bounds__(kScanThreads)
scan_kernel(const int32_t* counts, int64_t bins, int parts, int64_t* pos,
            int64_t* d_offsets, int write_offsets, int64_t* d_total) {
  __shared__ long long tot[ZR_MAX_PARTS + 1];
  __shared__ long long part[kScanGroup][kScanThreads];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t per = (bins + kScanThreads - 1) / kScanThreads;
  const int64_t b0 = min((int64_t)t * per, bins), b1 = min(b0 + per, bins);

  for (int p = t; p <= parts; p += kScanThreads) tot[p] = 0;
  __syncthreads();
  for (int p = 0; p < parts; ++p) {
    long long s = 0;
    for (int64_t b = b0; b < b1; ++b) s += counts[b * parts + p];
    for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
    if (lane == 0 && s) atomicAdd((unsigned long long*)&tot[p], (unsigned long long)s);
  }
  __syncthreads();
  if (t == 0) {
    long long run = 0;
    for (int p = 0; p < parts; ++p) {
      long long c = tot[p];
      tot[p] = run;
      run += c;
    }
    tot[parts] = run;
    if (d_total) *d_total = run;
  }
  __syncthreads();
  if (write_offsets)
    for (int p = t; p <= parts; p += kScanThreads) d_offsets[p] = tot[p];

  for (int g0 = 0; g0 < parts; g0 += kScanGroup) {
    const int gn = min(kScanGroup, parts - g0);
    for (int g = 0; g < gn; ++g) {
      long long s = 0;
      for (int64_t b = b0; b < b1; ++b) s += counts[b * parts + g0 + g];
      part[g][t] = s;
    }
    __syncthreads();
    // Warp g: exclusive scan of part[g][0 .. kScanThreads).
    if (warp < gn) {
      constexpr int kPerLane = kScanThreads / 32;
      long long loc[kPerLane];
      long long sum = 0;
#pragma unroll
      for (int q = 0; q < kPerLane; ++q) {
        loc[q] = part[warp][lane * kPerLane + q];
        sum += loc[q];
      }
      long long incl = sum;
      for (int o = 1; o < 32; o <<= 1) {
        long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      long long run = incl - sum;
#pragma unroll
      for (int q = 0; q < kPerLane; ++q) {
        part[warp][lane * kPerLane + q] = run;
        run += loc[q];
      }
    }
    __syncthreads();
    for (int g = 0; g < gn; ++g) {
      const int p = g0 + g;
      long long run = tot[p] + part[g][t];
      for (int64_t b = b0; b < b1; ++b) {
        pos[b * parts + p] = run;
        run += counts[b * parts + p];
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- 4. write
__global__ void __launch_bounds__(kThreads)
bin_write_kernel(const __grid_constant__ Lists lists, int n, int64_t bins, const int32_t* starts,
                 H0 h, int parts, int average, const int64_t* pos, int32_t* out_idx,
                 float* out_val, int64_t out_cap, int32_t* status) {
  extern __shared__ __align__(16) unsigned char smem[];
  float* acc = reinterpret_cast<float*>(smem);                                  // kW
  uint32_t* bits = reinterpret_cast<uint32_t*>(smem + kW * sizeof(float));     // kWords
  long long* wbase = reinterpret_cast<long long*>(smem + kW * sizeof(float) + kWords * 4);  // kWarps*parts
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float fn = (float)n;

  for (int64_t b = blockIdx.x; b < bins; b += gridDim.x) {
    const int64_t base = b << kLogW;
    for (int t = threadIdx.x; t < kW; t += kThreads) acc[t] = -0.0f;
    for (int t = threadIdx.x; t < kWords; t += kThreads) bits[t] = 0;
    for (int t = threadIdx.x; t < kWarps * parts; t += kThreads) wbase[t] = 0;
    __syncthreads();
    // Rank-ordered fold: one rank at a time, a barrier in between.
    for (int r = 0; r < n; ++r) {
      int64_t s, e;
      segment(starts, bins, r, b, lists.nnz[r], s, e);
      if (s == e) continue;  // block-uniform
      const int32_t* idx = lists.idx[r];
      const float* val = lists.val[r];
      for (int64_t i = s + threadIdx.x; i < e; i += kThreads) {
        const int64_t slot = (int64_t)idx[i] - base;
        if (slot >= 0 && slot < kW) {
          acc[slot] = __fadd_rn(acc[slot], val[i]);
          atomicOr(&bits[slot >> 5], 1u << (slot & 31));
        } else {
          flag(status, ZR_ERR_INPUT_UNSORTED);
        }
      }
      __syncthreads();
    }
    // Pass 1: per-warp counts per partition over the warp's words, in order.
    for (int j = 0; j < kWordsPerWarp; ++j) {
      const int word = warp * kWordsPerWarp + j;
      const bool present = (bits[word] >> lane) & 1u;
      const uint32_t key = (uint32_t)(base + word * 32 + lane);
      const int p = present ? (parts > 1 ? (int)h(key) : 0) : parts;
      const unsigned peers = __match_any_sync(0xffffffffu, p);
      if (present && (peers & lanemask_lt()) == 0) wbase[warp * parts + p] += __popc(peers);
      __syncwarp();
    }
    __syncthreads();
    // Exclusive scan over warps, per partition, from the bin's base position.
    for (int p = threadIdx.x; p < parts; p += kThreads) {
      long long run = pos[b * parts + p];
      for (int w = 0; w < kWarps; ++w) {
        long long c = wbase[w * parts + p];
        wbase[w * parts + p] = run;
        run += c;
      }
    }
    __syncthreads();
    // Pass 2: emit members in key order; equal partitions keep lane order.
    for (int j = 0; j < kWordsPerWarp; ++j) {
      const int word = warp * kWordsPerWarp + j;
      const bool present = (bits[word] >> lane) & 1u;
      const int slot = word * 32 + lane;
      const uint32_t key = (uint32_t)(base + slot);
      const int p = present ? (parts > 1 ? (int)h(key) : 0) : parts;
      const unsigned peers = __match_any_sync(0xffffffffu, p);
      if (present) {
        const long long dst = wbase[warp * parts + p] + __popc(peers & lanemask_lt());
        float v = acc[slot];
        if (average) v = __fdiv_rn(v, fn);
        if (dst >= 0 && dst < out_cap) {  // only malformed input can fail this
          out_idx[dst] = (int32_t)key;
          out_val[dst] = v;
        } else {
          flag(status, ZR_ERR_INPUT_UNSORTED);
        }
      }
      __syncwarp();
      if (present && (peers & lanemask_lt()) == 0) wbase[warp * parts + p] += __popc(peers);
      __syncwarp();
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- partition
__global__ void __launch_bounds__(kPartThreads)
part_count_kernel(const int32_t* idx, int64_t nnz, int64_t tiles, H0 h, int parts,
                  int32_t* counts) {
  __shared__ int32_t cnt[ZR_MAX_PARTS];
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    for (int q = threadIdx.x; q < parts; q += kPartThreads) cnt[q] = 0;
    __syncthreads();
    const int64_t lo = t * kPartTile, hi = min(lo + kPartTile, nnz);
    for (int64_t i = lo + threadIdx.x; i < lo + kPartTile; i += kPartThreads) {
      const bool live = i < hi;
      const int p = live ? (int)h((uint32_t)idx[i]) : parts;
      const unsigned peers = __match_any_sync(0xffffffffu, p);
      if (live && (peers & lanemask_lt()) == 0) atomicAdd(&cnt[p], __popc(peers));
    }
    __syncthreads();
    for (int q = threadIdx.x; q < parts; q += kPartThreads) counts[t * parts + q] = cnt[q];
    __syncthreads();
  }
}

// Each warp owns kPartTile / warps consecutive entries of the tile and walks
// them 32 at a time, so the entries of one partition leave in input order.
__global__ void __launch_bounds__(kPartThreads)
part_write_kernel(const int32_t* idx, const float* val, int64_t nnz, int64_t tiles, H0 h,
                  int parts, const int64_t* pos, int32_t* out_idx, float* out_val) {
  extern __shared__ __align__(16) unsigned char smem[];
  long long* wbase = reinterpret_cast<long long*>(smem);  // warps * parts
  constexpr int kPW = kPartThreads / 32;
  constexpr int kPerWarp = kPartTile / kPW;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    for (int q = threadIdx.x; q < kPW * parts; q += kPartThreads) wbase[q] = 0;
    __syncthreads();
    const int64_t lo = t * kPartTile + (int64_t)warp * kPerWarp;
    const int64_t hi = min(t * kPartTile + kPartTile, nnz);
    for (int j = 0; j < kPerWarp; j += 32) {
      const int64_t i = lo + j + lane;
      const bool live = i < hi;
      const int p = live ? (int)h((uint32_t)idx[i]) : parts;
      const unsigned peers = __match_any_sync(0xffffffffu, p);
      if (live && (peers & lanemask_lt()) == 0) wbase[warp * parts + p] += __popc(peers);
      __syncwarp();
    }
    __syncthreads();
    for (int q = threadIdx.x; q < parts; q += kPartThreads) {
      long long run = pos[t * parts + q];
      for (int w = 0; w < kPW; ++w) {
        long long c = wbase[w * parts + q];
        wbase[w * parts + q] = run;
        run += c;
      }
    }
    __syncthreads();
    for (int j = 0; j < kPerWarp; j += 32) {
      const int64_t i = lo + j + lane;
      const bool live = i < hi;
      const int32_t key = live ? idx[i] : 0;
      const int p = live ? (int)h((uint32_t)key) : parts;
      const unsigned peers = __match_any_sync(0xffffffffu, p);
      if (live) {
        const long long dst = wbase[warp * parts + p] + __popc(peers & lanemask_lt());
        out_idx[dst] = key;
        out_val[dst] = val[i];
      }
      __syncwarp();
      if (live && (peers & lanemask_lt()) == 0) wbase[warp * parts + p] += __popc(peers);
      __syncwarp();
    }
    __syncthreads();
  }
}

size_t write_smem_bytes(int parts) {
  return (size_t)kW * sizeof(float) + (size_t)kWords * 4 + (size_t)kWarps * parts * sizeof(long long);
}

bool ensure_write_smem() {
  static int done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (done[dev]) return true;
  if (cudaFuncSetAttribute(bin_write_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)write_smem_bytes(ZR_MAX_PARTS)) != cudaSuccess)
    return false;
  done[dev] = 1;
  return true;
}

int64_t clamp_grid(int64_t units, int per_sm) {
  int64_t g = (int64_t)sm_count() * per_sm;
  if (g > units) g = units;
  return g < 1 ? 1 : g;
}

}  // namespace

size_t sparse_workspace_bytes(int n, int64_t dense_size, int n_parts) {
  const int64_t bins = (dense_size + kW - 1) / kW;
  const int parts = n_parts > 0 ? n_parts : 1;
  return sparse_layout(n, bins, parts).total;
}

zr_status sparse_launch(const int32_t* const* idx, const float* const* val, const int64_t* nnz,
                        int n, int64_t dense_size, int n_parts, uint64_t part_seed, int average,
                        int32_t* out_idx, float* out_val, int64_t out_cap, int64_t* d_out_nnz,
                        int64_t* d_offsets, void* ws, cudaStream_t stream) {
  const int64_t bins = (dense_size + kW - 1) / kW;
  const int parts = n_parts > 0 ? n_parts : 1;
  const SparseLayout L = sparse_layout(n, bins, parts);
  unsigned char* w = static_cast<unsigned char*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w + L.status);
  int32_t* starts = reinterpret_cast<int32_t*>(w + L.starts);
  int32_t* counts = reinterpret_cast<int32_t*>(w + L.counts);
  int64_t* pos = reinterpret_cast<int64_t*>(w + L.pos);

  Lists lists;
  int64_t max_nnz = 0;
  for (int r = 0; r < ZR_MAX_RANKS; ++r) {
    const bool live = r < n && nnz[r] > 0;
    lists.idx[r] = live ? idx[r] : nullptr;
    lists.val[r] = live ? val[r] : nullptr;
    lists.nnz[r] = r < n ? nnz[r] : 0;
    if (r < n && nnz[r] > max_nnz) max_nnz = nnz[r];
  }
  H0 h = make_h0(part_seed, (uint32_t)parts);
  if (!ensure_write_smem()) return ZR_ERR_CUDA;
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), stream) != cudaSuccess) return ZR_ERR_CUDA;

  {
    int64_t gx = (max_nnz + 1 + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (gx > cap) gx = cap;
    if (gx < 1) gx = 1;
    bin_starts_kernel<<<dim3((unsigned)gx, (unsigned)n), 256, 0, stream>>>(lists, dense_size, bins,
                                                                           starts, status);
  }
  bin_count_kernel<<<(unsigned)clamp_grid(bins, 4), kThreads, 0, stream>>>(
      lists, n, bins, starts, h, parts, counts, status);
  scan_kernel<<<1, kScanThreads, 0, stream>>>(counts, bins, parts, pos, d_offsets,
                                               (n_parts > 0 && d_offsets) ? 1 : 0, d_out_nnz);
  bin_write_kernel<<<(unsigned)clamp_grid(bins, 4), kThreads, write_smem_bytes(parts), stream>>>(
      lists, n, bins, starts, h, parts, average, pos, out_idx, out_val, out_cap, status);
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
}

size_t partition_workspace_bytes(int64_t nnz, int n_parts) {
  const int64_t tiles = (nnz + kPartTile - 1) / kPartTile;
  return 256 + align256((size_t)tiles * n_parts * sizeof(int32_t)) +
         align256((size_t)tiles * n_parts * sizeof(int64_t));
}

zr_status partition_launch(const int32_t* idx, const float* val, int64_t nnz, int n_parts,
                           uint64_t part_seed, int32_t* out_idx, float* out_val,
                           int64_t* d_offsets, void* ws, cudaStream_t stream) {
  const int64_t tiles = (nnz + kPartTile - 1) / kPartTile;
  unsigned char* w = static_cast<unsigned char*>(ws);
  int32_t* counts = reinterpret_cast<int32_t*>(w + 256);
  int64_t* pos = reinterpret_cast<int64_t*>(w + 256 + align256((size_t)tiles * n_parts * sizeof(int32_t)));
  H0 h = make_h0(part_seed, (uint32_t)n_parts);
  if (tiles > 0)
    part_count_kernel<<<(unsigned)clamp_grid(tiles, 4), kPartThreads, 0, stream>>>(
        idx, nnz, tiles, h, n_parts, counts);
  scan_kernel<<<1, kScanThreads, 0, stream>>>(counts, tiles, n_parts, pos, d_offsets, 1, nullptr);
  if (tiles > 0) {
    const size_t smem = (size_t)(kPartThreads / 32) * n_parts * sizeof(long long);
    part_write_kernel<<<(unsigned)clamp_grid(tiles, 4), kPartThreads, smem, stream>>>(
        idx, val, nnz, tiles, h, n_parts, pos, out_idx, out_val);
  }
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
}

}  // namespace zr
