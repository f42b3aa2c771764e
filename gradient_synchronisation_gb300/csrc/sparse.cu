// Sparse (COO) gradient aggregation and the h0 partition.
//
// What is computed (Zen page, section 2.1 "COO", Problem 1, section 3.2
// Technique #3 and Algorithm 1's first-level hash): the union of N sorted
// index lists, each union index carrying the rank-ordered sum of the values
// that hold it, split into n_parts partitions by the consistent hash h0 and
// written partition-major, ascending index inside a partition.
//
// GB300 design.  The key range [0, M) is cut into bins of W keys (W = 1024,
// wider only when the workspace would otherwise grow too large).  A bin is
// the work of one warp, so nothing inside a bin waits on a block barrier,
// and tens of warps per SM hide each other's memory latency:
//   1. starts:  one streaming pass over every list (16-byte loads) writes,
//      for every rank and bin, where the bin's entries start, and checks
//      that each list is strictly ascending and in range.
//   2. count:   per bin, a warp ORs the keys of every rank into the bin's
//      W-bit union bitmap (warp-private shared memory), hashes each member
//      and counts members per partition.
//   3. scan:    one CTA per partition turns the per-bin counts into each
//      bin's first output position in that partition.
//   4. write:   per bin, a warp walks the bin rank by rank in chunks of up
//      to 32 consecutive entries of one rank (the loads of 12 chunks in
//      flight; a warp-uniform cursor gives each chunk's rank), or, where
//      bins hold few entries, flattened in groups of 32 across rank
//      boundaries applied in ascending runs, and folds them into a
//      warp-private W-float window in ascending rank order, which is the
//      left fold of the holders' values.  Then the members are placed into
//      their partitions' runs: through per-lane partition counters where
//      bins hold few entries, partition by partition from per-partition
//      member bitmaps where they hold many, and by a counting sort above 32
//      partitions.  Each member's output position is its partition's offset
//      plus the bin's prefix from step 3 plus its rank inside the bin, so
//      members leave in ascending key order inside each partition.
//
// Every index taken from the inputs is range-checked before it addresses
// shared memory, bounds read from the workspace are clamped to the list
// lengths, and every output run (or position) is checked against the output
// capacity before it is written, so malformed input can only produce wrong
// output and a status word, never an out-of-bounds access.

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "zr.h"
#include "zr_device.cuh"
#include "zr_internal.h"

namespace zr {
namespace {

constexpr int kBinWarps = 8;             // warps per CTA in the count and write kernels
constexpr int kBinThreads = kBinWarps * 32;
constexpr int kStartsUnroll = 4;         // starts kernel: groups of 4 keys per thread per step
constexpr int kBatch = 4;                // flattened walk: groups of 32 entries per load batch (2-12 measured)
constexpr int kWriteWarps = 4;           // warps per CTA in the write kernel
constexpr int kWriteThreads = kWriteWarps * 32;

struct Lists {
  const int32_t* idx[ZR_MAX_RANKS];
  const float* val[ZR_MAX_RANKS];
  int64_t nnz[ZR_MAX_RANKS];
};

__device__ __forceinline__ void flag(int32_t* status, int code) { atomicCAS(status, 0, code); }

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// ------------------------------------------------------------ layout
// Bins are W = 2^log_w keys: 1024, widened (up to 4096) only when the
// per-(bin, partition) tables would exceed 2^24 entries.
constexpr int kChunkLog = 11;            // bins per scan chunk = 2048
constexpr int kChunkBins = 1 << kChunkLog;
constexpr int kScanThreads = kChunkBins / 2;

constexpr int64_t kWidenBelowPerBin = 128;  // densification: entries per 1024-key bin below which bins widen

struct Geometry {
  int log_w;
  int64_t bins;
};

Geometry geometry(int n, int64_t dense_size, int parts, int64_t total_nnz) {
  Geometry g;
  g.log_w = 10;
  for (;;) {
    g.bins = (dense_size + (1ll << g.log_w) - 1) >> g.log_w;
    if (g.log_w >= 12 || g.bins * (int64_t)(parts + n) <= (1ll << 24)) break;
    ++g.log_w;
  }
  (void)total_nnz;
  return g;
}

// Densification of lists with few entries per 1024-key bin (known at
// launch) takes 2048-key bins: half the bins for the same entries (C4:
// 0.038 -> 0.036 ms; the union's writer measured no faster, its occupancy
// falls with the wider window).  The workspace is sized for the narrowest
// bins, so it holds the wider ones.
Geometry densify_geometry(int n, int64_t dense_size, int64_t total_nnz) {
  Geometry g = geometry(n, dense_size, 0, total_nnz);
  if (g.log_w == 10 && total_nnz >= 0 && total_nnz < kWidenBelowPerBin * g.bins) {
    g.log_w = 11;
    g.bins = (dense_size + (1ll << g.log_w) - 1) >> g.log_w;
  }
  return g;
}

// Workspace: [status] (cleared by a memset), then the bin starts, the
// per-bin counts, the per-chunk totals, the per-bin exclusive prefixes and
// the partition totals.
struct SparseLayout {
  size_t starts, cnt, ctot, excl, tot, total;
};

SparseLayout sparse_layout(int n, int64_t bins, int parts) {
  SparseLayout L;
  const int64_t chunks = (bins + kChunkBins - 1) >> kChunkLog;
  L.starts = 256;
  L.cnt = L.starts + align256((size_t)n * (size_t)(bins + 1) * 4);
  L.ctot = L.cnt + align256((size_t)parts * bins * 4);
  L.excl = L.ctot + align256((size_t)parts * chunks * 8);
  L.tot = L.excl + align256((size_t)parts * bins * 8);
  L.total = L.tot + align256((size_t)parts * 8);
  return L;
}


// ------------------------------------------------------------ 1. starts
// Grid: x over groups of 4 positions, y = rank.  starts[r][b] = first
// position whose key is in bin >= b (nnz if none); every list is checked
// strictly ascending and in range.  32-bit index arithmetic throughout
// (positions, keys and bins all fit).
//
// The groups of 4 real keys are grid-strided, kStartsUnroll per thread and
// step (their loads issued together): per key a range and order check, its
// bin (clamped, so out-of-range keys cannot address past the row) and, at a
// bin change, the row entries of the bins it starts (more than one only
// across empty bins).  CTA 0 then takes the ragged tail (the last nnz mod 4
// keys) on one thread and the end marker, position nnz, which starts every
// bin after the last key's, on all of its threads.
__device__ __forceinline__ int clamped_bin(int key, int log_w, int bins) {
  return min(max(key >> log_w, -1), bins);  // a negative key gives -1
}

__global__ void __launch_bounds__(256)
bin_starts_kernel(const __grid_constant__ Lists lists, int dense_size, int log_w, int bins,
                  int32_t* starts, int32_t* status) {
  __shared__ int s_last_bin;
  const int r = blockIdx.y;
  const int nnz = (int)lists.nnz[r];
  const int32_t* idx = lists.idx[r];
  int32_t* row = starts + (size_t)r * (bins + 1);
  const bool vec = (reinterpret_cast<uintptr_t>(idx) & 15) == 0;
  const int full = nnz >> 2;  // groups of 4 real keys
  constexpr int kU = kStartsUnroll;
  const int stride = gridDim.x * blockDim.x;
  bool bad = false;
  for (int q0 = blockIdx.x * blockDim.x + threadIdx.x; q0 < full; q0 += kU * stride) {
    int4 kv[kU];
    int prev[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int q = q0 + u * stride;
      kv[u] = make_int4(0, 0, 0, 0);
      prev[u] = -1;
      if (q < full) {
        if (vec) {
          kv[u] = __ldg(reinterpret_cast<const int4*>(idx) + q);
        } else {
          kv[u].x = __ldg(idx + 4 * q);
          kv[u].y = __ldg(idx + 4 * q + 1);
          kv[u].z = __ldg(idx + 4 * q + 2);
          kv[u].w = __ldg(idx + 4 * q + 3);
        }
        if (q > 0) prev[u] = __ldg(idx + 4 * q - 1);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int q = q0 + u * stride;
      if (q >= full) continue;
      const int key[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
      int p = prev[u];
      int bp = p < 0 ? -1 : clamped_bin(p, log_w, bins);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k = key[e];
        // p >= k also rejects a negative first key (p is -1 there)
        bad |= (unsigned)k >= (unsigned)dense_size || k <= p;
        const int bk = clamped_bin(k, log_w, bins);
        if (bk > bp) {
          row[bp + 1] = 4 * q + e;
          for (int bb = bp + 2; bb <= bk; ++bb) row[bb] = 4 * q + e;  // empty bins
          bp = bk;
        }
        p = k;
      }
    }
  }
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0) {
      int p = full > 0 ? __ldg(idx + 4 * full - 1) : -1;
      int bp = p < 0 ? -1 : clamped_bin(p, log_w, bins);
      for (int i = 4 * full; i < nnz; ++i) {
        const int k = __ldg(idx + i);
        bad |= (unsigned)k >= (unsigned)dense_size || k <= p;
        const int bk = clamped_bin(k, log_w, bins);
        for (int bb = bp + 1; bb <= bk; ++bb) row[bb] = i;
        bp = max(bp, bk);
        p = k;
      }
      s_last_bin = bp;
    }
    __syncthreads();
    // the end marker: position nnz starts every bin after the last key's
    for (int bb = s_last_bin + 1 + threadIdx.x; bb <= bins; bb += blockDim.x) row[bb] = nnz;
  }
  if (bad) flag(status, ZR_ERR_INPUT_UNSORTED);
}

// ------------------------------------------------------------ bin walk
// A warp's view of one bin: lane r (and r + 32) holds rank r's first list
// position in the bin (lo) and its entry count (len), clamped to the list.
struct BinRows {
  int lo[2], len[2];
};

// A bin's raw start rows for ranks lane and lane + 32, loaded ahead of use
// so that the next bin's loads are in flight while the current bin works.
struct BinFetch {
  int lo[2], hi[2];
};

__device__ __forceinline__ BinFetch bin_fetch(const int32_t* starts, int n, int bins, int b) {
  const int lane = threadIdx.x & 31;
  BinFetch f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = lane + 32 * h;
    f.lo[h] = f.hi[h] = 0;
    if (r < n) {
      const int32_t* row = starts + (size_t)r * (bins + 1) + b;
      f.lo[h] = __ldcg(row);
      f.hi[h] = __ldcg(row + 1);
    }
  }
  return f;
}

__device__ __forceinline__ BinRows bin_rows(const Lists& lists, int n, const BinFetch& f) {
  const int lane = threadIdx.x & 31;
  BinRows R;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = lane + 32 * h;
    int lo = 0, len = 0;
    if (r < n) {
      const int nnz = (int)lists.nnz[r];
      lo = min(max(f.lo[h], 0), nnz);
      len = min(max(f.hi[h], lo), nnz) - lo;
    }
    R.lo[h] = lo;
    R.len[h] = len;
  }
  return R;
}

// Rank r's value (r < 64, the same on every lane) from the lane holding it.
__device__ __forceinline__ int rank_get(const int (&v)[2], int r) {
  return __shfl_sync(0xffffffffu, (r & 32) ? v[1] : v[0], r & 31);
}

// Walks the bin rank by rank, lowest rank first, in chunks of up to 32
// consecutive entries of one rank: lane l takes entry c + l of the rank's
// chunk at entry offset c.  The loads of kChunks chunks are issued together
// (load(t, rank, pos) fills slot t), then apply(t, ok) runs for the chunks
// in order, ok saying whether the lane holds an entry.  A list is strictly
// ascending, so the keys of one chunk are distinct and a chunk is applied
// at once; chunks go in rank order, so a key held by several ranks meets
// the lowest rank first.  The cursor (rank, its first position and count,
// the next chunk's offset) is the same on every lane, so the walk's
// branches and the shuffles that fetch the next rank's row are uniform.
template <int kChunks, typename Load, typename Apply>
__device__ __forceinline__ void walk_bin(const BinRows& R, int n, Load&& load, Apply&& apply) {
  const int lane = threadIdx.x & 31;
  int r = -1, lo = 0, len = 0, c = 0;
  auto advance = [&]() {
    for (++r; r < n; ++r) {
      len = rank_get(R.len, r);
      if (len > 0) {
        lo = rank_get(R.lo, r);
        c = 0;
        return;
      }
    }
  };
  advance();
  while (r < n) {
    bool ok[kChunks];
    int got = 0;
#pragma unroll
    for (int t = 0; t < kChunks; ++t) {
      ok[t] = false;
      if (r < n) {
        const int i = c + lane;
        if (i < len) {
          ok[t] = true;
          load(t, r, lo + i);
        }
        c += 32;
        if (c >= len) advance();
        got = t + 1;
      }
    }
#pragma unroll
    for (int t = 0; t < kChunks; ++t) {
      if (t < got) {
        apply(t, ok[t]);
        __syncwarp();
      }
    }
  }
}

// The count pass walks a bin flattened: rank r's entries are positions
// [lo[r], lo[r] + len) of its list and [epre[r], epre[r+1]) of the bin's
// rank-major flattened sequence.
struct BinRanks {
  int lo[ZR_MAX_RANKS];
  int epre[ZR_MAX_RANKS + 1];
};

// Clamps the fetched rows to the list lengths and fills R (warp-collective;
// ends with __syncwarp).  Returns the bin's entry count.
__device__ __forceinline__ int bin_commit(const Lists& lists, int n, const BinFetch& f,
                                          BinRanks& R) {
  const int lane = threadIdx.x & 31;
  int carry = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (32 * h >= n) break;
    const int r = lane + 32 * h;
    int lo = 0, len = 0;
    if (r < n) {
      const int nnz = (int)lists.nnz[r];
      lo = min(max(f.lo[h], 0), nnz);
      len = min(max(f.hi[h], lo), nnz) - lo;
    }
    const int incl = warp_incl_scan(len);
    if (r < n) {
      R.lo[r] = lo;
      R.epre[r] = carry + incl - len;
    }
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) R.epre[n] = carry;
  __syncwarp();
  return carry;
}

// Walks the bin's flattened entries 32 at a time (lane l takes position
// k0 + l), kBatch groups per batch: load(t, rank, pos) is issued for every
// entry of a batch, then apply(rank) runs once for the batch, where rank[t]
// is the lane's rank in group t (-1 where the lane holds no entry).  Every
// lane keeps a cursor on its current rank and moves it forward only when
// its position passes the rank's end, so ranks are non-decreasing in
// (group, lane) order.  apply is called by every lane, so it may use warp
// collectives.
template <typename Load, typename Apply>
__device__ __forceinline__ void for_bin_entries(const Lists& lists, int n, const BinRanks& R,
                                                int total, int32_t* status, Load&& load,
                                                Apply&& apply) {
  const int lane = threadIdx.x & 31;
  int cr = 0, cend = R.epre[1];
  int off = R.lo[0];  // list position = off + k inside rank cr
  int lim = (int)lists.nnz[0];
  for (int k0 = 0; k0 < total; k0 += 32 * kBatch) {
    int rank[kBatch];
#pragma unroll
    for (int t = 0; t < kBatch; ++t) {
      const int k = k0 + 32 * t + lane;
      rank[t] = -1;
      if (k < total) {
        if (k >= cend && cr < n - 1) {
          int cstart;
          do {
            ++cr;
            cstart = cend;
            cend = R.epre[cr + 1];
          } while (k >= cend && cr < n - 1);
          off = R.lo[cr] - cstart;
          lim = (int)lists.nnz[cr];
        }
        const int pos = off + k;
        if ((unsigned)pos < (unsigned)lim) {
          rank[t] = cr;
          load(t, cr, pos);
        } else {
          flag(status, ZR_ERR_INTERNAL);  // cannot happen; skipped, never read
        }
      }
    }
    apply(k0, rank);
  }
}

// ------------------------------------------------------------ 2. count
// Per bin, a warp builds the bin's union bitmap and counts its members per
// partition; lane p then publishes cnt[p][b].  Sparse bins (fewer entries
// than W/4) count at the entry that sets a bit (the first holder); dense
// bins OR every key in without waiting for the old word and then hash the
// bitmap one word per step, a lane per key.  Bins are dealt to warps with a
// grid-wide stride, so a dense region of the key range is spread over many
// warps, and no warp waits on another.
__global__ void __launch_bounds__(kBinThreads)
bin_count_kernel(const __grid_constant__ Lists lists, int n, int log_w, int bins,
                 const int32_t* starts, H0 h, int parts, int32_t* cnt_g, int32_t* status) {
  __shared__ uint32_t ubits_all[kBinWarps][128];
  __shared__ int32_t wc_all[kBinWarps][ZR_MAX_PARTS];
  __shared__ BinRanks ranks_all[kBinWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t* ub = ubits_all[warp];
  int32_t* wc = wc_all[warp];
  BinRanks& R = ranks_all[warp];
  const H0 hash = h;
  const int words = 1 << (log_w - 5);
  const int W = 1 << log_w;
  const int nwarps = gridDim.x * kBinWarps;
  for (int p = lane; p < parts; p += 32) wc[p] = 0;
  int b = blockIdx.x * kBinWarps + warp;
  BinFetch fetch = {};
  if (b < bins) fetch = bin_fetch(starts, n, bins, b);
  for (; b < bins; b += nwarps) {
    const uint32_t base = (uint32_t)b << log_w;
    for (int w = lane; w < words; w += 32) ub[w] = 0;
    const int total = bin_commit(lists, n, fetch, R);
    if (b + nwarps < bins) fetch = bin_fetch(starts, n, bins, b + nwarps);
    int key[kBatch];
    auto load = [&](int t, int r, int pos) { key[t] = __ldg(lists.idx[r] + pos); };
    if (total * 4 < W) {
      for_bin_entries(lists, n, R, total, status, load, [&](int, const int (&rank)[kBatch]) {
#pragma unroll
        for (int t = 0; t < kBatch; ++t) {
          const uint32_t slot = (uint32_t)key[t] - base;
          if (rank[t] >= 0 && slot < (uint32_t)W) {
            const uint32_t bit = 1u << (slot & 31);
            if (!(atomicOr(&ub[slot >> 5], bit) & bit)) {
              const int p = parts > 1 ? (int)hash((uint32_t)key[t]) : 0;
              if ((unsigned)p < (unsigned)parts) atomicAdd(&wc[p], 1);
              else flag(status, ZR_ERR_INTERNAL);
            }
          }
        }
      });
      __syncwarp();
    } else {
      for_bin_entries(lists, n, R, total, status, load, [&](int, const int (&rank)[kBatch]) {
#pragma unroll
        for (int t = 0; t < kBatch; ++t) {
          const uint32_t slot = (uint32_t)key[t] - base;
          if (rank[t] >= 0 && slot < (uint32_t)W) atomicOr(&ub[slot >> 5], 1u << (slot & 31));
        }
      });
      __syncwarp();
      for (int w = 0; w < words; ++w) {
        if ((ub[w] >> lane) & 1u) {
          const int p = parts > 1 ? (int)hash(base + (uint32_t)(w * 32 + lane)) : 0;
          if ((unsigned)p < (unsigned)parts) atomicAdd(&wc[p], 1);
          else flag(status, ZR_ERR_INTERNAL);
        }
      }
      __syncwarp();
    }
    for (int p = lane; p < parts; p += 32) {
      __stcg(cnt_g + (size_t)p * bins + b, wc[p]);
      wc[p] = 0;
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------ 3. scan
// Two launches over grid (chunk of 2048 bins, partition): the first sums
// each chunk's counts, the second adds the earlier chunks' sums (the carry)
// to a block-wide scan of its chunk: excl[p][b] = sum_{b' < b} cnt[p][b'].
// The last chunk also writes the partition total.
__device__ __forceinline__ long long block_sum(long long v, long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  long long t = 0;
  if (warp == 0) {
    t = lane < (int)(blockDim.x >> 5) ? red[lane] : 0;
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  }
  return t;  // valid in warp 0
}

__global__ void __launch_bounds__(kScanThreads)
bin_chunk_sum_kernel(const int32_t* cnt_g, int bins, long long* ctot_g) {
  __shared__ long long red[kScanThreads / 32];
  const int c = blockIdx.x, p = blockIdx.y, chunks = gridDim.x;
  const int b0 = (c << kChunkLog) + threadIdx.x * 2;
  const int32_t* row = cnt_g + (size_t)p * bins;
  long long v = 0;
  if (b0 < bins) v += __ldcg(row + b0);
  if (b0 + 1 < bins) v += __ldcg(row + b0 + 1);
  const long long t = block_sum(v, red);
  if (threadIdx.x == 0) ctot_g[(size_t)p * chunks + c] = t;
}

__global__ void __launch_bounds__(kScanThreads)
bin_scan_kernel(const int32_t* cnt_g, const long long* ctot_g, int bins, long long* excl_g,
                long long* tot_g) {
  __shared__ long long red[kScanThreads / 32];
  __shared__ long long s_carry;
  const int c = blockIdx.x, p = blockIdx.y, chunks = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  long long before = 0;
  for (int j = tid; j < c; j += kScanThreads) before += __ldcg(ctot_g + (size_t)p * chunks + j);
  const long long carry_sum = block_sum(before, red);
  if (tid == 0) s_carry = carry_sum;
  __syncthreads();
  const int b0 = (c << kChunkLog) + tid * 2;
  const int32_t* row = cnt_g + (size_t)p * bins;
  const int v0 = b0 < bins ? __ldcg(row + b0) : 0;
  const int v1 = b0 + 1 < bins ? __ldcg(row + b0 + 1) : 0;
  const int s = v0 + v1;
  const int incl = warp_incl_scan(s);
  if (lane == 31) red[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const long long x = red[lane];
    long long xi = x;
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, xi, o);
      if (lane >= o) xi += y;
    }
    red[lane] = xi - x;
    if (lane == 31 && c == chunks - 1) tot_g[p] = s_carry + xi;
  }
  __syncthreads();
  const long long run = s_carry + red[warp] + (incl - s);
  long long* out = excl_g + (size_t)p * bins;
  if (b0 < bins) out[b0] = run;
  if (b0 + 1 < bins) out[b0 + 1] = run + v0;
}

// ------------------------------------------------------------ 4. write
// offs[0..parts] = exclusive prefix of the partition totals (shared memory);
// block 0 of the grid also writes d_offsets and the grand total.
__device__ void load_partition_offsets(const long long* tot_g, int parts, long long* offs,
                                       int64_t* d_offsets, int64_t* d_total) {
  for (int p = threadIdx.x; p < parts; p += blockDim.x) offs[p] = __ldcg(tot_g + p);
  __syncthreads();
  if (threadIdx.x == 0) {
    long long acc = 0;
    for (int p = 0; p < parts; ++p) {
      const long long t = offs[p];
      offs[p] = acc;
      acc += t;
    }
    offs[parts] = acc;
    if (blockIdx.x == 0) {
      if (d_offsets)
        for (int p = 0; p <= parts; ++p) d_offsets[p] = offs[p];
      if (d_total) *d_total = acc;
    }
  }
  __syncthreads();
}

// How the writer places a bin's members into their partitions' runs:
//   kPlaceLane  per-lane partition counters (at most 32 partitions; bins with
//               few members, where a pass per partition would mostly idle);
//   kPlaceMask  per-partition member bitmaps, emitted partition by partition
//               (at most 32 partitions; bins with many members);
//   kPlaceSort  a counting sort of the bin's member list (any partition count).
enum Placement { kPlaceLane = 0, kPlaceMask = 1, kPlaceSort = 2 };

// Warp-private shared memory of the writer; acc[W] (f32) comes first, so
// that it is 16-byte aligned, then ub[W/32] and
//   kPlaceLane: the lanes' partition counters (32 rows of row_words(parts)
//               words, two 16-bit counters per word) and the bin's run
//               bases gbs[parts] (i64);
//   kPlaceMask: the member bitmaps pm[parts][W/32];
//   kPlaceSort: run[parts] (i32), wdelta[parts] (i64), mlist[W] and
//               stage[W] (u16).
__host__ __device__ inline int row_words(int parts) {
  return ((parts + 1) >> 1) | 1;  // odd, so lane rows fall in distinct banks
}

template <int kPlace>
__host__ __device__ inline size_t warp_smem_bytes(int log_w, int parts) {
  const size_t W = (size_t)1 << log_w, words = W / 32, P = (size_t)parts;
  size_t b = W * 4 + words * 4;
  if (kPlace == kPlaceLane) b += 32 * 4 * (size_t)row_words(parts) + P * 8;
  else if (kPlace == kPlaceMask) b += words * 4 * P;
  else b += ((P + 1) & ~(size_t)1) * 4 + P * 8 + W * 4;
  return (b + 15) & ~(size_t)15;
}

// The 1/N average: none, a multiply by the exact reciprocal (N a power of
// two, where it equals the correctly rounded quotient), or the correctly
// rounded division.
enum AvgKind { kAvgNone = 0, kAvgPow2 = 1, kAvgDiv = 2 };

template <int kAvg>
__device__ __forceinline__ float averaged(float v, float fn, float inv) {
  if (kAvg == kAvgPow2) return v * inv;
  if (kAvg == kAvgDiv) return __fdiv_rn(v, fn);
  return v;
}

constexpr int kWriteChunks = 12;  // chunk loads per batch (4, 8, 12, 16 measured on C5b; 12 fastest)
// Average entries per 1024-key bin from which the writer emits partition by
// partition (kPlaceMask): measured on the C4 embedding lists (82 entries a
// bin, per-lane counters faster) and the C5b top-k lists (819 a bin, the
// bitmaps faster).
constexpr int64_t kMaskMinPerBin = 256;

// Per bin:
//   fold    the bin's entries rank by rank (walk_bin) into acc[], which
//           starts at -0.0, the identity of the fold (-0.0 + x == x for
//           every x that is not a NaN), so every member ends as the left fold
//           of its holders in rank order; the union bitmap ub is ORed alongside.
//   kPlaceLane:
//     count lane l takes the ub words of keys [32 wpl l, 32 wpl (l + 1)) (its
//           members, in key order), hashes each member and counts it in its
//           own row of 16-bit counters, one per partition, two per word;
//     scan  a prefix over the lanes of each counter word (two partitions at
//           once) turns the rows into each lane's first position inside the
//           bin's run of every partition; the totals are checked against the
//           count pass and the output bounds;
//     emit  each lane walks its members again in key order and writes each
//           to gbs[p] + its counter, then advances the counter.
//   kPlaceMask:
//     mask  lane l takes ub words l, l + 32, ...: each member is hashed and
//           its bit set in pm[p] (a lane owns its words, so no two lanes
//           write one word);
//     emit  partition by partition, lane l takes pm[p] words l, l + 32, ...;
//           a prefix of their popcounts over the lanes gives each lane the
//           position of its first member inside the bin's run of p, and the
//           lane writes its members in ascending key order;
//   kPlaceSort:
//     list  the members' slots in ascending key order (mlist);
//     place a stable counting sort of mlist by partition into stage[]
//           (match_any groups the lanes of one partition);
//     emit  stage[] 32 entries at a time to offs[p] + excl[p][b] + its rank
//           inside the bin's run of partition p.
// ub, the counters and pm are cleared after use; acc is reset per bin.
template <int kPlace, int kAvg>
__global__ void __launch_bounds__(kWriteThreads)
bin_write_kernel(const __grid_constant__ Lists lists, int n, int log_w, int bins,
                 const int32_t* starts, H0 h, int parts, const int32_t* cnt_g,
                 const long long* excl_g, const long long* tot_g, int32_t* out_idx,
                 float* out_val, int64_t out_cap, int64_t* d_offsets, int64_t* d_total,
                 int32_t* status) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ long long offs[ZR_MAX_PARTS + 1];
  __shared__ BinRanks flat_all[kPlace == kPlaceLane ? kWriteWarps : 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int W = 1 << log_w;
  const int words = W >> 5;
  constexpr bool kLane = kPlace == kPlaceLane;
  constexpr bool kMask = kPlace == kPlaceMask;
  unsigned char* mine = smem + (size_t)warp * warp_smem_bytes<kPlace>(log_w, parts);
  float* acc = reinterpret_cast<float*>(mine);
  const H0 hash = h;
  const float fn = (float)n, inv = 1.0f / (float)n;
  const unsigned lt = lanemask_lt();
  load_partition_offsets(tot_g, parts, offs, d_offsets, d_total);

  const int wpl = words >> 5;  // bitmap words per lane
  const int rs = row_words(parts);
  uint32_t* ub = reinterpret_cast<uint32_t*>(acc + W);
  uint32_t* rows = nullptr;
  long long* gbs = nullptr;
  uint32_t* pm = nullptr;
  long long* wdelta = nullptr;
  int32_t* run = nullptr;
  uint16_t* mlist = nullptr;
  uint16_t* stage = nullptr;
  if (kLane) {
    rows = ub + words;
    gbs = reinterpret_cast<long long*>(rows + 32 * rs);
    for (int i = lane; i < words + 32 * rs; i += 32) ub[i] = 0;  // ub and the rows
  } else if (kMask) {
    pm = ub + words;
    for (int i = lane; i < words * (parts + 1); i += 32) ub[i] = 0;  // ub and pm
  } else {
    run = reinterpret_cast<int32_t*>(ub + words);
    wdelta = reinterpret_cast<long long*>(run + ((parts + 1) & ~1));
    mlist = reinterpret_cast<uint16_t*>(wdelta + parts);
    stage = mlist + W;
    for (int i = lane; i < words; i += 32) ub[i] = 0;
  }
  __syncwarp();

  const int nwarps = gridDim.x * kWriteWarps;
  int b = blockIdx.x * kWriteWarps + warp;
  // next bin's start rows, and (kLane, kMask) lane p's count and prefix for it
  BinFetch fetch = {};
  int pc_next = 0;
  long long pe_next = 0;
  if (b < bins) {
    fetch = bin_fetch(starts, n, bins, b);
    if ((kLane || kMask) && lane < parts) {
      pc_next = __ldcg(cnt_g + (size_t)lane * bins + b);
      pe_next = __ldcg(excl_g + (size_t)lane * bins + b);
    }
  }
  for (; b < bins; b += nwarps) {
    const uint32_t base = (uint32_t)b << log_w;
    const BinRows R = bin_rows(lists, n, fetch);
    const BinFetch fetch_cur = fetch;
    const int pc = pc_next;
    const long long pe = pe_next;
    if (b + nwarps < bins) {
      fetch = bin_fetch(starts, n, bins, b + nwarps);
      if ((kLane || kMask) && lane < parts) {
        pc_next = __ldcg(cnt_g + (size_t)lane * bins + b + nwarps);
        pe_next = __ldcg(excl_g + (size_t)lane * bins + b + nwarps);
      }
    }
    for (int i = lane; i < (W >> 2); i += 32)
      reinterpret_cast<float4*>(acc)[i] = make_float4(-0.0f, -0.0f, -0.0f, -0.0f);
    __syncwarp();

    // fold
    if (kLane) {
      // Sparse bins: the flattened walk (groups of 32 entries across rank
      // boundaries).  Keys that strictly ascend across a group's lanes are
      // distinct and apply at once; otherwise each maximal ascending run of
      // lanes goes in lane order, so a key held by two ranks meets the lower
      // rank first.
      BinRanks& F = flat_all[warp];
      const int total = bin_commit(lists, n, fetch_cur, F);
      int fkey[kBatch];
      float fval[kBatch];
      for_bin_entries(
          lists, n, F, total, status,
          [&](int t, int r, int pos) {
            fkey[t] = __ldg(lists.idx[r] + pos);
            fval[t] = __ldg(lists.val[r] + pos);
          },
          [&](int k0, const int (&rank)[kBatch]) {
#pragma unroll
            for (int t = 0; t < kBatch; ++t) {
              if (k0 + 32 * t < total) {
                const uint32_t slot = (uint32_t)fkey[t] - base;
                const bool live = rank[t] >= 0;
                const bool in = live && slot < (uint32_t)W;
                const int prev = __shfl_up_sync(0xffffffffu, fkey[t], 1);
                const unsigned desc =
                    __ballot_sync(0xffffffffu, live && lane > 0 && prev >= fkey[t]);
                const int run_id = __popc(desc & (lt | (1u << lane)));
                const int runs = __popc(desc) + 1;
                for (int q = 0; q < runs; ++q) {
                  if (in && run_id == q) {
                    acc[slot] = __fadd_rn(acc[slot], fval[t]);
                    atomicOr(&ub[slot >> 5], 1u << (slot & 31));
                  }
                  __syncwarp();
                }
              }
            }
          });
    } else {
      int key[kWriteChunks];
      float val[kWriteChunks];
      walk_bin<kWriteChunks>(
          R, n,
          [&](int t, int r, int pos) {
            key[t] = __ldg(lists.idx[r] + pos);
            val[t] = __ldg(lists.val[r] + pos);
          },
          [&](int t, bool ok) {
            const uint32_t slot = (uint32_t)key[t] - base;
            if (ok && slot < (uint32_t)W) {
              acc[slot] = __fadd_rn(acc[slot], val[t]);
              atomicOr(&ub[slot >> 5], 1u << (slot & 31));
            }
          });
    }

    if (kLane) {
      uint32_t* row = rows + lane * rs;
      uint16_t* row16 = reinterpret_cast<uint16_t*>(row);
      // count
      for (int q = 0; q < wpl; ++q) {
        const int w = lane * wpl + q;
        uint32_t bits = ub[w];
        while (bits) {
          const int bit = __ffs(bits) - 1;
          bits &= bits - 1;
          const int p = parts > 1 ? (int)hash(base + (uint32_t)(w * 32 + bit)) : 0;
          if ((unsigned)p < (unsigned)parts) row16[p] = (uint16_t)(row16[p] + 1);
          else flag(status, ZR_ERR_INTERNAL);
        }
      }
      // scan (every field stays below 2^16: a bin has at most 4096 members)
      int mytot = 0;
      for (int q = 0; q < (parts + 1) >> 1; ++q) {
        const uint32_t v = row[q];
        const uint32_t incl = (uint32_t)warp_incl_scan((int)v);
        row[q] = incl - v;
        const uint32_t tq = __shfl_sync(0xffffffffu, incl, 31);
        if ((lane >> 1) == q) mytot = (int)((lane & 1) ? tq >> 16 : tq & 0xffffu);
      }
      // The count pass saw the same entries, so every run has the counted
      // size and lies inside the output; a bin where one does not is not
      // written.
      bool bad = false;
      if (lane < parts) {
        const long long g = offs[lane] + pe;
        bad = mytot != pc || g < 0 || g + pc > out_cap;
        gbs[lane] = g;
      }
      const bool skip = __any_sync(0xffffffffu, bad);
      if (skip && lane == 0) flag(status, ZR_ERR_INTERNAL);
      __syncwarp();
      // emit
      for (int q = 0; q < wpl; ++q) {
        const int w = lane * wpl + q;
        uint32_t bits = skip ? 0u : ub[w];
        ub[w] = 0;
        while (bits) {
          const int bit = __ffs(bits) - 1;
          bits &= bits - 1;
          const int slot = w * 32 + bit;
          const int p = parts > 1 ? (int)hash(base + (uint32_t)slot) : 0;
          if ((unsigned)p < (unsigned)parts) {
            const int at = row16[p];
            row16[p] = (uint16_t)(at + 1);
            const long long dst = gbs[p] + at;
            out_idx[dst] = (int32_t)(base + (uint32_t)slot);
            out_val[dst] = averaged<kAvg>(acc[slot], fn, inv);
          }
        }
      }
      for (int q = 0; q < rs; ++q) row[q] = 0;
      __syncwarp();
      continue;
    }

    if (kMask) {
      // mask
      for (int w = lane; w < words; w += 32) {
        uint32_t bits = ub[w];
        ub[w] = 0;
        while (bits) {
          const int bit = __ffs(bits) - 1;
          bits &= bits - 1;
          const int p = parts > 1 ? (int)hash(base + (uint32_t)(w * 32 + bit)) : 0;
          if ((unsigned)p < (unsigned)parts) pm[p * words + w] |= 1u << bit;
          else flag(status, ZR_ERR_INTERNAL);
        }
      }
      __syncwarp();
      // emit
      const long long gb = lane < parts ? offs[lane] + pe : 0;
      for (int p = 0; p < parts; ++p) {
        const long long g = __shfl_sync(0xffffffffu, gb, p);
        const int want = __shfl_sync(0xffffffffu, pc, p);
        // The count pass saw the same entries, so the run has want members
        // and lies inside the output; a run that does not is not written.
        const bool fits = g >= 0 && g + want <= out_cap;
        int32_t* oi = out_idx + (fits ? g : 0);
        float* ov = out_val + (fits ? g : 0);
        uint32_t* pmp = pm + p * words;
        int carry = 0;
        for (int w0 = 0; w0 < words; w0 += 32) {
          const int w = w0 + lane;
          uint32_t bits = 0;
          if (w < words) {
            bits = pmp[w];
            pmp[w] = 0;
          }
          const int c = __popc(bits);
          const int incl = warp_incl_scan(c);
          int at = carry + incl - c;
          carry += __shfl_sync(0xffffffffu, incl, 31);
          if (!fits || carry > want) continue;
          while (bits) {
            const int bit = __ffs(bits) - 1;
            bits &= bits - 1;
            const int slot = w * 32 + bit;
            oi[at] = (int32_t)(base + (uint32_t)slot);
            ov[at] = averaged<kAvg>(acc[slot], fn, inv);
            ++at;
          }
        }
        if (lane == 0 && (!fits || carry != want))
          flag(status, fits ? ZR_ERR_INTERNAL : ZR_ERR_INPUT_UNSORTED);
      }
      __syncwarp();
      continue;
    }

    // list: lane l owns words [l * wpl, (l + 1) * wpl)
    int mine_cnt = 0;
    for (int q = 0; q < wpl; ++q) mine_cnt += __popc(ub[lane * wpl + q]);
    const int incl = warp_incl_scan(mine_cnt);
    const int members = __shfl_sync(0xffffffffu, incl, 31);
    int at = incl - mine_cnt;
    for (int q = 0; q < wpl; ++q) {
      const int w = lane * wpl + q;
      uint32_t bits = ub[w];
      ub[w] = 0;
      while (bits) {
        const int bit = __ffs(bits) - 1;
        bits &= bits - 1;
        mlist[at++] = (uint16_t)(w * 32 + bit);
      }
    }
    // This bin's partition runs: run[p] (bin-local start) and the global base.
    int expect = 0;
    for (int p0 = 0; p0 < parts; p0 += 32) {
      const int p = p0 + lane;
      const int c = p < parts ? __ldcg(cnt_g + (size_t)p * bins + b) : 0;
      const long long e = p < parts ? __ldcg(excl_g + (size_t)p * bins + b) : 0;
      const int pincl = warp_incl_scan(c);
      if (p < parts) {
        run[p] = expect + pincl - c;
        wdelta[p] = offs[p] + e - (expect + pincl - c);
      }
      expect += __shfl_sync(0xffffffffu, pincl, 31);
    }
    __syncwarp();
    if (members != expect) {
      // The count pass saw the same entries, so this cannot happen.
      if (lane == 0) flag(status, ZR_ERR_INTERNAL);
      __syncwarp();
      continue;
    }
    // place
    for (int j0 = 0; j0 < members; j0 += 32) {
      const int j = j0 + lane;
      const bool live = j < members;
      const int slot = live ? mlist[j] : 0;
      int p = live ? (int)hash(base + (uint32_t)slot) : parts;
      if (live && (unsigned)p >= (unsigned)parts) {
        flag(status, ZR_ERR_INTERNAL);
        p = parts;
      }
      const bool ok = live && p < parts;
      const unsigned peers = __match_any_sync(0xffffffffu, p);
      if (ok) {
        const int sidx = run[p] + __popc(peers & lt);
        if ((unsigned)sidx < (unsigned)members) stage[sidx] = (uint16_t)slot;
        else flag(status, ZR_ERR_INTERNAL);
      }
      __syncwarp();
      if (ok && (peers & lt) == 0) run[p] += __popc(peers);
      __syncwarp();
    }
    // emit
    for (int j = lane; j < members; j += 32) {
      const int slot = stage[j];
      const uint32_t k = base + (uint32_t)slot;
      const int p = (int)hash(k);
      if (slot < W && (unsigned)p < (unsigned)parts) {
        const long long dst = wdelta[p] + j;
        if (dst >= 0 && dst < out_cap) {
          out_idx[dst] = (int32_t)k;
          out_val[dst] = averaged<kAvg>(acc[slot], fn, inv);
        } else {
          flag(status, ZR_ERR_INPUT_UNSORTED);
        }
      } else {
        flag(status, ZR_ERR_INTERNAL);
      }
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------ densification
// Union sizes of rank groups (Zen section 2.3, the densification ratios
// gamma_k of Equations (1) and (2)).  Per bin, a warp ORs 1 << r into a
// 64-bit holder mask per key for every entry of rank r; then, for every key
// with a holder, level L folds the mask so that bit i * 2^L holds the OR of
// group i's 2^L ranks, and the set bits at multiples of 2^L count the
// groups of size 2^L whose union holds the key.  Sums per level stay in
// registers until one atomic per warp at the end (per-CTA partial sums and a
// one-CTA reduction measured slower on C4: the extra launch costs more than
// the atomics).
constexpr int kDensWarps = 4;
constexpr int kDensChunks = 12;   // as the writer's

// Bits 0, 2^L, 2 * 2^L, ... of a holder mask: the first rank of every group
// of 2^L consecutive ranks.
template <typename M>
__device__ __forceinline__ M group_sel(int level) {
  switch (level) {
    case 1: return (M)0x5555555555555555ull;
    case 2: return (M)0x1111111111111111ull;
    case 3: return (M)0x0101010101010101ull;
    case 4: return (M)0x0001000100010001ull;
    case 5: return (M)0x0000000100000001ull;
    default: return (M)1;
  }
}

__device__ __forceinline__ int popc_mask(uint32_t m) { return __popc(m); }
__device__ __forceinline__ int popc_mask(unsigned long long m) { return __popcll(m); }

// M: the holder mask type (32-bit up to 32 ranks, else 64-bit); kLogN:
// log2 of the rank count; kFlat: the flattened walk (lists with few entries
// per bin on average) or the rank-by-rank walk.  Per warp: masks mk[W] and
// the list of the bin's keys in first-holder order, mlist[W] (u16).
template <typename M, int kLogN, bool kFlat>
__global__ void __launch_bounds__(kDensWarps * 32)
densify_kernel(const __grid_constant__ Lists lists, int n, int log_w, int bins,
               const int32_t* starts, int64_t total_nnz, unsigned long long* counts,
               int32_t* status) {
  extern __shared__ __align__(16) unsigned char dens_smem[];
  __shared__ BinRanks flat_all[kFlat ? kDensWarps : 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int W = 1 << log_w;
  M* mk = reinterpret_cast<M*>(dens_smem + (size_t)warp * W * (sizeof(M) + 2));
  uint16_t* mlist = reinterpret_cast<uint16_t*>(mk + W);
  const unsigned lt = lanemask_lt();
  unsigned long long cnt[kLogN > 0 ? kLogN : 1] = {};
  const int nwarps = gridDim.x * kDensWarps;
  for (int i = lane; i < W; i += 32) mk[i] = 0;  // then cleared as it is read
  for (int b = blockIdx.x * kDensWarps + warp; b < bins; b += nwarps) {
    const uint32_t base = (uint32_t)b << log_w;
    // lane r (and r + 32) holds rank r's slice of this bin
    int lo[2], hi[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = lane + 32 * h;
      lo[h] = hi[h] = 0;
      if (r < n) {
        const int32_t* row = starts + (size_t)r * (bins + 1) + b;
        const int nnz = (int)lists.nnz[r];
        lo[h] = min(max(__ldcg(row), 0), nnz);
        hi[h] = min(max(__ldcg(row + 1), lo[h]), nnz);
      }
    }
    __syncwarp();
    int members = 0;
    BinFetch fetch;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      fetch.lo[h] = lo[h];
      fetch.hi[h] = hi[h];
    }
    if (kFlat) {
      BinRanks& F = flat_all[warp];
      const int total = bin_commit(lists, n, fetch, F);
      // Sparse bins: the flattened walk (groups of 32 entries across rank
      // boundaries, as the writer's), the masks ORed with shared-memory
      // atomics, since two lanes of a group may hold one key; the atomic's
      // old value says which entry is the key's first holder.
      int fkey[kBatch];
      for_bin_entries(
          lists, n, F, total, status,
          [&](int t, int r, int pos) { fkey[t] = __ldg(lists.idx[r] + pos); },
          [&](int, const int (&rank)[kBatch]) {
#pragma unroll
            for (int t = 0; t < kBatch; ++t) {
              const uint32_t slot = (uint32_t)fkey[t] - base;
              bool first = false;
              if (rank[t] >= 0 && slot < (uint32_t)W)
                first = atomicOr(&mk[slot], (M)1 << rank[t]) == 0;
              const unsigned fresh = __ballot_sync(0xffffffffu, first);
              if (first) mlist[members + __popc(fresh & lt)] = (uint16_t)slot;
              members += __popc(fresh);
            }
          });
    } else {
    // Rank by rank in chunks of up to 32 entries (walk_bin, 12 chunks' loads
    // in flight): a list is strictly ascending, so the lanes of one chunk
    // hold distinct keys and a plain read-modify-write of the mask is
    // race-free; chunks are ordered by a warp barrier.  A key whose mask was
    // empty joins the member list.
    BinRows R;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      R.lo[h] = lo[h];
      R.len[h] = hi[h] - lo[h];
    }
    int key[kDensChunks], rk[kDensChunks];
    walk_bin<kDensChunks>(
        R, n,
        [&](int t, int r, int pos) {
          key[t] = __ldg(lists.idx[r] + pos);
          rk[t] = r;
        },
        [&](int t, bool ok) {
          const uint32_t slot = (uint32_t)key[t] - base;
          bool first = false;
          if (ok && slot < (uint32_t)W) {
            const M old = mk[slot];
            mk[slot] = old | ((M)1 << rk[t]);
            first = old == 0;
          }
          const unsigned fresh = __ballot_sync(0xffffffffu, first);
          if (first) mlist[members + __popc(fresh & lt)] = (uint16_t)slot;
          members += __popc(fresh);
        });
    }
    __syncwarp();
    // every member: fold its mask level by level and count the groups
    for (int j = lane; j < members; j += 32) {
      const int slot = mlist[j];
      M m = mk[slot];
      mk[slot] = 0;
#pragma unroll
      for (int level = 1; level <= kLogN; ++level) {
        m |= m >> (1 << (level - 1));
        cnt[level - 1] += popc_mask((M)(m & group_sel<M>(level)));
      }
    }
    __syncwarp();
  }
#pragma unroll
  for (int level = 1; level <= kLogN; ++level) {
    unsigned long long v = cnt[level - 1];
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0 && v) atomicAdd(&counts[level], v);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) atomicAdd(&counts[0], (unsigned long long)total_nnz);
}

// ------------------------------------------------------------ launch helpers
int per_sm(const void* fn, int threads, size_t smem) {
  int b = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, threads, smem) != cudaSuccess || b < 1)
    b = 1;
  return b;
}

int64_t grid_for(int64_t units, int blocks_per_sm) {
  int64_t g = (int64_t)sm_count() * blocks_per_sm;
  if (g > units) g = units;
  return g < 1 ? 1 : g;
}

// The write kernel for a placement (partition masks or the sort) and an
// average mode.
template <int kPlace>
const void* write_kernel_avg(int avg_kind) {
  if (avg_kind == kAvgPow2) return (const void*)bin_write_kernel<kPlace, kAvgPow2>;
  if (avg_kind == kAvgDiv) return (const void*)bin_write_kernel<kPlace, kAvgDiv>;
  return (const void*)bin_write_kernel<kPlace, kAvgNone>;
}

const void* write_kernel(int place, int avg_kind) {
  if (place == kPlaceLane) return write_kernel_avg<kPlaceLane>(avg_kind);
  if (place == kPlaceMask) return write_kernel_avg<kPlaceMask>(avg_kind);
  return write_kernel_avg<kPlaceSort>(avg_kind);
}

size_t write_smem(int place, int log_w, int parts) {
  const size_t per_warp = place == kPlaceLane   ? warp_smem_bytes<kPlaceLane>(log_w, parts)
                          : place == kPlaceMask ? warp_smem_bytes<kPlaceMask>(log_w, parts)
                                                : warp_smem_bytes<kPlaceSort>(log_w, parts);
  return kWriteWarps * per_warp;
}

// Per-device cached occupancy, and the dynamic shared-memory opt-in of the
// write kernels (done once per device).
struct DeviceInfo {
  std::atomic<int> ready{0};
  int count_per_sm = 1;
};

// One thread fills a device's entry (under the lock); later calls read it
// after seeing `ready`.
DeviceInfo* device_info() {
  static DeviceInfo info[64];
  static std::mutex init_lock;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  DeviceInfo& d = info[dev];
  if (d.ready.load(std::memory_order_acquire)) return &d;
  std::lock_guard<std::mutex> guard(init_lock);
  if (!d.ready.load(std::memory_order_relaxed)) {
    for (int place = 0; place < 3; ++place) {
      const int most = (int)write_smem(place, 12, place == kPlaceSort ? ZR_MAX_PARTS : 32);
      for (int a = 0; a < 3; ++a)
        if (cudaFuncSetAttribute(write_kernel(place, a),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 most) != cudaSuccess)
          return nullptr;
    }
    d.count_per_sm = per_sm((const void*)bin_count_kernel, kBinThreads, 0);
    d.ready.store(1, std::memory_order_release);
  }
  return &d;
}

}  // namespace

size_t sparse_workspace_bytes(int n, int64_t dense_size, int n_parts) {
  const int parts = n_parts > 0 ? n_parts : 1;
  const Geometry g = geometry(n, dense_size, parts, -1);  // narrowest bins: an upper bound
  return sparse_layout(n, g.bins, parts).total;
}

zr_status sparse_launch(const int32_t* const* idx, const float* const* val, const int64_t* nnz,
                        int n, int64_t dense_size, int n_parts, uint64_t part_seed, int average,
                        int32_t* out_idx, float* out_val, int64_t out_cap, int64_t* d_out_nnz,
                        int64_t* d_offsets, void* ws, cudaStream_t stream) {
  const int parts = n_parts > 0 ? n_parts : 1;
  Lists lists;
  int64_t max_nnz = 0, total_nnz = 0;
  for (int r = 0; r < ZR_MAX_RANKS; ++r) {
    const bool live = r < n && nnz[r] > 0;
    lists.idx[r] = live ? idx[r] : nullptr;
    lists.val[r] = live ? val[r] : nullptr;
    lists.nnz[r] = r < n ? nnz[r] : 0;
    if (r < n) {
      max_nnz = nnz[r] > max_nnz ? nnz[r] : max_nnz;
      total_nnz += nnz[r];
    }
  }
  const Geometry g = geometry(n, dense_size, parts, total_nnz);
  const SparseLayout L = sparse_layout(n, g.bins, parts);
  unsigned char* w = static_cast<unsigned char*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  int32_t* starts = reinterpret_cast<int32_t*>(w + L.starts);
  int32_t* cnt = reinterpret_cast<int32_t*>(w + L.cnt);
  long long* excl = reinterpret_cast<long long*>(w + L.excl);
  long long* tot = reinterpret_cast<long long*>(w + L.tot);
  const int bins = (int)g.bins;
  const H0 h = make_h0(part_seed, (uint32_t)parts);
  DeviceInfo* dinfo = device_info();
  if (!dinfo) return ZR_ERR_CUDA;
  // the status word starts at zero
  if (cudaMemsetAsync(w, 0, L.starts, stream) != cudaSuccess) return ZR_ERR_CUDA;
  {
    // one wave of CTAs over the n lists
    const int64_t groups = max_nnz / 4 + 1;
    int64_t gx = (groups + 256 * kStartsUnroll - 1) / (256 * kStartsUnroll);
    const int64_t cap = ((int64_t)sm_count() * 8 + n - 1) / n;
    if (gx > cap) gx = cap;
    if (gx < 1) gx = 1;
    bin_starts_kernel<<<dim3((unsigned)gx, (unsigned)n), 256, 0, stream>>>(
        lists, (int)dense_size, g.log_w, bins, starts, status);
  }
  const int chunks = (bins + kChunkBins - 1) >> kChunkLog;
  long long* ctot = reinterpret_cast<long long*>(w + L.ctot);
  {
    const int64_t warp_units = (g.bins + kBinWarps - 1) / kBinWarps;
    bin_count_kernel<<<(unsigned)grid_for(warp_units, dinfo->count_per_sm), kBinThreads, 0,
                       stream>>>(lists, n, g.log_w, bins, starts, h, parts, cnt, status);
  }
  if (chunks > 1)  // with one chunk the scan needs no carry
    bin_chunk_sum_kernel<<<dim3((unsigned)chunks, (unsigned)parts), kScanThreads, 0, stream>>>(
        cnt, bins, ctot);
  bin_scan_kernel<<<dim3((unsigned)chunks, (unsigned)parts), kScanThreads, 0, stream>>>(
      cnt, ctot, bins, excl, tot);
  int64_t* offsets_out = n_parts > 0 ? d_offsets : nullptr;
  const int avg_kind = !average ? kAvgNone : ((n & (n - 1)) == 0 ? kAvgPow2 : kAvgDiv);
  const int64_t write_units = (g.bins + kWriteWarps - 1) / kWriteWarps;
  // Bins with many members (on average) are emitted partition by partition,
  // others through per-lane counters; more than 32 partitions take the sort.
  const int place = parts > 32                                        ? kPlaceSort
                    : g.log_w == 10 && total_nnz >= kMaskMinPerBin * g.bins ? kPlaceMask
                                                                        : kPlaceLane;
  const size_t smem = write_smem(place, g.log_w, parts);
  const void* fn = write_kernel(place, avg_kind);
  const int o = per_sm(fn, kWriteThreads, smem);
  const unsigned grid = (unsigned)grid_for(write_units, o);
  const int32_t* cnt_c = cnt;
  const long long* excl_c = excl;
  const long long* tot_c = tot;
  void* args[] = {(void*)&lists, (void*)&n, (void*)&g.log_w, (void*)&bins, (void*)&starts,
                  (void*)&h, (void*)&parts, (void*)&cnt_c, (void*)&excl_c, (void*)&tot_c,
                  (void*)&out_idx, (void*)&out_val, (void*)&out_cap, (void*)&offsets_out,
                  (void*)&d_out_nnz, (void*)&status};
  if (cudaLaunchKernel(fn, dim3(grid), dim3(kWriteThreads), args, smem, stream) != cudaSuccess)
    return ZR_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
}

// The densification kernel for the rank count: 32-bit masks up to 32 ranks
// (log2 n <= 5), 64-bit masks above (log2 n = 6).
template <bool kFlat>
const void* densify_fn_walk(bool wide, int logn) {
  if (wide) return (const void*)densify_kernel<unsigned long long, 6, kFlat>;
  switch (logn) {
    case 0: return (const void*)densify_kernel<uint32_t, 0, kFlat>;
    case 1: return (const void*)densify_kernel<uint32_t, 1, kFlat>;
    case 2: return (const void*)densify_kernel<uint32_t, 2, kFlat>;
    case 3: return (const void*)densify_kernel<uint32_t, 3, kFlat>;
    case 4: return (const void*)densify_kernel<uint32_t, 4, kFlat>;
    default: return (const void*)densify_kernel<uint32_t, 5, kFlat>;
  }
}

const void* densify_fn(bool wide, int logn, bool flat) {
  return flat ? densify_fn_walk<true>(wide, logn) : densify_fn_walk<false>(wide, logn);
}

// Densification workspace: [status] then the bin starts (the sparse
// layout's first region, with no partitions).
size_t densify_workspace_bytes(int n, int64_t dense_size) {
  const Geometry g = geometry(n, dense_size, 0, -1);
  return sparse_layout(n, g.bins, 1).cnt;  // status + starts
}

zr_status densify_launch(const int32_t* const* idx, const int64_t* nnz, int n, int64_t dense_size,
                         int64_t* d_union_counts, void* ws, cudaStream_t stream) {
  Lists lists;
  int64_t max_nnz = 0, total_nnz = 0;
  for (int r = 0; r < ZR_MAX_RANKS; ++r) {
    const bool live = r < n && nnz[r] > 0;
    lists.idx[r] = live ? idx[r] : nullptr;
    lists.val[r] = nullptr;
    lists.nnz[r] = r < n ? nnz[r] : 0;
    if (r < n) {
      max_nnz = nnz[r] > max_nnz ? nnz[r] : max_nnz;
      total_nnz += nnz[r];
    }
  }
  int logn = 0;
  while ((1 << logn) < n) ++logn;
  const Geometry g = densify_geometry(n, dense_size, total_nnz);
  const SparseLayout L = sparse_layout(n, g.bins, 1);
  unsigned char* w = static_cast<unsigned char*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  int32_t* starts = reinterpret_cast<int32_t*>(w + L.starts);
  const int bins = (int)g.bins;
  if (cudaMemsetAsync(w, 0, L.starts, stream) != cudaSuccess) return ZR_ERR_CUDA;
  if (cudaMemsetAsync(d_union_counts, 0, (size_t)(logn + 1) * 8, stream) != cudaSuccess)
    return ZR_ERR_CUDA;
  {
    const int64_t groups = max_nnz / 4 + 1;
    int64_t gx = (groups + 256 * kStartsUnroll - 1) / (256 * kStartsUnroll);
    const int64_t cap = ((int64_t)sm_count() * 8 + n - 1) / n;
    if (gx > cap) gx = cap;
    if (gx < 1) gx = 1;
    bin_starts_kernel<<<dim3((unsigned)gx, (unsigned)n), 256, 0, stream>>>(
        lists, (int)dense_size, g.log_w, bins, starts, status);
  }
  const bool wide = n > 32;
  const size_t per_key = (wide ? 8 : 4) + 2;  // mask + member list entry
  const size_t smem = (size_t)kDensWarps * ((size_t)1 << g.log_w) * per_key;
  // lists with few entries per bin on average take the flattened walk
  const bool flat = total_nnz < kMaskMinPerBin * g.bins;
  const void* fn = densify_fn(wide, logn, flat);
  static std::atomic<bool> attr_set[64];
  static std::mutex attr_lock;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ZR_ERR_CUDA;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> guard(attr_lock);
    for (int fl = 0; fl < 2; ++fl)
      for (int lg = 0; lg <= 5; ++lg)
        for (int wd = 0; wd < 2; ++wd)
          if (cudaFuncSetAttribute(densify_fn(wd == 1, lg, fl == 1),
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)((size_t)kDensWarps * 4096 * (wd ? 10 : 6))) != cudaSuccess)
            return ZR_ERR_CUDA;
    attr_set[dev].store(true, std::memory_order_release);
  }
  const int64_t units = (g.bins + kDensWarps - 1) / kDensWarps;
  const unsigned grid = (unsigned)grid_for(units, per_sm(fn, kDensWarps * 32, smem));
  int log_w = g.log_w;
  unsigned long long* counts = reinterpret_cast<unsigned long long*>(d_union_counts);
  void* args[] = {(void*)&lists, (void*)&n,         (void*)&log_w,  (void*)&bins,
                  (void*)&starts, (void*)&total_nnz, (void*)&counts, (void*)&status};
  if (cudaLaunchKernel(fn, dim3(grid), dim3(kDensWarps * 32), args, smem, stream) != cudaSuccess)
    return ZR_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
}

}  // namespace zr
