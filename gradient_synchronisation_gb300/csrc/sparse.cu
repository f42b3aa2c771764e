// Sparse (COO) gradient aggregation and the h0 partition.
//
// What is computed (Zen page, section 2.1 "COO", Problem 1, section 3.2
// Technique #3 and Algorithm 1's first-level hash): the union of N sorted
// index lists, each union index carrying the rank-ordered sum of the values
// that hold it, split into n_parts partitions by the consistent hash h0 and
// written partition-major, ascending index inside a partition.
//
// GB300 design.  The key range [0, M) is cut into bins of W keys (W = 16384
// for up to 8 ranks, halving as the rank count doubles so that the per-rank
// bitmaps of one bin stay at 16 KB of shared memory).  Work inside a bin is
// proportional to its entries, not to W:
//   1. sample:  every 64th index of every list gives, for each rank and bin,
//      a position at most 63 entries before the bin's first entry (one
//      32-byte sector in eight of the index bytes is read).
//   2. count:   per bin, OR the keys of every rank into a W-bit union bitmap
//      in shared memory (checking that each list is strictly ascending and
//      in range) and count the union members per partition; per-bin counts
//      plus atomically summed segment and partition totals give every bin
//      its output positions without any CTA waiting for another.
//   3. write:   per bin, build one bitmap per rank and its per-word prefix
//      counts plus a holder mask per key, stage the bin's values in shared
//      memory (16-byte loads over all ranks' ranges at once), then walk the union members in ascending key order, a warp
//      at a time over 32-word windows (a warp-level load-balancing search
//      maps lanes to members).  Each member gathers its holders' values in
//      ascending rank order straight from the input lists (the position of a
//      key in rank r's list is the bin's start plus a bitmap prefix count)
//      and folds them left from -0.0 (-0.0 + x == x for every x, so this is
//      exactly "start from the first holder's value").  A warp-level stable
//      multi-split on the partition id places each member.
//
// Every index taken from the inputs is range-checked before it addresses
// shared memory, segment bounds read from the workspace are clamped to the
// list lengths, and every output position is checked against the output
// capacity, so malformed input can only produce wrong output and a status
// word, never an out-of-bounds access.

#include <cuda_runtime.h>
#include <stdint.h>

#include "zr.h"
#include "zr_device.cuh"
#include "zr_internal.h"

namespace zr {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kSample = 64;              // stride of the sampling pass
constexpr int kLogW = 13;                // bin width W = 8192 keys
constexpr int kWords = (1 << kLogW) / 32;  // union bitmap words per bin
constexpr int kStage = 8192;             // entries of one bin staged in shared memory
constexpr int kPartTile = 4096;          // zr_partition: entries per tile
constexpr int kPartThreads = 512;

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

// Position (0-based) of the n-th set bit of x; x must have more than n bits set.
__device__ __forceinline__ int select_bit(uint32_t x, int n) {
  int pos = 0;
  int c = __popc(x & 0xFFFFu);
  if (n >= c) { n -= c; x >>= 16; pos += 16; }
  c = __popc(x & 0xFFu);
  if (n >= c) { n -= c; x >>= 8; pos += 8; }
  c = __popc(x & 0xFu);
  if (n >= c) { n -= c; x >>= 4; pos += 4; }
  c = __popc(x & 0x3u);
  if (n >= c) { n -= c; x >>= 2; pos += 2; }
  if (n >= (int)(x & 1u)) pos += 1;
  return pos;
}

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// Smallest lane whose inclusive prefix exceeds j (the lanes hold a
// non-decreasing prefix); every lane searches for its own j.
__device__ __forceinline__ int owner_lane(int incl, int j) {
  int pos = 0;
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) {
    const int v = __shfl_sync(0xffffffffu, incl, pos + s - 1);
    if (v <= j) pos += s;
  }
  return pos;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// ------------------------------------------------------------ positions
// Output positions come from per-unit (bin or tile) member counts per
// partition, with two order-free sums kept beside them: the totals of every
// segment of kSeg consecutive units and the grand total per partition, both
// accumulated with integer atomics.  The first output position of unit u in
// partition p is then
//   sum_{p' < p} total[p'] + sum_{segments before u's} seg[.][p]
//                          + sum_{units of u's segment before u} cnt[.][p],
// which a CTA assembles with one round of parallel loads; no CTA ever waits
// for another.
constexpr int kSegLog = 6;
constexpr int kSeg = 1 << kSegLog;

__device__ void publish_counts(int64_t u, const int32_t* cnt, int parts, int32_t* cnt_g,
                               unsigned long long* seg_g, unsigned long long* tot_g) {
  for (int p = threadIdx.x; p < parts; p += blockDim.x) {
    const int32_t c = cnt[p];
    __stcg(cnt_g + u * parts + p, c);
    if (c) {
      atomicAdd(seg_g + (u >> kSegLog) * parts + p, (unsigned long long)c);
      atomicAdd(tot_g + p, (unsigned long long)c);
    }
  }
}

// offs[0..parts] = exclusive prefix of the totals (shared memory); block 0
// of the grid also writes it to d_offsets and the grand total to d_total.
__device__ void partition_offsets(const unsigned long long* tot_g, int parts, long long* offs,
                                  int64_t* d_offsets, int64_t* d_total) {
  __syncthreads();
  if (threadIdx.x == 0) {
    long long acc = 0;
    for (int p = 0; p < parts; ++p) {
      offs[p] = acc;
      acc += (long long)__ldcg(tot_g + p);
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

// base[p] = first output position of unit u in partition p (shared memory),
// a warp per partition.  The caller puts a barrier after it.
__device__ void unit_base(int64_t u, int parts, const long long* offs, const int32_t* cnt_g,
                          const unsigned long long* seg_g, long long* base) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, warps = blockDim.x >> 5;
  const int segs = (int)(u >> kSegLog);
  const int64_t first = (int64_t)segs << kSegLog;
  const int rest = (int)(u - first);
  for (int p = warp; p < parts; p += warps) {
    unsigned long long s = 0;
    for (int j = lane; j < segs; j += 32) s += __ldcg(seg_g + (int64_t)j * parts + p);
    for (int j = lane; j < rest; j += 32) s += (unsigned long long)__ldcg(cnt_g + (first + j) * parts + p);
    for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
    if (lane == 0) base[p] = offs[p] + (long long)s;
  }
}

// ------------------------------------------------------------ layout
struct Geometry {
  int log_w;   // bin width W = 2^log_w keys
  int words;   // W / 32
  int64_t bins;
};

// Bins are W = 8192 keys for any rank count: the writer folds a bin into a
// W-float window in shared memory.
Geometry geometry(int, int64_t dense_size) {
  Geometry g;
  g.log_w = kLogW;
  g.words = kWords;
  g.bins = (dense_size + (1ll << kLogW) - 1) >> kLogW;
  return g;
}

// Per-(bin, warp, partition) member counts let the writer place members
// without recounting them; kept when they fit in 16 MB of workspace.
bool keep_warp_counts(int64_t bins, int parts) {
  return (double)bins * kWarps * parts <= (double)(1 << 22);
}

// [status | totals | segment totals] are contiguous so one memset clears them.
struct SparseLayout {
  size_t tot, seg, coarse, cnt, wcnt, total;
};

SparseLayout sparse_layout(int n, int64_t bins, int parts) {
  SparseLayout L;
  const int64_t segs = (bins + kSeg - 1) >> kSegLog;
  L.tot = 256;
  L.seg = L.tot + align256((size_t)parts * 8);
  L.coarse = L.seg + align256((size_t)segs * parts * 8);
  L.cnt = L.coarse + align256((size_t)n * (size_t)(bins + 1) * 4);
  L.wcnt = L.cnt + align256((size_t)bins * parts * 4);
  L.total = L.wcnt + (keep_warp_counts(bins, parts) ? align256((size_t)bins * kWarps * parts * 4) : 0);
  return L;
}

// ------------------------------------------------------------ 1. sample
__device__ __forceinline__ int64_t bin_of(int64_t key, int log_w, int64_t bins) {
  return key < 0 ? -1 : min(key >> log_w, bins);
}

// Grid: x over samples (plus one thread for the end), y = rank.
// coarse[r][b] = position of the first sample whose bin is >= b (nnz if none).
__global__ void sample_kernel(const __grid_constant__ Lists lists, int64_t dense_size, int log_w,
                              int64_t bins, int32_t* coarse, int32_t* status) {
  const int r = blockIdx.y;
  const int64_t nnz = lists.nnz[r];
  const int32_t* idx = lists.idx[r];
  const int64_t samples = (nnz + kSample - 1) / kSample;
  int32_t* row = coarse + (size_t)r * (bins + 1);
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j <= samples;
       j += (int64_t)gridDim.x * blockDim.x) {
    int64_t b_here, at;
    if (j < samples) {
      const int64_t key = idx[j * kSample];
      if (key < 0 || key >= dense_size) flag(status, ZR_ERR_INPUT_UNSORTED);
      if (j > 0 && key <= (int64_t)idx[(j - 1) * kSample]) flag(status, ZR_ERR_INPUT_UNSORTED);
      b_here = bin_of(key, log_w, bins);
      at = j * kSample;
    } else {
      b_here = bins;
      at = nnz;
    }
    const int64_t b_prev = j == 0 ? -1 : bin_of(idx[(j - 1) * kSample], log_w, bins);
    for (int64_t b = b_prev + 1; b <= b_here; ++b) row[b] = (int32_t)at;
  }
}

// Entries of bin b in rank r lie inside [lo, hi).
__device__ __forceinline__ void bin_range(const int32_t* coarse, int64_t bins, int r, int64_t b,
                                          int64_t nnz, int64_t& lo, int64_t& hi) {
  const int32_t* row = coarse + (size_t)r * (bins + 1);
  lo = min(max((int64_t)row[b] - (kSample - 1), (int64_t)0), nnz);
  hi = min(max((int64_t)row[b + 1], lo), nnz);
}

// Walks the union members of the calling warp's words in ascending key
// order, 32 members at a time, and calls f(live, key, word, bit, p, peers)
// with every lane of the warp (peers: lanes of the same partition p; p is
// `parts` for lanes without a member).
template <typename F>
__device__ __forceinline__ void for_members(const uint32_t* ubits, int c0, int c1, int64_t base,
                                            const H0& hash, int parts, F&& f) {
  const int lane = threadIdx.x & 31;
  const int win = (c1 - c0) < 32 ? (c1 - c0) : 32;
  for (int c = c0; c < c1; c += win) {
    const uint32_t wbits = lane < win ? ubits[c + lane] : 0u;
    const int cntl = __popc(wbits);
    const int incl = warp_incl_scan(cntl);
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    for (int q = 0; q < total; q += 32) {
      const int j = q + lane;
      const bool live = j < total;
      const int o = owner_lane(incl, j);
      const uint32_t ow = __shfl_sync(0xffffffffu, wbits, o);
      const int oex = __shfl_sync(0xffffffffu, incl - cntl, o);
      const int bit = live ? select_bit(ow, j - oex) : 0;
      const int wd = c + o;
      const uint32_t key = (uint32_t)(base + wd * 32 + bit);
      const int p = live ? (parts > 1 ? (int)hash(key) : 0) : parts;
      const unsigned peers = __match_any_sync(0xffffffffu, p);
      f(live, key, wd, bit, p, peers);
    }
  }
}

// ------------------------------------------------------------ bin entries
// Where the entries of one bin lie in every rank's list, and how the block
// walks them: each rank's range [lo, hi) is cut into 16-byte chunks (4
// entries; when the list is 16-byte aligned) plus at most 3 + 3 single
// entries at its ends, and the chunks of all ranks are walked as one
// flattened sequence so that many independent loads are in flight.
struct BinRanges {
  int64_t lo[ZR_MAX_RANKS], hi[ZR_MAX_RANKS];
  int64_t vlo[ZR_MAX_RANKS];           // first chunk (in chunks of 4 entries)
  int32_t cpre[ZR_MAX_RANKS + 1];      // prefix of chunk counts
  int32_t spre[ZR_MAX_RANKS + 1];      // prefix of single-entry counts
  int32_t epre[ZR_MAX_RANKS + 1];      // prefix of range lengths (staging offsets)
};

// Two halves, so that a kernel can issue other independent loads between
// them: bin_ranges_load (threads r < n read the sampled bounds) and, after a
// barrier, bin_ranges_finish (thread 0 lays out chunks and singles).
__device__ __forceinline__ void bin_ranges_load(const Lists& lists, int n, const int32_t* coarse,
                                                int64_t bins, int64_t b, BinRanges& R) {
  for (int r = threadIdx.x; r < n; r += blockDim.x) {
    int64_t lo, hi;
    bin_range(coarse, bins, r, b, lists.nnz[r], lo, hi);
    R.lo[r] = lo;
    R.hi[r] = hi;
  }
}

__device__ __forceinline__ void bin_ranges_finish(const Lists& lists, int n, BinRanges& R) {
  if (threadIdx.x == 0) {
    int32_t c = 0, sgl = 0, e = 0;
    for (int r = 0; r < n; ++r) {
      const int64_t lo = R.lo[r], hi = R.hi[r];
      const bool vec = (reinterpret_cast<uintptr_t>(lists.idx[r]) & 15) == 0 &&
                       (reinterpret_cast<uintptr_t>(lists.val[r]) & 15) == 0;
      int64_t vlo = (lo + 3) >> 2, vhi = hi >> 2;
      if (!vec || vlo > vhi) vlo = vhi = (lo + 3) >> 2;
      R.vlo[r] = vlo;
      R.cpre[r] = c;
      R.spre[r] = sgl;
      R.epre[r] = e;
      const int64_t chunks = (vec && vhi > vlo) ? vhi - vlo : 0;
      c += (int32_t)chunks;
      sgl += (int32_t)((hi - lo) - 4 * chunks);
      e += (int32_t)(hi - lo);
    }
    R.cpre[n] = c;
    R.spre[n] = sgl;
    R.epre[n] = e;
  }
}

// Rank owning flattened item k of a prefix array (largest r with pre[r] <= k).
__device__ __forceinline__ int owner_rank(const int32_t* pre, int n, int32_t k) {
  int lo = 0, hi = n;  // pre[lo] <= k < pre[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] <= k) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Single entries of rank r: the head [lo, 4*vlo) and the tail after the
// chunks (or the whole range when the list cannot be read in chunks).
__device__ __forceinline__ int64_t single_pos(const BinRanges& R, int r, int32_t j) {
  const int64_t lo = R.lo[r];
  const int64_t head = min(R.vlo[r] * 4, R.hi[r]) - lo;
  const int64_t chunks = R.cpre[r + 1] - R.cpre[r];
  return j < head ? lo + j : lo + head + 4 * chunks + (j - head);
}

// Calls f(r, i, key, prev, val) for every entry i of every rank's range of
// the bin, with prev = the key at i-1 (or -1 at i = 0).  kVals loads the
// values as well.
template <bool kVals, typename F>
__device__ __forceinline__ void for_entries(const Lists& lists, int n, const BinRanges& R, F&& f) {
  constexpr int kUnroll = 2;
  const int32_t chunks = R.cpre[n];
  for (int32_t k0 = threadIdx.x; k0 < chunks; k0 += blockDim.x * kUnroll) {
    int4 key[kUnroll];
    float4 val[kUnroll];
    int32_t prev[kUnroll];
    int rr[kUnroll];
    int64_t at[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t k = k0 + u * blockDim.x;
      if (k < chunks) {
        const int r = owner_rank(R.cpre, n, k);
        const int64_t c = R.vlo[r] + (k - R.cpre[r]);
        rr[u] = r;
        at[u] = 4 * c;
        key[u] = __ldg(reinterpret_cast<const int4*>(lists.idx[r]) + c);
        prev[u] = at[u] > 0 ? __ldg(lists.idx[r] + at[u] - 1) : -1;
        if (kVals) val[u] = __ldg(reinterpret_cast<const float4*>(lists.val[r]) + c);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int32_t k = k0 + u * blockDim.x;
      if (k < chunks) {
        f(rr[u], at[u] + 0, key[u].x, prev[u], kVals ? val[u].x : 0.0f);
        f(rr[u], at[u] + 1, key[u].y, key[u].x, kVals ? val[u].y : 0.0f);
        f(rr[u], at[u] + 2, key[u].z, key[u].y, kVals ? val[u].z : 0.0f);
        f(rr[u], at[u] + 3, key[u].w, key[u].z, kVals ? val[u].w : 0.0f);
      }
    }
  }
  const int32_t singles = R.spre[n];
  for (int32_t k = threadIdx.x; k < singles; k += blockDim.x) {
    const int r = owner_rank(R.spre, n, k);
    const int64_t i = single_pos(R, r, k - R.spre[r]);
    const int32_t key = __ldg(lists.idx[r] + i);
    const int32_t prev = i > 0 ? __ldg(lists.idx[r] + i - 1) : -1;
    f(r, i, key, prev, kVals ? __ldg(lists.val[r] + i) : 0.0f);
  }
}

// ------------------------------------------------------------ 2. count
__global__ void __launch_bounds__(kThreads)
union_count_kernel(const __grid_constant__ Lists lists, int n, int64_t dense_size, int log_w,
                   int words, int64_t bins, const int32_t* coarse, H0 h, int parts,
                   int32_t* cnt_g, unsigned long long* seg_g, unsigned long long* tot_g,
                   int32_t* wcnt_g, int32_t* status) {
  __shared__ uint32_t ubits[kWords];
  __shared__ int32_t cnt[ZR_MAX_PARTS];
  __shared__ int32_t wcnt[kWarps * ZR_MAX_PARTS];
  __shared__ BinRanges R;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int64_t W = 1ll << log_w;
  const H0 hash = h;
  const int per_warp = words / kWarps;
  for (int64_t b = blockIdx.x; b < bins; b += gridDim.x) {
    for (int w = tid; w < words; w += kThreads) ubits[w] = 0;
    for (int i = tid; i < kWarps * parts; i += kThreads) wcnt[i] = 0;
    const int64_t base = b << log_w;
    bin_ranges_load(lists, n, coarse, bins, b, R);
    __syncthreads();
    bin_ranges_finish(lists, n, R);
    __syncthreads();
    // Union bitmap; every list is checked strictly ascending and in range
    // (the ranges of consecutive bins overlap, so every adjacent pair of
    // every list is seen by some bin).
    bool bad = false;
    for_entries<false>(lists, n, R, [&](int, int64_t i, int32_t key, int32_t prev, float) {
      if (key < 0 || key >= dense_size || (i > 0 && key <= prev)) bad = true;
      const int64_t slot = (int64_t)key - base;
      if (slot >= 0 && slot < W) atomicOr(&ubits[slot >> 5], 1u << (slot & 31));
    });
    if (bad) flag(status, ZR_ERR_INPUT_UNSORTED);
    __syncthreads();
    // Members per (warp, partition) over the warp's words (the same split of
    // words the writer uses); a lane takes one half of a word at a time.
    {
      const int lane = tid & 31;
      for (int hw = lane; hw < 2 * per_warp; hw += 32) {
        const int wd = warp * per_warp + (hw >> 1);
        uint32_t bits = ubits[wd] & ((hw & 1) ? 0xFFFF0000u : 0x0000FFFFu);
        while (bits) {
          const int bit = __ffs(bits) - 1;
          bits &= bits - 1;
          const uint32_t key = (uint32_t)(base + wd * 32 + bit);
          atomicAdd(&wcnt[warp * parts + (parts > 1 ? (int)hash(key) : 0)], 1);
        }
      }
    }
    __syncthreads();
    for (int p = tid; p < parts; p += kThreads) {
      int s = 0;
      for (int w = 0; w < kWarps; ++w) s += wcnt[w * parts + p];
      cnt[p] = s;
    }
    if (wcnt_g)
      for (int i = tid; i < kWarps * parts; i += kThreads) __stcg(wcnt_g + b * kWarps * parts + i, wcnt[i]);
    __syncthreads();
    publish_counts(b, cnt, parts, cnt_g, seg_g, tot_g);
    __syncthreads();
  }
}

// ------------------------------------------------------------ 3. write
// Shared memory of the writer: the bin's window of folded values, its union
// bitmap, its staged entries (rank-major) and the per-warp output bases.
__host__ __device__ inline size_t write_smem_bytes(int parts) {
  return (size_t)kWords * 32 * 4 + (size_t)kWords * 4 + (size_t)kStage * 8 +
         (size_t)kWarps * parts * 8 + (size_t)parts * 8;
}

__global__ void __launch_bounds__(kThreads)
union_write_kernel(const __grid_constant__ Lists lists, int n, int64_t bins, const int32_t* coarse,
                   H0 h, int parts, int average, const int32_t* cnt_g,
                   const unsigned long long* seg_g, const unsigned long long* tot_g,
                   const int32_t* wcnt_g, int32_t* out_idx, float* out_val, int64_t out_cap,
                   int64_t* d_offsets, int64_t* d_total, int32_t* status) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ BinRanges R;
  __shared__ long long offs[ZR_MAX_PARTS + 1];
  float* acc = reinterpret_cast<float*>(smem);                       // [W]
  uint32_t* ubits = reinterpret_cast<uint32_t*>(acc + kWords * 32);  // [words]
  int32_t* skey = reinterpret_cast<int32_t*>(ubits + kWords);        // [kStage]
  float* sval = reinterpret_cast<float*>(skey + kStage);             // [kStage]
  long long* wbase = reinterpret_cast<long long*>(sval + kStage);    // [kWarps][parts]
  long long* ubase = wbase + kWarps * parts;                         // [parts]
  const int tid = threadIdx.x, warp = tid >> 5;
  constexpr int W = 1 << kLogW;
  constexpr int per_warp = kWords / kWarps;
  const float fn = (float)n;
  const H0 hash = h;
  partition_offsets(tot_g, parts, offs, d_offsets, d_total);

  for (int64_t b = blockIdx.x; b < bins; b += gridDim.x) {
    const int64_t base = b << kLogW;
    // Every global load of the prologue is issued before one barrier: the
    // sampled bounds, the position sums and the per-warp member counts.
    for (int i = tid; i < W; i += kThreads) acc[i] = -0.0f;
    for (int i = tid; i < kWords; i += kThreads) ubits[i] = 0;
    bin_ranges_load(lists, n, coarse, bins, b, R);
    unit_base(b, parts, offs, cnt_g, seg_g, ubase);
    for (int i = tid; i < kWarps * parts; i += kThreads)
      wbase[i] = wcnt_g ? (long long)__ldcg(wcnt_g + b * kWarps * parts + i) : 0;
    __syncthreads();
    bin_ranges_finish(lists, n, R);
    for (int p = tid; p < parts; p += kThreads) {  // per-warp bases
      long long run = ubase[p];
      for (int w = 0; w < kWarps; ++w) {
        const long long c = wbase[w * parts + p];
        wbase[w * parts + p] = run;
        if (wcnt_g) run += c;
      }
    }
    __syncthreads();
    const int total = R.epre[n];
    if (total <= kStage) {
      // Stage every rank's range at once (16-byte loads, many in flight).
      for_entries<true>(lists, n, R, [&](int r, int64_t i, int32_t key, int32_t, float v) {
        const int e = R.epre[r] + (int)(i - R.lo[r]);
        skey[e] = key;
        sval[e] = v;
      });
      __syncthreads();
      // Fold rank by rank in ascending rank order: acc starts at -0.0 and
      // -0.0 + x == x, so each member ends as the left fold of its holders.
      for (int r = 0; r < n; ++r) {
        for (int e = R.epre[r] + tid; e < R.epre[r + 1]; e += kThreads) {
          const int64_t slot = (int64_t)skey[e] - base;
          if (slot >= 0 && slot < W) {
            acc[slot] = __fadd_rn(acc[slot], sval[e]);
            atomicOr(&ubits[slot >> 5], 1u << (slot & 31));
          }
        }
        __syncthreads();
      }
    } else {
      // A bin too large to stage: the same fold straight from the lists.
      __syncthreads();
      for (int r = 0; r < n; ++r) {
        const int32_t* idx = lists.idx[r];
        const float* val = lists.val[r];
        for (int64_t i = R.lo[r] + tid; i < R.hi[r]; i += kThreads) {
          const int64_t slot = (int64_t)idx[i] - base;
          if (slot >= 0 && slot < W) {
            acc[slot] = __fadd_rn(acc[slot], val[i]);
            atomicOr(&ubits[slot >> 5], 1u << (slot & 31));
          }
        }
        __syncthreads();
      }
    }
    const int c0 = warp * per_warp, c1 = c0 + per_warp;
    if (!wcnt_g) {
      // Count members per (warp, partition), then an exclusive scan over warps.
      for_members(ubits, c0, c1, base, hash, parts,
                  [&](bool live, uint32_t, int, int, int p, unsigned peers) {
                    if (live && (peers & lanemask_lt()) == 0) wbase[warp * parts + p] += __popc(peers);
                    __syncwarp();
                  });
      __syncthreads();
      for (int p = tid; p < parts; p += kThreads) {
        long long run = ubase[p];
        for (int w = 0; w < kWarps; ++w) {
          const long long t = wbase[w * parts + p] - ubase[p];
          wbase[w * parts + p] = run;
          run += t;
        }
      }
      __syncthreads();
    }
    // Place and write the members in ascending key order per partition.
    for_members(ubits, c0, c1, base, hash, parts,
                [&](bool live, uint32_t key, int wd, int bit, int p, unsigned peers) {
                  if (live) {
                    const long long dst = wbase[warp * parts + p] + __popc(peers & lanemask_lt());
                    float v = acc[wd * 32 + bit];
                    if (average) v = __fdiv_rn(v, fn);
                    if (dst >= 0 && dst < out_cap) {
                      out_idx[dst] = (int32_t)key;
                      out_val[dst] = v;
                    } else {
                      flag(status, ZR_ERR_INPUT_UNSORTED);
                    }
                  }
                  __syncwarp();
                  if (live && (peers & lanemask_lt()) == 0) wbase[warp * parts + p] += __popc(peers);
                  __syncwarp();
                });
    __syncthreads();
  }
}

// ------------------------------------------------------------ partition
// [status | totals | segment totals] are contiguous so one memset clears them.
struct PartLayout {
  size_t tot, seg, cnt, total;
};

PartLayout part_layout(int64_t tiles, int parts) {
  PartLayout L;
  const int64_t segs = (tiles + kSeg - 1) >> kSegLog;
  L.tot = 256;
  L.seg = L.tot + align256((size_t)parts * 8);
  L.cnt = L.seg + align256((size_t)segs * parts * 8);
  L.total = L.cnt + align256((size_t)tiles * parts * 4);
  return L;
}

__global__ void __launch_bounds__(kPartThreads)
part_count_kernel(const int32_t* idx, int64_t nnz, int64_t tiles, H0 h, int parts,
                  int32_t* cnt_g, unsigned long long* seg_g, unsigned long long* tot_g) {
  __shared__ int32_t cnt[ZR_MAX_PARTS];
  const int tid = threadIdx.x;
  const H0 hash = h;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    for (int q = tid; q < parts; q += kPartThreads) cnt[q] = 0;
    __syncthreads();
    const int64_t lo = t * kPartTile, hi = min(lo + kPartTile, nnz);
    for (int64_t i = lo + tid; i < lo + kPartTile; i += kPartThreads) {
      const bool live = i < hi;
      const int p = live ? (int)hash((uint32_t)idx[i]) : parts;
      const unsigned peers = __match_any_sync(0xffffffffu, p);
      if (live && (peers & lanemask_lt()) == 0) atomicAdd(&cnt[p], __popc(peers));
    }
    __syncthreads();
    publish_counts(t, cnt, parts, cnt_g, seg_g, tot_g);
    __syncthreads();
  }
}

// Each warp owns kPartTile / warps consecutive entries of the tile and walks
// them 32 at a time, so the entries of one partition leave in input order.
__global__ void __launch_bounds__(kPartThreads)
part_write_kernel(const int32_t* idx, const float* val, int64_t nnz, int64_t tiles, H0 h,
                  int parts, const int32_t* cnt_g, const unsigned long long* seg_g,
                  const unsigned long long* tot_g, int32_t* out_idx, float* out_val,
                  int64_t* d_offsets) {
  extern __shared__ __align__(16) unsigned char smem[];
  long long* wbase = reinterpret_cast<long long*>(smem);  // warps * parts
  __shared__ long long offs[ZR_MAX_PARTS + 1];
  __shared__ long long ubase[ZR_MAX_PARTS];
  constexpr int kPW = kPartThreads / 32;
  constexpr int kPerWarp = kPartTile / kPW;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const H0 hash = h;
  partition_offsets(tot_g, parts, offs, d_offsets, nullptr);
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    for (int q = threadIdx.x; q < kPW * parts; q += kPartThreads) wbase[q] = 0;
    unit_base(t, parts, offs, cnt_g, seg_g, ubase);
    __syncthreads();
    const int64_t lo = t * kPartTile + (int64_t)warp * kPerWarp;
    const int64_t hi = min(t * kPartTile + kPartTile, nnz);
    for (int j = 0; j < kPerWarp; j += 32) {
      const int64_t i = lo + j + lane;
      const bool live = i < hi;
      const int p = live ? (int)hash((uint32_t)idx[i]) : parts;
      const unsigned peers = __match_any_sync(0xffffffffu, p);
      if (live && (peers & lanemask_lt()) == 0) wbase[warp * parts + p] += __popc(peers);
      __syncwarp();
    }
    __syncthreads();
    for (int q = threadIdx.x; q < parts; q += kPartThreads) {
      long long run = ubase[q];
      for (int w = 0; w < kPW; ++w) {
        const long long c = wbase[w * parts + q];
        wbase[w * parts + q] = run;
        run += c;
      }
    }
    __syncthreads();
    for (int j = 0; j < kPerWarp; j += 32) {
      const int64_t i = lo + j + lane;
      const bool live = i < hi;
      const int32_t key = live ? idx[i] : 0;
      const int p = live ? (int)hash((uint32_t)key) : parts;
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

// Per-device cached occupancy (and the dynamic shared-memory opt-in of the
// write kernels, done once per device).
struct DeviceInfo {
  int ready = 0;
  int count_per_sm = 1;
  int part_count_per_sm = 1;
};

DeviceInfo* device_info() {
  static DeviceInfo info[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  DeviceInfo& d = info[dev];
  if (!d.ready) {
    if (cudaFuncSetAttribute(union_write_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)write_smem_bytes(ZR_MAX_PARTS)) != cudaSuccess)
      return nullptr;
    d.count_per_sm = per_sm((const void*)union_count_kernel, kThreads, 0);
    d.part_count_per_sm = per_sm((const void*)part_count_kernel, kPartThreads, 0);
    d.ready = 1;
  }
  return &d;
}

}  // namespace

size_t sparse_workspace_bytes(int n, int64_t dense_size, int n_parts) {
  const Geometry g = geometry(n, dense_size);
  return sparse_layout(n, g.bins, n_parts > 0 ? n_parts : 1).total;
}

zr_status sparse_launch(const int32_t* const* idx, const float* const* val, const int64_t* nnz,
                        int n, int64_t dense_size, int n_parts, uint64_t part_seed, int average,
                        int32_t* out_idx, float* out_val, int64_t out_cap, int64_t* d_out_nnz,
                        int64_t* d_offsets, void* ws, cudaStream_t stream) {
  const Geometry g = geometry(n, dense_size);
  const int parts = n_parts > 0 ? n_parts : 1;
  const SparseLayout L = sparse_layout(n, g.bins, parts);
  unsigned char* w = static_cast<unsigned char*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  unsigned long long* tot = reinterpret_cast<unsigned long long*>(w + L.tot);
  unsigned long long* seg = reinterpret_cast<unsigned long long*>(w + L.seg);
  int32_t* coarse = reinterpret_cast<int32_t*>(w + L.coarse);
  int32_t* cnt = reinterpret_cast<int32_t*>(w + L.cnt);
  int32_t* wcnt = keep_warp_counts(g.bins, parts) ? reinterpret_cast<int32_t*>(w + L.wcnt) : nullptr;

  Lists lists;
  int64_t max_nnz = 0;
  for (int r = 0; r < ZR_MAX_RANKS; ++r) {
    const bool live = r < n && nnz[r] > 0;
    lists.idx[r] = live ? idx[r] : nullptr;
    lists.val[r] = live ? val[r] : nullptr;
    lists.nnz[r] = r < n ? nnz[r] : 0;
    if (r < n && nnz[r] > max_nnz) max_nnz = nnz[r];
  }
  const H0 h = make_h0(part_seed, (uint32_t)parts);
  DeviceInfo* dinfo = device_info();
  if (!dinfo) return ZR_ERR_CUDA;
  // status, partition totals and segment totals start at zero
  if (cudaMemsetAsync(w, 0, L.coarse, stream) != cudaSuccess) return ZR_ERR_CUDA;
  {
    const int64_t samples = (max_nnz + kSample - 1) / kSample;
    int64_t gx = (samples + 1 + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (gx > cap) gx = cap;
    if (gx < 1) gx = 1;
    sample_kernel<<<dim3((unsigned)gx, (unsigned)n), 256, 0, stream>>>(lists, dense_size, g.log_w,
                                                                       g.bins, coarse, status);
  }
  union_count_kernel<<<(unsigned)grid_for(g.bins, dinfo->count_per_sm), kThreads, 0, stream>>>(
      lists, n, dense_size, g.log_w, g.words, g.bins, coarse, h, parts, cnt, seg, tot, wcnt,
      status);
  {
    const size_t smem = write_smem_bytes(parts);
    const int o = per_sm((const void*)union_write_kernel, kThreads, smem);
    union_write_kernel<<<(unsigned)grid_for(g.bins, o), kThreads, smem, stream>>>(
        lists, n, g.bins, coarse, h, parts, average, cnt, seg, tot, wcnt, out_idx, out_val,
        out_cap, n_parts > 0 ? d_offsets : nullptr, d_out_nnz, status);
  }
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
}

size_t partition_workspace_bytes(int64_t nnz, int n_parts) {
  const int64_t tiles = (nnz + kPartTile - 1) / kPartTile;
  return part_layout(tiles, n_parts).total;
}

zr_status partition_launch(const int32_t* idx, const float* val, int64_t nnz, int n_parts,
                           uint64_t part_seed, int32_t* out_idx, float* out_val,
                           int64_t* d_offsets, void* ws, cudaStream_t stream) {
  const int64_t tiles = (nnz + kPartTile - 1) / kPartTile;
  const PartLayout L = part_layout(tiles, n_parts);
  unsigned char* w = static_cast<unsigned char*>(ws);
  unsigned long long* tot = reinterpret_cast<unsigned long long*>(w + L.tot);
  unsigned long long* seg = reinterpret_cast<unsigned long long*>(w + L.seg);
  int32_t* cnt = reinterpret_cast<int32_t*>(w + L.cnt);
  const H0 h = make_h0(part_seed, (uint32_t)n_parts);
  if (tiles == 0) {
    if (cudaMemsetAsync(d_offsets, 0, (size_t)(n_parts + 1) * 8, stream) != cudaSuccess)
      return ZR_ERR_CUDA;
    return ZR_OK;
  }
  DeviceInfo* dinfo = device_info();
  if (!dinfo) return ZR_ERR_CUDA;
  if (cudaMemsetAsync(w, 0, L.cnt, stream) != cudaSuccess) return ZR_ERR_CUDA;
  part_count_kernel<<<(unsigned)grid_for(tiles, dinfo->part_count_per_sm), kPartThreads, 0,
                      stream>>>(idx, nnz, tiles, h, n_parts, cnt, seg, tot);
  const size_t smem = (size_t)(kPartThreads / 32) * n_parts * sizeof(long long);
  part_write_kernel<<<(unsigned)grid_for(tiles, 4), kPartThreads, smem, stream>>>(
      idx, val, nnz, tiles, h, n_parts, cnt, seg, tot, out_idx, out_val, d_offsets);
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
}

}  // namespace zr
