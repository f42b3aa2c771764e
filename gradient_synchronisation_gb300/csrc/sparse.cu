// Sparse (COO) gradient aggregation and the h0 partition.
//
// What is computed (Zen page, section 2.1 "COO", Problem 1, section 3.2
// Technique #3 and Algorithm 1's first-level hash): the union of N sorted
// index lists, each union index carrying the rank-ordered sum of the values
// that hold it, split into n_parts partitions by the consistent hash h0 and
// written partition-major, ascending index inside a partition.
//
// GB300 design.  The key range [0, M) is cut into bins of W keys (W = 32768
// for up to 8 ranks, halving as the rank count doubles so that the per-rank
// bitmaps of one bin stay at 32 KB of shared memory).  Work inside a bin is
// proportional to its entries, not to W:
//   1. sample:  every 64th index of every list gives, for each rank and bin,
//      a position at most 63 entries before the bin's first entry (one
//      32-byte sector in eight of the index bytes is read).
//   2. count:   per bin, OR the keys of every rank into a W-bit union bitmap
//      in shared memory (checking that each list is strictly ascending and
//      in range), count the union members per partition, and turn the
//      (bin, partition) counts into output positions with a decoupled
//      look-back across bins taken in ticket order; the CTA that finishes
//      the last bin writes the partition offsets.  Every wait is bounded.
//   3. write:   per bin, build one bitmap per rank and its per-word prefix
//      counts, then walk the union members in ascending key order, a warp
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
constexpr int kMaxBinWords = 1024;       // W <= 32768 keys
constexpr int kRankWordsBudget = 8192;   // N * W/32 per-rank bitmap words per bin
constexpr int kPartTile = 4096;          // zr_partition: entries per tile
constexpr int kPartThreads = 512;
constexpr long long kSpinLimit = 1ll << 24;  // bounded look-back waits (about a second)

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

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(int32_t* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
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

// ------------------------------------------------------------ look-back
// Block-wide: publish the per-partition counts of unit u and compute the
// exclusive prefix over units 0..u-1 (decoupled look-back: units are taken in
// ticket order, so every predecessor belongs to a running or finished CTA).
// On return run[p] holds the exclusive prefix; excl[u][p] and incl[u][p] are
// written.  A wait longer than kSpinLimit polls records ZR_ERR_TIMEOUT and
// stops looking back (the result is then unspecified, but the kernel ends).
__device__ void lookback(int64_t u, const int32_t* cnt, int parts, int32_t* flags, int32_t* agg,
                         long long* incl, long long* excl, long long* run, int* s_flag,
                         int32_t* status) {
  const int tid = threadIdx.x;
  for (int p = tid; p < parts; p += blockDim.x) {
    __stcg(agg + u * parts + p, cnt[p]);
    run[p] = 0;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) st_release(flags + u, 1);
  int64_t pred = u - 1;
  while (pred >= 0) {
    if (tid == 0) {
      int f;
      long long spins = 0;
      while ((f = ld_acquire(flags + pred)) == 0) {
        if (++spins > kSpinLimit) {
          flag(status, ZR_ERR_TIMEOUT);
          f = 3;
          break;
        }
        __nanosleep(64);
      }
      *s_flag = f;
    }
    __syncthreads();
    const int f = *s_flag;
    if (f == 3) break;
    for (int p = tid; p < parts; p += blockDim.x)
      run[p] += (f == 2) ? __ldcg(incl + pred * parts + p) : (long long)__ldcg(agg + pred * parts + p);
    __syncthreads();
    if (f == 2) break;
    --pred;
  }
  __syncthreads();
  for (int p = tid; p < parts; p += blockDim.x) {
    __stcg(excl + u * parts + p, run[p]);
    __stcg(incl + u * parts + p, run[p] + cnt[p]);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) st_release(flags + u, 2);
}

// The CTA that finished the last unit turns its inclusive prefix (the
// per-partition totals) into partition offsets.
__device__ void write_offsets(const long long* run, const int32_t* cnt, int parts,
                              long long* offs, int64_t* d_offsets, int64_t* d_total) {
  if (threadIdx.x == 0) {
    long long acc = 0;
    for (int p = 0; p < parts; ++p) {
      offs[p] = acc;
      if (d_offsets) d_offsets[p] = acc;
      acc += run[p] + cnt[p];
    }
    offs[parts] = acc;
    if (d_offsets) d_offsets[parts] = acc;
    if (d_total) *d_total = acc;
  }
}

// ------------------------------------------------------------ layout
struct Geometry {
  int log_w;   // bin width W = 2^log_w keys
  int words;   // W / 32
  int64_t bins;
};

Geometry geometry(int n, int64_t dense_size) {
  int np2 = 1;
  while (np2 < n) np2 <<= 1;
  int words = kRankWordsBudget / np2;
  if (words > kMaxBinWords) words = kMaxBinWords;
  int log_w = 5;
  while ((1 << (log_w - 5)) < words) ++log_w;
  Geometry g;
  g.log_w = log_w;
  g.words = words;
  g.bins = (dense_size + (1ll << log_w) - 1) >> log_w;
  return g;
}

// [status, ticket | flags[B]] are contiguous so one memset clears them.
struct SparseLayout {
  size_t flags, offs, coarse, agg, incl, excl, total;
};

SparseLayout sparse_layout(int n, int64_t bins, int parts) {
  SparseLayout L;
  L.flags = 256;
  L.offs = L.flags + align256((size_t)bins * 4);
  L.coarse = L.offs + align256((size_t)(parts + 1) * 8);
  L.agg = L.coarse + align256((size_t)n * (size_t)(bins + 1) * 4);
  L.incl = L.agg + align256((size_t)bins * parts * 4);
  L.excl = L.incl + align256((size_t)bins * parts * 8);
  L.total = L.excl + align256((size_t)bins * parts * 8);
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

// ------------------------------------------------------------ 2. count
__global__ void __launch_bounds__(kThreads)
union_count_kernel(const __grid_constant__ Lists lists, int n, int64_t dense_size, int log_w,
                   int words, int64_t bins, const int32_t* coarse, H0 h, int parts,
                   int32_t* flags, int32_t* agg, long long* incl, long long* excl, long long* offs,
                   int64_t* d_offsets, int64_t* d_total, uint32_t* ticket, int32_t* status) {
  __shared__ uint32_t ubits[kMaxBinWords];
  __shared__ int32_t cnt[ZR_MAX_PARTS];
  __shared__ long long run[ZR_MAX_PARTS];
  __shared__ int64_t lo_s[ZR_MAX_RANKS], hi_s[ZR_MAX_RANKS];
  __shared__ int64_t s_bin;
  __shared__ int s_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t W = 1ll << log_w;
  const H0 hash = h;
  for (;;) {
    if (tid == 0) s_bin = atomicAdd(ticket, 1u);
    __syncthreads();
    const int64_t b = s_bin;
    if (b >= bins) break;
    const int64_t base = b << log_w;
    for (int w = tid; w < words; w += kThreads) ubits[w] = 0;
    for (int p = tid; p < parts; p += kThreads) cnt[p] = 0;
    for (int r = tid; r < n; r += kThreads) bin_range(coarse, bins, r, b, lists.nnz[r], lo_s[r], hi_s[r]);
    __syncthreads();
    for (int r = 0; r < n; ++r) {
      const int32_t* idx = lists.idx[r];
      for (int64_t i = lo_s[r] + tid; i < hi_s[r]; i += kThreads) {
        const int64_t key = idx[i];
        bool ok = key >= 0 && key < dense_size;
        if (i > 0 && key <= (int64_t)idx[i - 1]) ok = false;
        if (!ok) flag(status, ZR_ERR_INPUT_UNSORTED);
        const int64_t slot = key - base;
        if (slot >= 0 && slot < W) atomicOr(&ubits[slot >> 5], 1u << (slot & 31));
      }
    }
    __syncthreads();
    // Count the union members per partition, a warp per 32-word window;
    // lanes are mapped to members by a warp-level load-balancing search.
    for (int c = warp * 32; c < words; c += kWarps * 32) {
      const uint32_t wbits = ubits[c + lane];
      const int cntl = __popc(wbits);
      const int incl_l = warp_incl_scan(cntl);
      const int total = __shfl_sync(0xffffffffu, incl_l, 31);
      for (int q = 0; q < total; q += 32) {
        const int j = q + lane;
        const bool live = j < total;
        const int o = owner_lane(incl_l, j);
        const uint32_t ow = __shfl_sync(0xffffffffu, wbits, o);
        const int oex = __shfl_sync(0xffffffffu, incl_l - cntl, o);
        const int bit = live ? select_bit(ow, j - oex) : 0;
        const uint32_t key = (uint32_t)(base + (c + o) * 32 + bit);
        const int p = live ? (parts > 1 ? (int)hash(key) : 0) : parts;
        const unsigned peers = __match_any_sync(0xffffffffu, p);
        if (live && (peers & lanemask_lt()) == 0) atomicAdd(&cnt[p], __popc(peers));
      }
    }
    __syncthreads();
    lookback(b, cnt, parts, flags, agg, incl, excl, run, &s_flag, status);
    if (b == bins - 1) write_offsets(run, cnt, parts, offs, d_offsets, d_total);
    __syncthreads();
  }
}

// ------------------------------------------------------------ 3. write
struct WriteSmem {
  uint32_t* rbits;     // [n][words]
  uint16_t* rpre;      // [n][words]
  uint32_t* ubits;     // [words]
  long long* wbase;    // [kWarps][parts]
  long long* outbase;  // [parts]
  int64_t* seg0;       // [n]
  int64_t* lo;         // [n]
  int64_t* hi;         // [n]
  int32_t* below;      // [n]
};

__host__ __device__ inline size_t write_smem_bytes(int n, int words, int parts) {
  size_t b = 0;
  b += (size_t)n * words * 4;
  b += ((size_t)n * words * 2 + 255) & ~(size_t)255;
  b += (size_t)words * 4;
  b += (size_t)kWarps * parts * 8;
  b += (size_t)parts * 8;
  b += (size_t)n * 8 * 3;
  b += (size_t)n * 4;
  return b;
}

__device__ WriteSmem carve(unsigned char* s, int n, int words, int parts) {
  WriteSmem m;
  size_t o = 0;
  m.rbits = reinterpret_cast<uint32_t*>(s + o); o += (size_t)n * words * 4;
  m.rpre = reinterpret_cast<uint16_t*>(s + o); o += ((size_t)n * words * 2 + 255) & ~(size_t)255;
  m.ubits = reinterpret_cast<uint32_t*>(s + o); o += (size_t)words * 4;
  m.wbase = reinterpret_cast<long long*>(s + o); o += (size_t)kWarps * parts * 8;
  m.outbase = reinterpret_cast<long long*>(s + o); o += (size_t)parts * 8;
  m.seg0 = reinterpret_cast<int64_t*>(s + o); o += (size_t)n * 8;
  m.lo = reinterpret_cast<int64_t*>(s + o); o += (size_t)n * 8;
  m.hi = reinterpret_cast<int64_t*>(s + o); o += (size_t)n * 8;
  m.below = reinterpret_cast<int32_t*>(s + o);
  return m;
}

__global__ void __launch_bounds__(kThreads)
union_write_kernel(const __grid_constant__ Lists lists, int n, int log_w, int words, int64_t bins,
                   const int32_t* coarse, H0 h, int parts, int average, const long long* offs,
                   const long long* excl, int32_t* out_idx, float* out_val, int64_t out_cap,
                   int32_t* status) {
  extern __shared__ __align__(16) unsigned char smem[];
  const WriteSmem S = carve(smem, n, words, parts);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t W = 1ll << log_w;
  const int per_warp = words / kWarps;  // >= 8
  const int win = per_warp < 32 ? per_warp : 32;
  const float fn = (float)n;
  const H0 hash = h;

  for (int64_t b = blockIdx.x; b < bins; b += gridDim.x) {
    const int64_t base = b << log_w;
    for (int i = tid; i < n * words; i += kThreads) S.rbits[i] = 0;
    for (int r = tid; r < n; r += kThreads) {
      bin_range(coarse, bins, r, b, lists.nnz[r], S.lo[r], S.hi[r]);
      S.below[r] = 0;
    }
    for (int i = tid; i < kWarps * parts; i += kThreads) S.wbase[i] = 0;
    for (int p = tid; p < parts; p += kThreads)
      S.outbase[p] = __ldcg(offs + p) + __ldcg(excl + b * parts + p);
    __syncthreads();
    // Per-rank bitmaps of the bin; entries before the bin are counted to
    // find where the bin starts in each list.
    for (int r = 0; r < n; ++r) {
      const int32_t* idx = lists.idx[r];
      uint32_t* rb = S.rbits + (size_t)r * words;
      int below = 0;
      for (int64_t i = S.lo[r] + tid; i < S.hi[r]; i += kThreads) {
        const int64_t slot = (int64_t)idx[i] - base;
        if (slot >= 0 && slot < W) atomicOr(&rb[slot >> 5], 1u << (slot & 31));
        else if (slot < 0) ++below;
      }
      if (below) atomicAdd(&S.below[r], below);
    }
    __syncthreads();
    for (int r = tid; r < n; r += kThreads) S.seg0[r] = S.lo[r] + S.below[r];
    // Per-rank exclusive prefix of set bits per word: one warp per rank.
    for (int r = warp; r < n; r += kWarps) {
      const uint32_t* rb = S.rbits + (size_t)r * words;
      uint16_t* rp = S.rpre + (size_t)r * words;
      const int wpl = words / 32;
      int s = 0;
      for (int q = 0; q < wpl; ++q) s += __popc(rb[lane * wpl + q]);
      int run = warp_incl_scan(s) - s;
      for (int q = 0; q < wpl; ++q) {
        rp[lane * wpl + q] = (uint16_t)run;
        run += __popc(rb[lane * wpl + q]);
      }
    }
    for (int w = tid; w < words; w += kThreads) {
      uint32_t u = 0;
      for (int r = 0; r < n; ++r) u |= S.rbits[(size_t)r * words + w];
      S.ubits[w] = u;
    }
    __syncthreads();

    // Two passes over the warp's words, members in ascending key order:
    // pass 0 counts members per partition, pass 1 places and writes them.
    for (int pass = 0; pass < 2; ++pass) {
      for (int c = warp * per_warp; c < (warp + 1) * per_warp; c += win) {
        const uint32_t wbits = lane < win ? S.ubits[c + lane] : 0u;
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
          const bool leader = live && (peers & lanemask_lt()) == 0;
          if (pass == 1 && live) {
            const long long dst = S.wbase[warp * parts + p] + __popc(peers & lanemask_lt());
            const uint32_t m = 1u << bit;
            float acc = -0.0f;
            for (int r = 0; r < n; ++r) {
              const uint32_t rb = S.rbits[(size_t)r * words + wd];
              if (rb & m) {
                const int64_t pos =
                    S.seg0[r] + S.rpre[(size_t)r * words + wd] + __popc(rb & (m - 1));
                acc = __fadd_rn(acc, lists.val[r][pos]);
              }
            }
            if (average) acc = __fdiv_rn(acc, fn);
            if (dst >= 0 && dst < out_cap) {
              out_idx[dst] = (int32_t)key;
              out_val[dst] = acc;
            } else {
              flag(status, ZR_ERR_INPUT_UNSORTED);
            }
          }
          __syncwarp();
          if (leader) S.wbase[warp * parts + p] += __popc(peers);
          __syncwarp();
        }
      }
      __syncthreads();
      if (pass == 0) {
        // Exclusive scan over warps per partition, from the bin's base.
        for (int p = tid; p < parts; p += kThreads) {
          long long run = S.outbase[p];
          for (int w = 0; w < kWarps; ++w) {
            const long long t = S.wbase[w * parts + p];
            S.wbase[w * parts + p] = run;
            run += t;
          }
        }
        __syncthreads();
      }
    }
  }
}

// ------------------------------------------------------------ partition
struct PartLayout {
  size_t flags, offs, agg, incl, excl, total;
};

PartLayout part_layout(int64_t tiles, int parts) {
  PartLayout L;
  L.flags = 256;
  L.offs = L.flags + align256((size_t)tiles * 4);
  L.agg = L.offs + align256((size_t)(parts + 1) * 8);
  L.incl = L.agg + align256((size_t)tiles * parts * 4);
  L.excl = L.incl + align256((size_t)tiles * parts * 8);
  L.total = L.excl + align256((size_t)tiles * parts * 8);
  return L;
}

__global__ void __launch_bounds__(kPartThreads)
part_count_kernel(const int32_t* idx, int64_t nnz, int64_t tiles, H0 h, int parts,
                  int32_t* flags, int32_t* agg, long long* incl, long long* excl, long long* offs,
                  int64_t* d_offsets, uint32_t* ticket, int32_t* status) {
  __shared__ int32_t cnt[ZR_MAX_PARTS];
  __shared__ long long run[ZR_MAX_PARTS];
  __shared__ int64_t s_tile;
  __shared__ int s_flag;
  const int tid = threadIdx.x;
  const H0 hash = h;
  for (;;) {
    if (tid == 0) s_tile = atomicAdd(ticket, 1u);
    for (int q = tid; q < parts; q += kPartThreads) cnt[q] = 0;
    __syncthreads();
    const int64_t t = s_tile;
    if (t >= tiles) break;
    const int64_t lo = t * kPartTile, hi = min(lo + kPartTile, nnz);
    for (int64_t i = lo + tid; i < lo + kPartTile; i += kPartThreads) {
      const bool live = i < hi;
      const int p = live ? (int)hash((uint32_t)idx[i]) : parts;
      const unsigned peers = __match_any_sync(0xffffffffu, p);
      if (live && (peers & lanemask_lt()) == 0) atomicAdd(&cnt[p], __popc(peers));
    }
    __syncthreads();
    lookback(t, cnt, parts, flags, agg, incl, excl, run, &s_flag, status);
    if (t == tiles - 1) write_offsets(run, cnt, parts, offs, d_offsets, nullptr);
    __syncthreads();
  }
}

// Each warp owns kPartTile / warps consecutive entries of the tile and walks
// them 32 at a time, so the entries of one partition leave in input order.
__global__ void __launch_bounds__(kPartThreads)
part_write_kernel(const int32_t* idx, const float* val, int64_t nnz, int64_t tiles, H0 h,
                  int parts, const long long* offs, const long long* excl, int32_t* out_idx,
                  float* out_val) {
  extern __shared__ __align__(16) unsigned char smem[];
  long long* wbase = reinterpret_cast<long long*>(smem);  // warps * parts
  constexpr int kPW = kPartThreads / 32;
  constexpr int kPerWarp = kPartTile / kPW;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const H0 hash = h;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    for (int q = threadIdx.x; q < kPW * parts; q += kPartThreads) wbase[q] = 0;
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
      long long run = __ldcg(offs + q) + __ldcg(excl + t * parts + q);
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
// write kernel, done once per device).
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
    size_t biggest = 0;
    for (int n = 1; n <= ZR_MAX_RANKS; ++n) {
      const size_t s = write_smem_bytes(n, geometry(n, 1).words, ZR_MAX_PARTS);
      if (s > biggest) biggest = s;
    }
    if (cudaFuncSetAttribute(union_write_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)biggest) != cudaSuccess)
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
  uint32_t* ticket = reinterpret_cast<uint32_t*>(w + 4);
  int32_t* flags = reinterpret_cast<int32_t*>(w + L.flags);
  long long* offs = reinterpret_cast<long long*>(w + L.offs);
  int32_t* coarse = reinterpret_cast<int32_t*>(w + L.coarse);
  int32_t* agg = reinterpret_cast<int32_t*>(w + L.agg);
  long long* incl = reinterpret_cast<long long*>(w + L.incl);
  long long* excl = reinterpret_cast<long long*>(w + L.excl);

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
  // status, ticket and the look-back flags start at zero
  if (cudaMemsetAsync(w, 0, L.offs, stream) != cudaSuccess) return ZR_ERR_CUDA;
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
      lists, n, dense_size, g.log_w, g.words, g.bins, coarse, h, parts, flags, agg, incl, excl,
      offs, n_parts > 0 ? d_offsets : nullptr, d_out_nnz, ticket, status);
  {
    const size_t smem = write_smem_bytes(n, g.words, parts);
    const int o = per_sm((const void*)union_write_kernel, kThreads, smem);
    union_write_kernel<<<(unsigned)grid_for(g.bins, o), kThreads, smem, stream>>>(
        lists, n, g.log_w, g.words, g.bins, coarse, h, parts, average, offs, excl, out_idx,
        out_val, out_cap, status);
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
  int32_t* status = reinterpret_cast<int32_t*>(w);
  uint32_t* ticket = reinterpret_cast<uint32_t*>(w + 4);
  int32_t* flags = reinterpret_cast<int32_t*>(w + L.flags);
  long long* offs = reinterpret_cast<long long*>(w + L.offs);
  int32_t* agg = reinterpret_cast<int32_t*>(w + L.agg);
  long long* incl = reinterpret_cast<long long*>(w + L.incl);
  long long* excl = reinterpret_cast<long long*>(w + L.excl);
  const H0 h = make_h0(part_seed, (uint32_t)n_parts);
  if (tiles == 0) {
    if (cudaMemsetAsync(d_offsets, 0, (size_t)(n_parts + 1) * 8, stream) != cudaSuccess)
      return ZR_ERR_CUDA;
    return ZR_OK;
  }
  DeviceInfo* dinfo = device_info();
  if (!dinfo) return ZR_ERR_CUDA;
  if (cudaMemsetAsync(w, 0, L.offs, stream) != cudaSuccess) return ZR_ERR_CUDA;
  part_count_kernel<<<(unsigned)grid_for(tiles, dinfo->part_count_per_sm), kPartThreads, 0,
                      stream>>>(idx, nnz, tiles, h, n_parts, flags, agg, incl, excl, offs,
                                d_offsets, ticket, status);
  const size_t smem = (size_t)(kPartThreads / 32) * n_parts * sizeof(long long);
  part_write_kernel<<<(unsigned)grid_for(tiles, 4), kPartThreads, smem, stream>>>(
      idx, val, nnz, tiles, h, n_parts, offs, excl, out_idx, out_val);
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
}

}  // namespace zr
