// Zen's hash bitmap: encode a server's nonzero indices as one bit per element
// of its index set, and decode such bitmaps back to indices.
//
// What is computed (Zen page, section 3.3.2 "Hash bitmap", Figure 10 and
// Algorithm 2): with h0, I_p = {x in [0, M) : h0(x) = p}, ascending.  Encode
// sets bit j of partition p's bitmap when I_p[j] is one of the given nonzero
// indices; decode outputs I_p[j] for every set bit j.  Bit j is bit (j mod 32)
// of word floor(j / 32); partition p's words start at word offset
// sum_{q < p} ceil(|I_q| / 32).
//
// GB300 design.  Neither direction reads the index sets.  A directory built
// once per (M, P, seed) replaces them: h0 of every index, bit-sliced
// (ceil(log2 P) bits per index, against 32 for the index sets), and, for
// every range of 2048 consecutive indices, where the range starts inside
// every I_p (4 bytes per partition per range).  A warp takes one range at a
// time, 64 consecutive indices per lane:
//   slices  the lane loads its indices' partitions as NB 64-bit words: word b
//           holds bit b of the partition of each of its 64 indices (the
//           directory build hashes every index once to make them).
//   ranks   for each partition q an AND of the slices gives the lane's
//           indices in q, and its popcount the lane's count; a warp scan of
//           the counts (two partitions per scan, 16 bits each) gives the
//           lane's first position in I_q (directory entry + prefix), and a
//           popcount below an index its rank.  The warp's totals are checked
//           against the directory's counts.
//   encode  the nonzero indices are first marked in an M-bit membership map
//           (it stays in L2); each member sets its bit with a reduction OR
//           into the zeroed bitmaps.
//   decode  a popcount of every (partition, range) segment of the bitmaps and
//           a scan per partition give each segment's first output position;
//           the lane extracts its bits of q's segment (up to 64, three words)
//           and writes the index of every set bit.
// Memory traffic per call: the slices (M NB / 8 bytes), the membership map
// or the bitmaps (M / 8 bytes) and the U indices.  Every index that
// addresses memory is range-checked first; every output position is checked
// against the output capacity.

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "zr.h"
#include "zr_device.cuh"
#include "zr_internal.h"

namespace zr {
namespace {

constexpr int kLaneKeys = 64;                // indices per lane
constexpr int kRangeKeys = 32 * kLaneKeys;   // indices per warp range
constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kScanThreads = 1024;
constexpr int kMaxBits = 8;                  // ZR_MAX_PARTS = 2^8
constexpr int kChunk = 8;                    // partitions per member pass

static_assert(ZR_MAX_PARTS <= (1 << kMaxBits), "partition index fits the slices");
static_assert(kRangeKeys == ZR_HASH_RANGE, "the directory's range is the header's");

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

__device__ __forceinline__ void flag(int32_t* status, int code) { atomicCAS(status, 0, code); }

int64_t ranges_of(int64_t m) { return (m + kRangeKeys - 1) / kRangeKeys; }

int part_bits(int parts) {
  int nb = 0;
  while ((1 << nb) < parts) ++nb;
  return nb;
}

// Row stride of the per-(partition, range) count arrays: R + 1 entries
// rounded up to 4, so that every row starts 16-byte aligned.
int64_t row_stride(int64_t m) { return (ranges_of(m) + 1 + 3) & ~(int64_t)3; }

// Directory: [header 256 B | counts, P rows of row_stride ints | slices,
// u64[R][NB][32]].  The header names what the directory was built for.
constexpr int kDirHeader = 256;
constexpr long long kDirMagic = 0x5a52484449523031ll;  // "ZRHDIR01"
size_t dir_counts_bytes(int64_t m, int parts) { return align256((size_t)parts * row_stride(m) * 4); }

// Workspace: [status | membership map ceil(M/32) words | per (partition,
// range) set-bit counts, P x (R + 1)].
struct HbLayout {
  size_t mem, seg, total;
};

HbLayout hb_layout(int64_t m, int parts) {
  HbLayout L;
  L.mem = 256;
  L.seg = L.mem + align256((size_t)((m + 31) / 32) * 4);
  L.total = L.seg + align256((size_t)parts * (size_t)row_stride(m) * 4);
  return L;
}

struct HbGeom {
  int m;       // dense size M
  int parts;   // P
  int ranges;  // R = ceil(M / 2048)
  int stride;  // row stride of the count arrays
  unsigned long long seed;
  H0 h;
};

// ---------------------------------------------------------------- slices
template <int NB>
struct Slices {
  uint32_t lo[NB > 0 ? NB : 1], hi[NB > 0 ? NB : 1];
  uint64_t valid;  // the lane's indices below M
};

// Hashes the lane's indices x0 .. x0 + 63 (x0 a multiple of 64).
template <int NB>
__device__ __forceinline__ void slice_partitions(const HbGeom& G, int x0, Slices<NB>& S) {
  const long long left = (long long)G.m - x0;
  const int nvalid = left <= 0 ? 0 : (left >= kLaneKeys ? kLaneKeys : (int)left);
  S.valid = nvalid == kLaneKeys ? ~0ull : ((1ull << nvalid) - 1ull);
#pragma unroll
  for (int b = 0; b < (NB > 0 ? NB : 1); ++b) S.lo[b] = S.hi[b] = 0u;
  if (NB == 0 || nvalid == 0) return;
  uint64_t v = G.h.a * (uint64_t)(uint32_t)x0 + G.h.b;
  const uint32_t P = G.h.n_parts;
#pragma unroll
  for (int k = 0; k < kLaneKeys; ++k) {
    const uint32_t p = __umulhi((uint32_t)(v >> 32), P);
    v += G.h.a;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const uint32_t bit = (p >> b) & 1u;
      if (k < 32) S.lo[b] |= bit << k;
      else S.hi[b] |= bit << (k - 32);
    }
  }
}

// The lane's slices of range r from the directory (coalesced: word b of the
// 32 lanes is 256 contiguous bytes).
template <int NB>
__device__ __forceinline__ void load_slices(const HbGeom& G, const uint64_t* sl, int r, int x0,
                                            Slices<NB>& S) {
  const long long left = (long long)G.m - x0;
  const int nvalid = left <= 0 ? 0 : (left >= kLaneKeys ? kLaneKeys : (int)left);
  S.valid = nvalid == kLaneKeys ? ~0ull : ((1ull << nvalid) - 1ull);
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int b = 0; b < (NB > 0 ? NB : 1); ++b) {
    const uint64_t v = NB > 0 ? __ldg(sl + ((size_t)r * NB + b) * 32 + lane) : 0ull;
    S.lo[b] = (uint32_t)v;
    S.hi[b] = (uint32_t)(v >> 32);
  }
}

// The lane's indices with partition q.
template <int NB>
__device__ __forceinline__ uint64_t members_of(const Slices<NB>& S, int q) {
  uint32_t lo = (uint32_t)S.valid, hi = (uint32_t)(S.valid >> 32);
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const uint32_t flip = ((q >> b) & 1) ? 0u : ~0u;
    lo &= S.lo[b] ^ flip;
    hi &= S.hi[b] ^ flip;
  }
  return ((uint64_t)hi << 32) | lo;
}

// Exclusive warp scan of two 16-bit counts packed in one word (every sum
// here stays below 2^16, so the halves never carry into each other).
__device__ __forceinline__ uint32_t warp_excl_scan2(uint32_t v, uint32_t* total) {
  const int lane = threadIdx.x & 31;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  *total = __shfl_sync(0xffffffffu, x, 31);
  return x - v;
}

__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Position of the n-th set bit (n counted from 0) of x, which has more than
// n set bits: halving popcounts, no branches.
__device__ __forceinline__ int select64(uint64_t x, int n) {
  uint32_t w = (uint32_t)x;
  int base = 0;
  int c = __popc(w);
  if (n >= c) {
    n -= c;
    w = (uint32_t)(x >> 32);
    base = 32;
  }
#pragma unroll
  for (int half = 16; half > 0; half >>= 1) {
    c = __popc(w & ((1u << half) - 1u));
    if (n >= c) {
      n -= c;
      w >>= half;
      base += half;
    }
  }
  return base;
}

// Bits [lb, lb + c) of a bitmap, c <= 64, least significant first.
__device__ __forceinline__ uint64_t extract_bits(const uint32_t* bits, uint32_t lb, int c) {
  if (c <= 0) return 0ull;
  const uint32_t w = lb >> 5, sh = lb & 31u;
  const uint32_t last = (lb + (uint32_t)c - 1u) >> 5;
  uint64_t x = __ldg(bits + w);
  if (w + 1u <= last) x |= (uint64_t)__ldg(bits + w + 1u) << 32;
  x >>= sh;
  if (w + 2u <= last) x |= (uint64_t)__ldg(bits + w + 2u) << (64u - sh);  // sh > 0 here
  return c >= 64 ? x : (x & ((1ull << c) - 1ull));
}

// ---------------------------------------------------------------- offsets
// Per CTA: len[q] = |I_q| (the directory's end column) and woff[q] =
// sum_{q' < q} ceil(|I_q'| / 32), woff[P] the total word count.  Returns
// false (for the whole CTA) when the directory was built for another (M, P,
// seed) or its lengths do not add up to M.  Warp 0, 8 partitions per lane.
// Ends with __syncthreads.
__device__ bool word_offsets(const HbGeom& G, const long long* hdr, const int32_t* cnt,
                             int32_t* len, uint32_t* woff) {
  __shared__ int s_ok;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    int l[8];
    long long n = 0;
    uint32_t w = 0;
    bool ok = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = lane * 8 + i;
      l[i] = q < G.parts ? __ldg(cnt + (size_t)q * G.stride + G.ranges) : 0;
      ok = ok && l[i] >= 0;
      n += l[i];
      w += ((uint32_t)l[i] + 31u) >> 5;
    }
    uint32_t x = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    uint32_t run = x - w;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = lane * 8 + i;
      if (q < G.parts) {
        len[q] = l[i];
        woff[q] = run;
      }
      run += ((uint32_t)l[i] + 31u) >> 5;
    }
    if (lane == 31) woff[G.parts] = x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
    ok = __all_sync(0xffffffffu, ok);
    // the directory was built for this (M, P, seed)
    const bool same = __ldg(hdr) == kDirMagic && __ldg(hdr + 1) == G.m && __ldg(hdr + 2) == G.parts &&
                      (unsigned long long)__ldg(hdr + 3) == G.seed;
    if (lane == 0) s_ok = ok && same && n == G.m;
  }
  __syncthreads();
  return s_ok != 0;
}

// Entry r of row q of a count array, for every lane: lanes hold the rows of
// partitions lane and lane + 32 ... (preloaded once per range); partitions
// past 64 are loaded directly (a broadcast load).
struct RowCache {
  int v[2];
};

__device__ __forceinline__ RowCache row_cache(const HbGeom& G, const int32_t* a, int r) {
  const int lane = threadIdx.x & 31;
  RowCache c;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int q = lane + 32 * h;
    c.v[h] = q < G.parts ? __ldg(a + (size_t)q * G.stride + r) : 0;
  }
  return c;
}

__device__ __forceinline__ int row_get(const HbGeom& G, const int32_t* a, const RowCache& c,
                                       int q, int r) {
  if (q < 32) return __shfl_sync(0xffffffffu, c.v[0], q);
  if (q < 64) return __shfl_sync(0xffffffffu, c.v[1], q - 32);
  return __ldg(a + (size_t)q * G.stride + r);
}

// ---------------------------------------------------------------- directory
// Slices of every range, and cnt[q][r] = range r's count of partition q (the
// scan kernel then turns each row into exclusive prefixes); cnt[q][R] = 0.
template <int NB>
__global__ void __launch_bounds__(kThreads)
hb_dir_build_kernel(const HbGeom G, long long* hdr, int32_t* cnt, uint64_t* sl) {
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    hdr[0] = kDirMagic;
    hdr[1] = G.m;
    hdr[2] = G.parts;
    hdr[3] = (long long)G.seed;
  }
  constexpr int kU = NB <= 4 ? (1 << NB) / 2 + 1 : 1;
  for (int r = blockIdx.x * kWarps + (threadIdx.x >> 5); r < G.ranges; r += gridDim.x * kWarps) {
    Slices<NB> S;
    slice_partitions<NB>(G, r * kRangeKeys + lane * kLaneKeys, S);
#pragma unroll
    for (int b = 0; b < NB; ++b)
      sl[((size_t)r * NB + b) * 32 + lane] = ((uint64_t)S.hi[b] << 32) | S.lo[b];
#pragma unroll kU
    for (int q = 0; q < (1 << NB); q += 2) {
      if (q >= G.parts) break;
      const uint32_t c0 = (uint32_t)__popcll(members_of<NB>(S, q));
      const uint32_t c1 = q + 1 < G.parts ? (uint32_t)__popcll(members_of<NB>(S, q + 1)) : 0u;
      const uint32_t t = warp_sum_u32(c0 | (c1 << 16));
      if (lane == 0) {
        cnt[(size_t)q * G.stride + r] = (int32_t)(t & 0xffffu);
        if (q + 1 < G.parts) cnt[(size_t)(q + 1) * G.stride + r] = (int32_t)(t >> 16);
      }
    }
  }
  if (blockIdx.x == 0)
    for (int q = threadIdx.x; q < G.parts; q += blockDim.x) cnt[(size_t)q * G.stride + G.ranges] = 0;
}

// In place, one CTA per row: entries 0 .. n-1 of row q (rows `stride` ints
// apart, 16-byte aligned) become their exclusive prefix sum, so the last
// entry ends as the row total.  32 entries per thread per pass.
constexpr int kScanPer = 32;

__global__ void __launch_bounds__(kScanThreads) hb_scan_kernel(int32_t* a, int n, int stride) {
  __shared__ int32_t s_warp[kScanThreads / 32];
  __shared__ int32_t s_tot;
  int32_t* row = a + (size_t)blockIdx.x * stride;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int carry = 0;
  for (int base = 0; base < n; base += kScanThreads * kScanPer) {
    const int i0 = base + tid * kScanPer;
    int v[kScanPer];
#pragma unroll
    for (int j = 0; j < kScanPer; j += 4) {
      if (i0 + j + 4 <= stride) {
        const int4 x = *reinterpret_cast<const int4*>(row + i0 + j);
        v[j] = i0 + j < n ? x.x : 0;
        v[j + 1] = i0 + j + 1 < n ? x.y : 0;
        v[j + 2] = i0 + j + 2 < n ? x.z : 0;
        v[j + 3] = i0 + j + 3 < n ? x.w : 0;
      } else {
        v[j] = v[j + 1] = v[j + 2] = v[j + 3] = 0;
      }
    }
    int s = 0;
#pragma unroll
    for (int j = 0; j < kScanPer; ++j) s += v[j];
    int x = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      const int w = s_warp[lane];
      int xw = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, xw, o);
        if (lane >= o) xw += y;
      }
      s_warp[lane] = xw - w;
      if (lane == 31) s_tot = xw;
    }
    __syncthreads();
    int run = carry + s_warp[warp] + (x - s);
#pragma unroll
    for (int j = 0; j < kScanPer; j += 4) {
      int o[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        o[t] = run;
        run += v[j + t];
      }
      if (i0 + j + 4 <= stride) {
        if (i0 + j + 4 <= n) {
          *reinterpret_cast<int4*>(row + i0 + j) = make_int4(o[0], o[1], o[2], o[3]);
        } else {
#pragma unroll
          for (int t = 0; t < 4; ++t)
            if (i0 + j + t < n) row[i0 + j + t] = o[t];
        }
      }
    }
    carry += s_tot;
    __syncthreads();
  }
}

// ---------------------------------------------------------------- encode
__global__ void hb_mark_kernel(const int32_t* keys, int64_t n_keys, int64_t m, uint32_t* mem,
                               int32_t* status) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_keys;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t k = keys[i];
    if (k >= 0 && k < m) atomicOr(&mem[k >> 5], 1u << (k & 31));
    else flag(status, ZR_ERR_INPUT_UNSORTED);
  }
}

struct EncArgs {
  HbGeom G;
  const long long* hdr;  // directory header
  const int32_t* cnt;    // directory counts
  const uint64_t* sl;    // directory slices
  const uint32_t* mem;
  uint32_t* out;
  long long out_cap;
  long long* d_woff;
  int32_t* status;
};

template <int NB>
__global__ void __launch_bounds__(kThreads) hb_encode_kernel(const __grid_constant__ EncArgs A) {
  __shared__ int32_t s_len[ZR_MAX_PARTS];
  __shared__ uint32_t s_woff[ZR_MAX_PARTS + 1];
  __shared__ uint64_t s_eq[kWarps][kChunk][32];
  __shared__ uint32_t s_first[kWarps][kChunk][32];
  const HbGeom& G = A.G;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (!word_offsets(G, A.hdr, A.cnt, s_len, s_woff)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag(A.status, ZR_ERR_INVALID_ARG);
    return;
  }
  if (blockIdx.x == 0)
    for (int q = threadIdx.x; q <= G.parts; q += blockDim.x) A.d_woff[q] = s_woff[q];
  if ((long long)s_woff[G.parts] > A.out_cap) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag(A.status, ZR_ERR_CAPACITY);
    return;
  }
  const int mwords = (int)(((long long)G.m + 31) >> 5);  // M + 31 can pass 2^31 - 1
  for (int r = blockIdx.x * kWarps + warp; r < G.ranges; r += gridDim.x * kWarps) {
    const int x0 = r * kRangeKeys + lane * kLaneKeys;
    const RowCache c_s = row_cache(G, A.cnt, r), c_e = row_cache(G, A.cnt, r + 1);
    Slices<NB> S;
    load_slices<NB>(G, A.sl, r, x0, S);
    uint64_t mb = 0;
    const int w0 = x0 >> 5;
    if (w0 < mwords) mb = __ldg(A.mem + w0);
    if (w0 + 1 < mwords) mb |= (uint64_t)__ldg(A.mem + w0 + 1) << 32;
    mb &= S.valid;
    bool bad = false;
    for (int q0 = 0; q0 < G.parts; q0 += kChunk) {
      // ranks: the lane's indices of every partition of the chunk and the
      // position j of its first one in I_q
      uint64_t in_chunk = 0;
#pragma unroll
      for (int qi = 0; qi < kChunk; qi += 2) {
        const int q = q0 + qi;
        if (q >= G.parts) break;
        uint64_t eq[2];
        eq[0] = members_of<NB>(S, q);
        eq[1] = q + 1 < G.parts ? members_of<NB>(S, q + 1) : 0ull;
        uint32_t tot;
        const uint32_t ex2 = warp_excl_scan2(
            (uint32_t)__popcll(eq[0]) | ((uint32_t)__popcll(eq[1]) << 16), &tot);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int qq = q + h;
          if (qq >= G.parts) break;
          const int s = row_get(G, A.cnt, c_s, qq, r);
          const int e = row_get(G, A.cnt, c_e, qq, r + 1);
          if (s < 0 || e > s_len[qq] || e - s != (int)((tot >> (16 * h)) & 0xffffu)) {
            bad = true;
            eq[h] = 0ull;  // no member of qq is placed from this range
          }
          s_eq[warp][qi + h][lane] = eq[h];
          s_first[warp][qi + h][lane] = (uint32_t)s + ((ex2 >> (16 * h)) & 0xffffu);
          in_chunk |= eq[h];
        }
      }
      __syncwarp();
      // members of the chunk, dealt to the lanes: member j belongs to the
      // lane l with mex_l <= j < mex_l + count_l, at its (j - mex_l)-th
      // member index
      const uint64_t mbc = mb & in_chunk;
      uint32_t tm;
      const uint32_t mex = warp_excl_scan2((uint32_t)__popcll(mbc), &tm);
      for (uint32_t j0 = 0; j0 < tm; j0 += 32) {
        const uint32_t j = j0 + lane;
        int l = 0;
#pragma unroll
        for (int step = 16; step > 0; step >>= 1) {
          const uint32_t v = __shfl_sync(0xffffffffu, mex, (l + step) & 31);
          if (l + step < 32 && v <= j) l += step;
        }
        const uint32_t t = j - __shfl_sync(0xffffffffu, mex, l);
        const uint32_t mlo = __shfl_sync(0xffffffffu, (uint32_t)mbc, l);
        const uint32_t mhi = __shfl_sync(0xffffffffu, (uint32_t)(mbc >> 32), l);
        if (j < tm) {
          const int kp = select64(((uint64_t)mhi << 32) | mlo, (int)t);
          const uint32_t x = (uint32_t)(r * kRangeKeys + l * kLaneKeys + kp);
          const int q = (int)G.h(x);
          const int qi = q - q0;
          if ((unsigned)qi < (unsigned)kChunk && q < G.parts) {
            const uint64_t eq = s_eq[warp][qi][l];
            const uint32_t rank = (uint32_t)__popcll(eq & ((1ull << kp) - 1ull));
            const uint32_t jq = s_first[warp][qi][l] + rank;
            if ((int)jq < s_len[q] && ((eq >> kp) & 1ull)) {
              const uint32_t bit = s_woff[q] * 32u + jq;
              atomicOr(A.out + (bit >> 5), 1u << (bit & 31u));
            } else {
              flag(A.status, ZR_ERR_INVALID_ARG);
            }
          } else {
            flag(A.status, ZR_ERR_INVALID_ARG);  // slices that disagree with h0
          }
        }
      }
      __syncwarp();
    }
    if (bad && lane == 0) flag(A.status, ZR_ERR_INVALID_ARG);
  }
}

// ---------------------------------------------------------------- decode
// seg[q][r] = set bits of partition q's bitmap in range r's segment
// [cnt[q][r], cnt[q][r+1]); seg[q][R] = 0.  A warp per range, a lane per
// partition, each lane over its segment's words (four loads in flight).
// CTA 0 also checks that no padding bit is set.
__global__ void __launch_bounds__(kThreads)
hb_seg_count_kernel(const HbGeom G, const long long* hdr, const int32_t* cnt,
                    const uint32_t* bits, int32_t* seg, int32_t* status) {
  __shared__ int32_t s_len[ZR_MAX_PARTS];
  __shared__ uint32_t s_woff[ZR_MAX_PARTS + 1];
  const int lane = threadIdx.x & 31;
  if (!word_offsets(G, hdr, cnt, s_len, s_woff)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag(status, ZR_ERR_INVALID_ARG);
    return;
  }
  if (blockIdx.x == 0) {
    for (int q = threadIdx.x; q < G.parts; q += blockDim.x) {
      seg[(size_t)q * G.stride + G.ranges] = 0;
      const int rem = s_len[q] & 31;
      if (rem && (bits[s_woff[q] + ((uint32_t)s_len[q] >> 5)] >> rem) != 0u)
        flag(status, ZR_ERR_INVALID_ARG);  // a padding bit is set
    }
  }
  for (int r = blockIdx.x * kWarps + (threadIdx.x >> 5); r < G.ranges; r += gridDim.x * kWarps) {
    for (int q = lane; q < G.parts; q += 32) {
      const int s = __ldg(cnt + (size_t)q * G.stride + r);
      const int e = __ldg(cnt + (size_t)q * G.stride + r + 1);
      uint32_t c = 0;
      if (s >= 0 && e >= s && e <= s_len[q]) {
        if (e > s) {
          const uint32_t lo = s_woff[q] * 32u + (uint32_t)s, hi = s_woff[q] * 32u + (uint32_t)e;
          const uint32_t w0 = lo >> 5, w1 = (hi - 1u) >> 5;
          for (uint32_t w = w0; w <= w1; w += 4) {
            uint32_t x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) x[u] = w + u <= w1 ? __ldg(bits + w + u) : 0u;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (w + u == w0) x[u] &= ~0u << (lo & 31u);
              if (w + u == w1 && (hi & 31u)) x[u] &= ~0u >> (32u - (hi & 31u));
              c += __popc(x[u]);
            }
          }
        }
      } else {
        flag(status, ZR_ERR_INVALID_ARG);
      }
      seg[(size_t)q * G.stride + r] = (int32_t)c;
    }
  }
}

struct DecArgs {
  HbGeom G;
  const long long* hdr;  // directory header
  const int32_t* cnt;    // directory counts
  const uint64_t* sl;    // directory slices
  const uint32_t* bits;
  const int32_t* seg;    // exclusive prefix per partition; seg[q][R] = partition total
  int32_t* out;
  long long out_cap;
  long long* d_koff;
  int32_t* status;
};

template <int NB>
__global__ void __launch_bounds__(kThreads, 8) hb_decode_kernel(const __grid_constant__ DecArgs A) {
  __shared__ int32_t s_len[ZR_MAX_PARTS];
  __shared__ uint32_t s_woff[ZR_MAX_PARTS + 1];
  __shared__ long long s_koff[ZR_MAX_PARTS + 1];
  __shared__ uint64_t s_eq[kWarps][kChunk][32];
  __shared__ uint64_t s_mk[kWarps][kChunk][32];
  __shared__ uint32_t s_mex[kWarps][kChunk][32];
  __shared__ long long s_ob[kWarps][kChunk];
  __shared__ uint32_t s_cm[kWarps][kChunk + 1];
  const HbGeom& G = A.G;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (!word_offsets(G, A.hdr, A.cnt, s_len, s_woff)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag(A.status, ZR_ERR_INVALID_ARG);
    return;
  }
  if (threadIdx.x < 32) {
    // key offsets: exclusive prefix of the partition totals, 8 per lane
    long long t[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = lane * 8 + i;
      t[i] = q < G.parts ? __ldg(A.seg + (size_t)q * G.stride + G.ranges) : 0;
      sum += t[i];
    }
    long long x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    long long run = x - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = lane * 8 + i;
      if (q < G.parts) s_koff[q] = run;
      run += t[i];
    }
    if (lane == 31) {
      s_koff[G.parts] = x;
      if (blockIdx.x == 0 && x > A.out_cap) flag(A.status, ZR_ERR_CAPACITY);
    }
  }
  __syncthreads();
  if (blockIdx.x == 0)
    for (int q = threadIdx.x; q <= G.parts; q += blockDim.x) A.d_koff[q] = s_koff[q];
  for (int r = blockIdx.x * kWarps + warp; r < G.ranges; r += gridDim.x * kWarps) {
    const int x0 = r * kRangeKeys + lane * kLaneKeys;
    const RowCache c_s = row_cache(G, A.cnt, r), c_e = row_cache(G, A.cnt, r + 1);
    const RowCache c_g = row_cache(G, A.seg, r);
    Slices<NB> S;
    load_slices<NB>(G, A.sl, r, x0, S);
    bool bad = false;
    for (int q0 = 0; q0 < G.parts; q0 += kChunk) {
      // per partition of the chunk: the lane's indices (eq), its bits of the
      // segment (mk: bit t set iff its t-th index of q is a member) and the
      // members of the lanes before it (mex)
      // pass 1: the lane's indices of every partition of the chunk and the
      // first bit of them in q's segment (lb; the slot of s_mex holds it)
#pragma unroll
      for (int qi = 0; qi < kChunk; qi += 2) {
        const int q = q0 + qi;
        if (q >= G.parts) break;
        uint64_t eq[2];
        eq[0] = members_of<NB>(S, q);
        eq[1] = q + 1 < G.parts ? members_of<NB>(S, q + 1) : 0ull;
        uint32_t tot;
        const uint32_t ex2 = warp_excl_scan2(
            (uint32_t)__popcll(eq[0]) | ((uint32_t)__popcll(eq[1]) << 16), &tot);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int qq = q + h;
          uint32_t lb = 0;
          if (qq < G.parts) {
            const int s = row_get(G, A.cnt, c_s, qq, r);
            const int e = row_get(G, A.cnt, c_e, qq, r + 1);
            if (s < 0 || e > s_len[qq] || e - s != (int)((tot >> (16 * h)) & 0xffffu)) {
              bad = true;
              eq[h] = 0ull;  // nothing of qq is decoded from this range
            }
            lb = s_woff[qq] * 32u + (uint32_t)s + ((ex2 >> (16 * h)) & 0xffffu);
          }
          s_eq[warp][qi + h][lane] = eq[h];
          s_mex[warp][qi + h][lane] = lb;
        }
      }
      // pass 2: the lane's bits of every segment, all loads in flight at once
#pragma unroll
      for (int qi = 0; qi < kChunk; ++qi) {
        if (q0 + qi >= G.parts) break;
        s_mk[warp][qi][lane] =
            extract_bits(A.bits, s_mex[warp][qi][lane], __popcll(s_eq[warp][qi][lane]));
      }
      // pass 3: members of the lanes before (mex) and of the partitions
      // before (cm), output bases
      uint32_t cm = 0;
#pragma unroll
      for (int qi = 0; qi < kChunk; qi += 2) {
        const int q = q0 + qi;
        if (q >= G.parts) break;
        const uint64_t mk0 = s_mk[warp][qi][lane];
        const uint64_t mk1 = q + 1 < G.parts ? s_mk[warp][qi + 1][lane] : 0ull;
        uint32_t mtot;
        const uint32_t mex2 = warp_excl_scan2(
            (uint32_t)__popcll(mk0) | ((uint32_t)__popcll(mk1) << 16), &mtot);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int qq = q + h;
          const int g = qq < G.parts ? row_get(G, A.seg, c_g, qq, r) : 0;
          if (qq >= G.parts) s_mk[warp][qi + h][lane] = 0ull;
          s_mex[warp][qi + h][lane] = (mex2 >> (16 * h)) & 0xffffu;
          if (lane == 0) {
            s_cm[warp][qi + h] = cm;
            s_ob[warp][qi + h] = qq < G.parts ? s_koff[qq] + g : 0;
          }
          cm += (mtot >> (16 * h)) & 0xffffu;
        }
      }
      if (lane == 0)
        for (int qi = ((G.parts - q0 < kChunk ? G.parts - q0 : kChunk) + 1) & ~1; qi <= kChunk; ++qi)
          s_cm[warp][qi] = cm;
      __syncwarp();
      // the chunk's members, partition-major, dealt to the lanes
      for (uint32_t j0 = 0; j0 < cm; j0 += 32) {
        const uint32_t j = j0 + lane;
        if (j < cm) {
          int qi = 0;
#pragma unroll
          for (int i = 1; i < kChunk; ++i)
            if (s_cm[warp][i] <= j) qi = i;
          const uint32_t jj = j - s_cm[warp][qi];
          int l = 0;
#pragma unroll
          for (int step = 16; step > 0; step >>= 1)
            if (l + step < 32 && s_mex[warp][qi][l + step] <= jj) l += step;
          const int t = (int)(jj - s_mex[warp][qi][l]);
          const int rb = select64(s_mk[warp][qi][l], t);
          const int kp = select64(s_eq[warp][qi][l], rb);
          const long long o = s_ob[warp][qi] + jj;
          if (o < A.out_cap) A.out[o] = r * kRangeKeys + l * kLaneKeys + kp;
          else flag(A.status, s_koff[G.parts] > A.out_cap ? ZR_ERR_CAPACITY : ZR_ERR_INTERNAL);
        }
      }
      __syncwarp();
    }
    if (bad && lane == 0) flag(A.status, ZR_ERR_INVALID_ARG);
  }
}

// ---------------------------------------------------------------- host side
using DirFn = void (*)(const HbGeom, long long*, int32_t*, uint64_t*);
using EncFn = void (*)(const EncArgs);
using DecFn = void (*)(const DecArgs);

template <int NB>
void fill_fns(DirFn* d, EncFn* e, DecFn* c) {
  d[NB] = hb_dir_build_kernel<NB>;
  e[NB] = hb_encode_kernel<NB>;
  c[NB] = hb_decode_kernel<NB>;
}

struct Fns {
  DirFn dir[kMaxBits + 1];
  EncFn enc[kMaxBits + 1];
  DecFn dec[kMaxBits + 1];
  Fns() {
    fill_fns<0>(dir, enc, dec);
    fill_fns<1>(dir, enc, dec);
    fill_fns<2>(dir, enc, dec);
    fill_fns<3>(dir, enc, dec);
    fill_fns<4>(dir, enc, dec);
    fill_fns<5>(dir, enc, dec);
    fill_fns<6>(dir, enc, dec);
    fill_fns<7>(dir, enc, dec);
    fill_fns<8>(dir, enc, dec);
  }
};

const Fns& fns() {
  static const Fns f;
  return f;
}

// CTAs of kThreads for a range-strided kernel: the ranges' warps, at most
// what the GPU holds at once.  The occupancy of each kernel (slot) is asked
// once per device.
constexpr int kSlots = 3 * (kMaxBits + 1) + 1;

int range_grid(const void* fn, int slot, int64_t ranges) {
  static std::atomic<int> per_sm[64][kSlots];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int per = per_sm[dev][slot].load(std::memory_order_relaxed);
  if (per < 1) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, fn, kThreads, 0) != cudaSuccess ||
        per < 1)
      per = 1;
    per_sm[dev][slot].store(per, std::memory_order_relaxed);
  }
  int64_t g = (ranges + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)sm_count() * per;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

HbGeom make_geom(int64_t m, int parts, uint64_t seed) {
  HbGeom G;
  G.m = (int)m;
  G.parts = parts;
  G.ranges = (int)ranges_of(m);
  G.stride = (int)row_stride(m);
  G.seed = seed;
  G.h = make_h0(seed, (uint32_t)parts);
  return G;
}

const long long* dir_header(const int32_t* d_dir) {
  return reinterpret_cast<const long long*>(d_dir);
}

const int32_t* dir_counts(const int32_t* d_dir) {
  return reinterpret_cast<const int32_t*>(reinterpret_cast<const unsigned char*>(d_dir) +
                                          kDirHeader);
}

const uint64_t* dir_slices(const int32_t* d_dir, int64_t m, int parts) {
  return reinterpret_cast<const uint64_t*>(reinterpret_cast<const unsigned char*>(d_dir) +
                                           kDirHeader + dir_counts_bytes(m, parts));
}

}  // namespace

size_t hash_directory_bytes(int64_t m, int n_parts) {
  return kDirHeader + dir_counts_bytes(m, n_parts) +
         (size_t)ranges_of(m) * (size_t)part_bits(n_parts) * 32 * sizeof(uint64_t);
}

size_t hash_bitmap_workspace_bytes(int64_t m, int n_parts) { return hb_layout(m, n_parts).total; }

zr_status hash_directory_launch(int64_t m, int n_parts, uint64_t part_seed, int32_t* d_dir,
                                cudaStream_t stream) {
  const HbGeom G = make_geom(m, n_parts, part_seed);
  const int nb = part_bits(n_parts);
  const DirFn fn = fns().dir[nb];
  long long* hdr = const_cast<long long*>(dir_header(d_dir));
  int32_t* cnt = const_cast<int32_t*>(dir_counts(d_dir));
  uint64_t* sl = const_cast<uint64_t*>(dir_slices(d_dir, m, n_parts));
  fn<<<range_grid((const void*)fn, nb, G.ranges), kThreads, 0, stream>>>(G, hdr, cnt, sl);
  hb_scan_kernel<<<n_parts, kScanThreads, 0, stream>>>(cnt, G.ranges + 1, G.stride);
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
}

zr_status hash_bitmap_encode_launch(const int32_t* d_dir, int64_t m, int n_parts,
                                    uint64_t part_seed, const int32_t* keys, int64_t n_keys,
                                    uint32_t* out_bits, int64_t out_cap_words,
                                    int64_t* d_word_offsets, void* ws, cudaStream_t stream) {
  const HbLayout L = hb_layout(m, n_parts);
  unsigned char* w = static_cast<unsigned char*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  uint32_t* mem = reinterpret_cast<uint32_t*>(w + L.mem);
  if (cudaMemsetAsync(w, 0, L.seg, stream) != cudaSuccess) return ZR_ERR_CUDA;  // status + map
  // every word a bitmap can have: sum ceil(|I_q| / 32) <= ceil(M / 32) + P
  int64_t zero_words = (m + 31) / 32 + n_parts;
  if (zero_words > out_cap_words) zero_words = out_cap_words;
  if (cudaMemsetAsync(out_bits, 0, (size_t)zero_words * 4, stream) != cudaSuccess)
    return ZR_ERR_CUDA;
  if (n_keys > 0) {
    int64_t g = (n_keys + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (g > cap) g = cap;
    hb_mark_kernel<<<(unsigned)g, 256, 0, stream>>>(keys, n_keys, m, mem, status);
  }
  EncArgs A;
  A.G = make_geom(m, n_parts, part_seed);
  A.hdr = dir_header(d_dir);
  A.cnt = dir_counts(d_dir);
  A.sl = dir_slices(d_dir, m, n_parts);
  A.mem = mem;
  A.out = out_bits;
  A.out_cap = out_cap_words;
  A.d_woff = reinterpret_cast<long long*>(d_word_offsets);
  A.status = status;
  const int nb = part_bits(n_parts);
  const EncFn fn = fns().enc[nb];
  fn<<<range_grid((const void*)fn, kMaxBits + 1 + nb, A.G.ranges), kThreads, 0, stream>>>(A);
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
}

zr_status hash_bitmap_decode_launch(const int32_t* d_dir, int64_t m, int n_parts,
                                    uint64_t part_seed, const uint32_t* bits, int32_t* out_keys,
                                    int64_t out_cap, int64_t* d_key_offsets, void* ws,
                                    cudaStream_t stream) {
  const HbLayout L = hb_layout(m, n_parts);
  unsigned char* w = static_cast<unsigned char*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  int32_t* seg = reinterpret_cast<int32_t*>(w + L.seg);
  if (cudaMemsetAsync(w, 0, 256, stream) != cudaSuccess) return ZR_ERR_CUDA;
  const HbGeom G = make_geom(m, n_parts, part_seed);
  hb_seg_count_kernel<<<range_grid((const void*)hb_seg_count_kernel, kSlots - 1, G.ranges),
                        kThreads, 0, stream>>>(G, dir_header(d_dir), dir_counts(d_dir), bits, seg,
                                               status);
  hb_scan_kernel<<<n_parts, kScanThreads, 0, stream>>>(seg, G.ranges + 1, G.stride);
  DecArgs A;
  A.G = G;
  A.hdr = dir_header(d_dir);
  A.cnt = dir_counts(d_dir);
  A.sl = dir_slices(d_dir, m, n_parts);
  A.bits = bits;
  A.seg = seg;
  A.out = out_keys;
  A.out_cap = out_cap;
  A.d_koff = reinterpret_cast<long long*>(d_key_offsets);
  A.status = status;
  const int nb = part_bits(n_parts);
  const DecFn fn = fns().dec[nb];
  fn<<<range_grid((const void*)fn, 2 * (kMaxBits + 1) + nb, G.ranges), kThreads, 0, stream>>>(A);
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
}

}  // namespace zr
