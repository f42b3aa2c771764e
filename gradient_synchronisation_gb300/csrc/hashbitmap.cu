// Zen's hash bitmap: encode a server's nonzero indices as one bit per element
// of its index set, and decode such bitmaps back to indices.
//
// What is computed (Zen page, section 3.3.2 "Hash bitmap", Figure 10 and
// Algorithm 2): with h0, I_p = {x in [0, M) : h0(x) = p}, sorted (built once
// by zr_hash_index_sets).  Encode sets bit j of partition p's bitmap when
// I_p[j] is one of the given nonzero indices; decode outputs I_p[j] for every
// set bit j.  Bit j is bit (j mod 32) of word floor(j / 32); partition p's
// words start at word offset sum_{q < p} ceil(|I_q| / 32).
//
// GB300 design.  Both directions stream the index sets once with 128-byte
// coalesced warp loads; a warp handles 32 consecutive bitmap words at a time.
//   encode: the nonzero indices are first marked in a membership bitmap of
//           M bits (workspace; it stays in L2), then lane l of the warp tests
//           element 32j + l of the word's index set and a ballot forms word j;
//           the elements of the next 4 words load while the current 4 test
//           their bits, and the 32 words leave as one coalesced store.
//   decode: per tile of 1024 words, a popcount pass and a one-CTA scan give
//           every tile its first output position; then each warp takes 32
//           words at a time, lane l word j = g0 + l, and the lane writes
//           I_p[32j + b] for every set bit b of its word at the word's output
//           base (a prefix of the popcounts over the lanes) plus the rank of
//           b among the word's set bits, up to 4 gathers in flight.
// Every index taken from the inputs is range-checked before it addresses
// memory; every output position is checked against the output capacity.

#include <cuda_runtime.h>
#include <stdint.h>

#include "zr.h"
#include "zr_internal.h"

namespace zr {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTileWords = 1024;  // decode tile
constexpr int kScanThreads = 1024;
constexpr int kEncBatch = 4;      // encode: words per load batch (4, 8 and 16 measured; 4 fastest)

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

__device__ __forceinline__ void flag(int32_t* status, int code) { atomicCAS(status, 0, code); }

int64_t words_bound(int64_t m, int parts) { return (m + 31) / 32 + parts; }

// Workspace: [status | word offsets (parts + 1) | membership bitmap | tile
// counts | tile bases].
struct HbLayout {
  size_t woff, mem, tcnt, tbase, total;
};

HbLayout hb_layout(int64_t m, int parts) {
  HbLayout L;
  const int64_t tiles = (words_bound(m, parts) + kTileWords - 1) / kTileWords;
  L.woff = 256;
  L.mem = L.woff + align256((size_t)(parts + 1) * 8);
  L.tcnt = L.mem + align256((size_t)((m + 31) / 32) * 4);
  L.tbase = L.tcnt + align256((size_t)tiles * 4);
  L.total = L.tbase + align256((size_t)tiles * 8);
  return L;
}

// woff[p] = sum_{q < p} ceil(|I_q| / 32), from the index-set offsets (one
// thread; parts <= 256).  Offsets that do not describe index sets of [0, m)
// (not starting at 0, not ending at m, or decreasing) give empty bitmaps, so
// the later kernels touch nothing; the function returns false for them.
__device__ bool word_offsets(const int64_t* set_off, int parts, int64_t m, int64_t* woff) {
  bool ok = set_off[0] == 0 && set_off[parts] == m;
  for (int p = 0; p < parts; ++p) ok = ok && set_off[p + 1] >= set_off[p];
  int64_t acc = 0;
  for (int p = 0; p <= parts; ++p) {
    woff[p] = acc;
    if (ok && p < parts) acc += (set_off[p + 1] - set_off[p] + 31) / 32;
  }
  return ok;
}

// The encoder's word offsets, also returned to the caller (woff_out).
__global__ void hb_word_offsets_kernel(const int64_t* set_off, int parts, int64_t m,
                                       int64_t* woff_ws, int64_t* woff_out, int32_t* status) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  const bool ok = word_offsets(set_off, parts, m, woff_ws);
  if (woff_out)
    for (int p = 0; p <= parts; ++p) woff_out[p] = woff_ws[p];
  if (!ok) flag(status, ZR_ERR_INVALID_ARG);
}

__global__ void hb_mark_kernel(const int32_t* keys, int64_t n_keys, int64_t m, uint32_t* mem,
                               int32_t* status) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_keys;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t k = keys[i];
    if (k >= 0 && k < m) atomicOr(&mem[k >> 5], 1u << (k & 31));
    else flag(status, ZR_ERR_INPUT_UNSORTED);
  }
}

// Partition of global word g, starting the search at p (words never go
// backwards inside a warp's run, so the search only moves forward).
__device__ __forceinline__ int word_part(const int64_t* woff, int parts, int64_t g, int p) {
  while (p < parts - 1 && g >= woff[p + 1]) ++p;
  return p;
}

__device__ __forceinline__ void load_offsets(const int64_t* woff_ws, const int64_t* set_off,
                                             int parts, int64_t* s_woff, int64_t* s_soff) {
  for (int p = threadIdx.x; p <= parts; p += blockDim.x) {
    s_woff[p] = woff_ws[p];
    s_soff[p] = set_off[p];
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads)
hb_encode_kernel(const int32_t* sets, const int64_t* set_off, int64_t m, int parts,
                 const int64_t* woff_ws, const uint32_t* mem, uint32_t* out, int64_t out_cap,
                 int32_t* status) {
  __shared__ int64_t s_woff[ZR_MAX_PARTS + 1], s_soff[ZR_MAX_PARTS + 1];
  load_offsets(woff_ws, set_off, parts, s_woff, s_soff);
  const int lane = threadIdx.x & 31;
  const int64_t total = s_woff[parts];
  if (total > out_cap) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag(status, ZR_ERR_CAPACITY);
    return;
  }
  const int64_t nwarps = (int64_t)gridDim.x * kWarps;
  for (int64_t g0 = ((int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5)) * 32; g0 < total;
       g0 += nwarps * 32) {
    int p = word_part(s_woff, parts, g0, 0);
    uint32_t mine = 0;
    // Batches of kEncBatch words: the index-set elements of the next batch
    // are loaded while the current batch looks up its membership bits, so
    // two batches' loads are in flight.
    int32_t x[2][kEncBatch];
    bool in[2][kEncBatch];
    auto load_batch = [&](int u0, int32_t (&xs)[kEncBatch], bool (&ins)[kEncBatch]) {
#pragma unroll
      for (int u = 0; u < kEncBatch; ++u) {
        const int64_t g = g0 + u0 + u;
        ins[u] = false;
        xs[u] = 0;
        if (u0 + u < 32 && g < total) {
          p = word_part(s_woff, parts, g, p);
          const int64_t pos = (g - s_woff[p]) * 32 + lane;
          if (pos < s_soff[p + 1] - s_soff[p]) {
            xs[u] = __ldg(sets + s_soff[p] + pos);
            ins[u] = true;
          }
        }
      }
    };
    load_batch(0, x[0], in[0]);
#pragma unroll
    for (int bt = 0; bt < 32 / kEncBatch; ++bt) {
      const int u0 = bt * kEncBatch;
      if (bt + 1 < 32 / kEncBatch) load_batch(u0 + kEncBatch, x[(bt + 1) & 1], in[(bt + 1) & 1]);
#pragma unroll
      for (int u = 0; u < kEncBatch; ++u) {
        bool bit = false;
        const int32_t xv = x[bt & 1][u];
        if (in[bt & 1][u]) {
          if (xv >= 0 && xv < m) bit = (__ldg(mem + (xv >> 5)) >> (xv & 31)) & 1u;
          else flag(status, ZR_ERR_INVALID_ARG);
        }
        const uint32_t w = __ballot_sync(0xffffffffu, bit);
        if (lane == u0 + u) mine = w;
      }
    }
    if (g0 + lane < total) out[g0 + lane] = mine;
  }
}

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

__global__ void __launch_bounds__(kThreads)
hb_tile_count_kernel(const uint32_t* bits, const int64_t* set_off, int parts, int64_t m,
                     int64_t* woff_ws, int32_t* tcnt, int32_t* status) {
  __shared__ int32_t s_sum[kWarps];
  __shared__ int64_t s_woff[ZR_MAX_PARTS + 1];
  // every CTA derives the word offsets; CTA 0 also stores them for the scan
  // and the decode
  if (threadIdx.x == 0) {
    const bool ok = word_offsets(set_off, parts, m, s_woff);
    if (blockIdx.x == 0) {
      for (int p = 0; p <= parts; ++p) woff_ws[p] = s_woff[p];
      if (!ok) flag(status, ZR_ERR_INVALID_ARG);
    }
  }
  __syncthreads();
  const int64_t total = s_woff[parts];
  const int64_t tiles = (total + kTileWords - 1) / kTileWords;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int64_t lo = t * kTileWords, hi = min(lo + kTileWords, total);
    int c = 0;
    for (int64_t g = lo + threadIdx.x; g < hi; g += kThreads) c += __popc(bits[g]);
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if ((threadIdx.x & 31) == 0) s_sum[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
      int s = 0;
      for (int w = 0; w < kWarps; ++w) s += s_sum[w];
      tcnt[t] = s;
    }
    __syncthreads();
  }
}

// One CTA: tile bases (exclusive prefix of the tile counts) and the key
// offsets of every partition.
__global__ void __launch_bounds__(kScanThreads)
hb_scan_kernel(const uint32_t* bits, const int64_t* woff_ws, int parts, const int32_t* tcnt,
               int64_t* tbase, int64_t* key_off, int64_t out_cap, int32_t* status) {
  __shared__ long long s_warp[kScanThreads / 32 + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t total = woff_ws[parts];
  const int64_t tiles = (total + kTileWords - 1) / kTileWords;
  long long carry = 0;
  for (int64_t t0 = 0; t0 < tiles; t0 += kScanThreads) {
    const int64_t t = t0 + tid;
    const int v = t < tiles ? tcnt[t] : 0;
    const int incl = warp_incl_scan(v);
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const long long x = s_warp[lane];
      long long xi = x;
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, xi, o);
        if (lane >= o) xi += y;
      }
      s_warp[lane] = xi - x;
      if (lane == 31) s_warp[32] = xi;
    }
    __syncthreads();
    if (t < tiles) tbase[t] = carry + s_warp[warp] + (incl - v);
    carry += s_warp[32];
    __syncthreads();
  }
  if (carry > out_cap && tid == 0) flag(status, ZR_ERR_CAPACITY);
  __syncthreads();
  // key offset of partition p: the set bits before its first word = its
  // tile's base plus the popcount of the tile's words before it; one warp
  // per partition (the tile bases above are visible after the barrier)
  for (int p = warp; p <= parts; p += kScanThreads / 32) {
    const int64_t w = woff_ws[p];
    const int64_t t = w / kTileWords;
    int c = 0;
    if (t < tiles)
      for (int64_t g = t * kTileWords + lane; g < w; g += 32) c += __popc(bits[g]);
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) key_off[p] = (t < tiles ? tbase[t] : carry) + c;
  }
}

__global__ void __launch_bounds__(kThreads)
hb_decode_kernel(const int32_t* sets, const int64_t* set_off, int parts, const uint32_t* bits,
                 const int64_t* woff_ws, const int64_t* tbase, int32_t* out, int64_t out_cap,
                 int32_t* status) {
  __shared__ int64_t s_woff[ZR_MAX_PARTS + 1], s_soff[ZR_MAX_PARTS + 1];
  __shared__ int32_t s_wsum[kWarps];
  load_offsets(woff_ws, set_off, parts, s_woff, s_soff);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t total = s_woff[parts];
  const int64_t tiles = (total + kTileWords - 1) / kTileWords;
  constexpr int kPerWarp = kTileWords / kWarps;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int64_t wlo = t * kTileWords + (int64_t)warp * kPerWarp;
    const int64_t whi = min(wlo + kPerWarp, min(t * kTileWords + kTileWords, total));
    int c = 0;
    for (int64_t g = wlo + lane; g < whi; g += 32) c += __popc(bits[g]);
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) s_wsum[warp] = c;
    __syncthreads();
    long long run = tbase[t];
    for (int w = 0; w < warp; ++w) run += s_wsum[w];
    // Lane l takes word g0 + l and walks its set bits: up to 4 gathers of
    // index-set elements in flight (read-only loads), then their stores at
    // the word's output base plus the bits' rank.
    int p = 0;
    for (int64_t g0 = wlo; g0 < whi; g0 += 32) {
      const int64_t g = g0 + lane;
      const uint32_t mine = g < whi ? bits[g] : 0u;
      const int cnt = __popc(mine);
      const int incl = warp_incl_scan(cnt);
      if (mine) {
        p = word_part(s_woff, parts, g, p);
        const int64_t set_lo = s_soff[p];
        const int64_t set_n = s_soff[p + 1] - set_lo;
        const int64_t pos0 = (g - s_woff[p]) * 32;
        long long o = run + incl - cnt;
        uint32_t w = mine;
        while (w) {
          int32_t key[4];
          long long at[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            at[i] = -1;
            if (w) {
              const int bit = __ffs(w) - 1;
              w &= w - 1;
              const int64_t pos = pos0 + bit;
              if (pos < set_n && o < out_cap) {
                key[i] = __ldg(sets + set_lo + pos);
                at[i] = o;
              } else {
                flag(status, ZR_ERR_INVALID_ARG);  // a bit past the set's end, or no room
              }
              ++o;
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (at[i] >= 0) out[at[i]] = key[i];
        }
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    __syncthreads();
  }
}

int grid_for(int64_t units, int per_sm) {
  int64_t g = (int64_t)sm_count() * per_sm;
  if (g > units) g = units;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

size_t hash_bitmap_workspace_bytes(int64_t m, int n_parts) { return hb_layout(m, n_parts).total; }

zr_status hash_bitmap_encode_launch(const int32_t* sets, const int64_t* d_set_offsets, int64_t m,
                                    int n_parts, const int32_t* keys, int64_t n_keys,
                                    uint32_t* out_bits, int64_t out_cap_words,
                                    int64_t* d_word_offsets, void* ws, cudaStream_t stream) {
  const HbLayout L = hb_layout(m, n_parts);
  unsigned char* w = static_cast<unsigned char*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  int64_t* woff = reinterpret_cast<int64_t*>(w + L.woff);
  uint32_t* mem = reinterpret_cast<uint32_t*>(w + L.mem);
  if (cudaMemsetAsync(w, 0, L.tcnt, stream) != cudaSuccess) return ZR_ERR_CUDA;  // status + bitmap
  hb_word_offsets_kernel<<<1, 32, 0, stream>>>(d_set_offsets, n_parts, m, woff, d_word_offsets,
                                                status);
  if (n_keys > 0)
    hb_mark_kernel<<<grid_for((n_keys + kThreads - 1) / kThreads, 8), kThreads, 0, stream>>>(
        keys, n_keys, m, mem, status);
  const int64_t warp_units = (words_bound(m, n_parts) + 31) / 32;
  hb_encode_kernel<<<grid_for((warp_units + kWarps - 1) / kWarps, 8), kThreads, 0, stream>>>(
      sets, d_set_offsets, m, n_parts, woff, mem, out_bits, out_cap_words, status);
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
}

zr_status hash_bitmap_decode_launch(const int32_t* sets, const int64_t* d_set_offsets, int64_t m,
                                    int n_parts, const uint32_t* bits, int32_t* out_keys,
                                    int64_t out_cap, int64_t* d_key_offsets, void* ws,
                                    cudaStream_t stream) {
  const HbLayout L = hb_layout(m, n_parts);
  unsigned char* w = static_cast<unsigned char*>(ws);
  int32_t* status = reinterpret_cast<int32_t*>(w);
  int64_t* woff = reinterpret_cast<int64_t*>(w + L.woff);
  int32_t* tcnt = reinterpret_cast<int32_t*>(w + L.tcnt);
  int64_t* tbase = reinterpret_cast<int64_t*>(w + L.tbase);
  if (cudaMemsetAsync(w, 0, 256, stream) != cudaSuccess) return ZR_ERR_CUDA;
  // Partition p's words start where the encoder put them: the offsets follow
  // from the index sets alone (the tile count kernel derives them).
  const int64_t tiles = (words_bound(m, n_parts) + kTileWords - 1) / kTileWords;
  hb_tile_count_kernel<<<grid_for(tiles, 4), kThreads, 0, stream>>>(bits, d_set_offsets, n_parts,
                                                                   m, woff, tcnt, status);
  hb_scan_kernel<<<1, kScanThreads, 0, stream>>>(bits, woff, n_parts, tcnt, tbase, d_key_offsets,
                                                 out_cap, status);
  hb_decode_kernel<<<grid_for(tiles, 4), kThreads, 0, stream>>>(
      sets, d_set_offsets, n_parts, bits, woff, tbase, out_keys, out_cap, status);
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
}

}  // namespace zr
