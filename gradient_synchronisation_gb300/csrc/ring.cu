// Fused single-pass ring all-reduce / SkipReduce for N rank buffers held in
// one GPU's memory.
//
// What the ring computes (SkipReduce page, section 4.2, Algorithms 1 and 2;
// 15-642 notes, "Ring AllReduce"): at Reduce-Scatter step s rank r sends slice
// (r - s + o) mod N to rank r+1, which adds it to its own copy; after the last
// step rank (c - 1 - o) mod N holds slice c fully reduced, divides it, and the
// AllGather copies it to every rank.  Skipping k steps (the loop starting at
// s = k) means slice c is first sent by rank s_c = (c + k - o) mod N and
// accumulates the N - k ranks s_c, s_c+1, ... in that order.
//
// On one GPU there is no wire: every element's result depends only on its N
// inputs and its slice, so one kernel reads each non-skipped rank's element
// once (in ring order, folding in fp32 registers), divides, and stores the
// result to all N buffers.  This is bit-identical to the literal ring because
// the association order is the same left fold and fp32 addition is
// commutative (receiver-side local + received == received + local).
//
// Layout: blockIdx.y is the slice c; blockIdx.x covers the slice's 16-byte
// vectors.  The fold order is uniform per block, so the rotated
// pointer list lives in shared memory and the inner loop has no divergence.
// Slice boundaries need not fall on 16-byte vectors: the (at most VEC-1)
// elements at each end of a slice that share a vector with the next slice go
// through a scalar path taken by block x == 0.

#include <cuda_runtime.h>
#include <stdint.h>

#include "zr.h"
#include "zr_device.cuh"
#include "zr_internal.h"

namespace zr {
namespace {

struct RingParams {
  const void* bufs[ZR_MAX_RANKS];
  int64_t m;       // elements per rank
  int64_t chunk;   // C = ceil(m / n)
  int32_t n;       // ranks
  int32_t k;       // skipped Reduce-Scatter steps
  int32_t mode;    // ZR_SKIP_STATIC / ZR_SKIP_RANDOM
  int32_t div_kind;  // 0: none, 1: multiply by exact power-of-two reciprocal, 2: IEEE divide
  float div;
  float inv;
  uint64_t seed;
  uint64_t step;
};

constexpr int kThreads = 128;
constexpr int kBatch = 8;   // ranks whose loads are issued back to back before folding
constexpr int kUnroll = 2;  // vectors per thread per pass

template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kVec = 4;  // elements per 16-byte vector
  __device__ static __forceinline__ void unpack(const uint4& w, float* f) {
    f[0] = __uint_as_float(w.x); f[1] = __uint_as_float(w.y);
    f[2] = __uint_as_float(w.z); f[3] = __uint_as_float(w.w);
  }
  __device__ static __forceinline__ uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                      __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
  __device__ static __forceinline__ float load1(const void* p, int64_t e) {
    return __ldcs(static_cast<const float*>(p) + e);
  }
  __device__ static __forceinline__ void store1(void* p, int64_t e, float v) {
    __stcs(static_cast<float*>(p) + e, v);
  }
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ static __forceinline__ void unpack(const uint4& w, float* f) {
    f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
    f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z); f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
  }
  __device__ static __forceinline__ uint4 pack(const float* f) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                      pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
  }
  __device__ static __forceinline__ float load1(const void* p, int64_t e) {
    unsigned short u = __ldcs(static_cast<const unsigned short*>(p) + e);
    return __uint_as_float((uint32_t)u << 16);
  }
  __device__ static __forceinline__ void store1(void* p, int64_t e, float v) {
    __stcs(static_cast<unsigned short*>(p) + e, __bfloat16_as_ushort(__float2bfloat16_rn(v)));
  }
};

__device__ __forceinline__ float apply_div(float x, const RingParams& P) {
  if (P.div_kind == 1) return __fmul_rn(x, P.inv);   // exact: x * 2^-j == x / 2^j
  if (P.div_kind == 2) return __fdiv_rn(x, P.div);
  return x;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
ring_fused_kernel(const __grid_constant__ RingParams P) {
  using E = Elem<T>;
  constexpr int V = E::kVec;
  __shared__ const void* s_src[ZR_MAX_RANKS];
  __shared__ void* s_dst[ZR_MAX_RANKS];

  const int n = P.n;
  const int c = blockIdx.y;
  const int cnt = n - P.k;
  const int o = (P.k == 0 || P.mode == ZR_SKIP_STATIC) ? 0 : random_offset(P.seed, P.step, n);
  const int start = ((c + P.k - o) % n + n) % n;
  for (int t = threadIdx.x; t < n; t += blockDim.x) {
    int r = start + t;
    if (r >= n) r -= n;
    s_src[t] = P.bufs[r];
    s_dst[t] = const_cast<void*>(P.bufs[t]);
  }
  __syncthreads();

  const int64_t lo = (int64_t)c * P.chunk;
  const int64_t hi = min(lo + P.chunk, P.m);
  if (lo >= hi) return;
  int64_t vlo = (lo + V - 1) / V;
  int64_t vhi = hi / V;
  if (vlo > vhi) vhi = vlo;  // the whole slice sits inside one vector

  // Scalar ends: [lo, vlo*V) and [vhi*V, hi), each fewer than V elements
  // (or the whole short slice).
  if (blockIdx.x == 0) {
    int64_t a0 = lo, a1 = min(vlo * V, hi);
    int64_t b0 = max(vhi * V, a1), b1 = hi;
    int64_t na = a1 - a0;
    int64_t tot = na + max((int64_t)0, b1 - b0);
    for (int64_t i = threadIdx.x; i < tot; i += blockDim.x) {
      int64_t e = (i < na) ? a0 + i : b0 + (i - na);
      float acc = E::load1(s_src[0], e);
      for (int t = 1; t < cnt; ++t) acc = __fadd_rn(acc, E::load1(s_src[t], e));
      acc = apply_div(acc, P);
      for (int r = 0; r < n; ++r) E::store1(s_dst[r], e, acc);
    }
  }

  // Aligned vectors: each thread takes kUnroll vectors a block apart and
  // issues the loads of both (up to kUnroll x kBatch 16-byte loads) before
  // folding either, so many bytes are in flight per SM.
  const int64_t stride = (int64_t)gridDim.x * blockDim.x * kUnroll;
  for (int64_t j0 = vlo + (int64_t)blockIdx.x * blockDim.x * kUnroll + threadIdx.x; j0 < vhi;
       j0 += stride) {
    float acc[kUnroll][V];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t j = j0 + (int64_t)u * blockDim.x;
      if (j < vhi) E::unpack(__ldcs(static_cast<const uint4*>(s_src[0]) + j), acc[u]);
    }
    for (int t = 1; t < cnt; t += kBatch) {
      uint4 w[kUnroll][kBatch];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t j = j0 + (int64_t)u * blockDim.x;
#pragma unroll
        for (int b = 0; b < kBatch; ++b)
          if (t + b < cnt && j < vhi) w[u][b] = __ldcs(static_cast<const uint4*>(s_src[t + b]) + j);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          if (t + b < cnt) {
            float f[V];
            E::unpack(w[u][b], f);
#pragma unroll
            for (int q = 0; q < V; ++q) acc[u][q] = __fadd_rn(acc[u][q], f[q]);
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t j = j0 + (int64_t)u * blockDim.x;
      if (j < vhi) {
#pragma unroll
        for (int q = 0; q < V; ++q) acc[u][q] = apply_div(acc[u][q], P);
        const uint4 out = E::pack(acc[u]);
        for (int r = 0; r < n; ++r) __stcs(static_cast<uint4*>(s_dst[r]) + j, out);
      }
    }
  }
}

// Grid: blockIdx.y is the slice; blockIdx.x covers the slice's vectors with
// about 1.25 passes of kUnroll vectors per thread.  Measured on GB300 for the
// C2 shape, covering the whole slice with short-lived blocks moves more bytes
// than a one-wave persistent grid (consecutive blocks sweep consecutive
// addresses), and evict-first stores beat write-back stores by a wide margin.
template <typename T>
zr_status launch(const RingParams& P, cudaStream_t stream) {
  constexpr int V = Elem<T>::kVec;
  const int64_t vecs_per_chunk = (P.chunk + V - 1) / V;
  const int64_t per_block = (int64_t)kThreads * kUnroll;
  int64_t gx = (vecs_per_chunk * 4 + per_block * 5 - 1) / (per_block * 5);
  if (gx > 0x7fffffff) gx = 0x7fffffff;
  if (gx < 1) gx = 1;
  dim3 grid((unsigned)gx, (unsigned)P.n);
  ring_fused_kernel<T><<<grid, kThreads, 0, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
}

}  // namespace

zr_status ring_launch(void* const* bufs, int n, int64_t m, zr_dtype dt, int k, int mode,
                      uint64_t seed, uint64_t step, int divisor, cudaStream_t stream) {
  RingParams P;
  for (int r = 0; r < ZR_MAX_RANKS; ++r) P.bufs[r] = r < n ? bufs[r] : nullptr;
  P.m = m;
  P.chunk = (m + n - 1) / n;
  P.n = n;
  P.k = k;
  P.mode = mode;
  P.seed = seed;
  P.step = step;
  int d = divisor == ZR_DIV_N ? n : (divisor == ZR_DIV_N_MINUS_K ? n - k : 1);
  P.div = (float)d;
  P.inv = 1.0f;
  if (divisor == ZR_DIV_NONE || d == 1) {
    P.div_kind = 0;
  } else if ((d & (d - 1)) == 0) {
    P.div_kind = 1;
    P.inv = 1.0f / (float)d;  // exact for a power of two
  } else {
    P.div_kind = 2;
  }
  if (m == 0) return ZR_OK;
  return dt == ZR_F32 ? launch<float>(P, stream) : launch<__nv_bfloat16>(P, stream);
}

}  // namespace zr
