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

// One ring operation (a tensor, or one bucket of a multi-bucket launch).
struct RingJob {
  int64_t m;         // elements per rank
  int64_t chunk;     // C = ceil(m / n)
  int32_t n;         // ranks
  int32_t k;         // skipped Reduce-Scatter steps
  int32_t o;         // slice offset (Random SkipReduce), 0 <= o < n
  int32_t div_kind;  // 0: none, 1: multiply by exact power-of-two reciprocal, 2: IEEE divide
  float div;
  float inv;
  int32_t rs_only;   // 1: write slice c only to its holder, (c - 1 - o) mod n
  int32_t ptr_base;  // first of this job's n rank pointers in the pointer table
  int32_t bps;       // blocks per slice
  int32_t pad;
  uint64_t drop_thr;   // AllReduce_Dropout threshold T (0: off)
  uint64_t drop_seed;
  uint64_t drop_step;
};

struct RingParams {
  const void* bufs[ZR_MAX_RANKS];
  RingJob job;
};

struct BucketParams {
  const void* bufs[ZR_MAX_BUCKET_BUFS];
  RingJob jobs[ZR_MAX_BUCKETS];
  int32_t block_start[ZR_MAX_BUCKETS + 1];  // prefix of n * bps over the jobs
  int32_t n_jobs;
};

constexpr int kThreads = 128;
// Default shape: kBatch ranks' loads issued back to back before folding,
// kUnroll vectors per thread per pass.  Smaller folds take more vectors per
// thread, so that a thread still keeps about 256 bytes of loads in flight:
// at most 2 ranks 8 vectors, at most 4 ranks 4 vectors, 5 or 6 ranks 3.
constexpr int kBatch = 8;
constexpr int kUnroll = 2;
constexpr int kTinyFold = 2;
constexpr int kTinyBatch = 2;
constexpr int kTinyUnroll = 8;
constexpr int kSmallBatch = 4;
constexpr int kSmallUnroll = 4;
constexpr int kMediumFold = 6;
constexpr int kMediumBatch = 6;
constexpr int kMediumUnroll = 3;
constexpr int64_t kOneWaveBytes = 64ll << 20;  // one-pass shape up to this launch size

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

__device__ __forceinline__ float apply_div(float x, const RingJob& J) {
  if (J.div_kind == 1) return __fmul_rn(x, J.inv);   // exact: x * 2^-j == x / 2^j
  if (J.div_kind == 2) return __fdiv_rn(x, J.div);
  return x;
}

// AllReduce_Dropout: the draw of element e on the receiving rank with draw
// stream `stream` is one 32-bit half of SplitMix64 output e / 2 of that
// stream, the high half for even e and the low half for odd e; the element
// is skipped when the draw is below T.
__device__ __forceinline__ uint32_t drop_draw(uint64_t stream, int64_t e) {
  const uint64_t o = splitmix_output(stream, (uint64_t)e >> 1);
  return (e & 1) ? (uint32_t)o : (uint32_t)(o >> 32);
}

struct RingShared {
  const void* src[ZR_MAX_RANKS];  // fold order of the slice
  void* dst[ZR_MAX_RANKS];        // rank buffers (or the holder only)
  uint64_t stream[ZR_MAX_RANKS];  // dropout: draw stream of the t-th folded rank
};

// One block's share of slice c of job J: blocks bx = 0 .. J.bps - 1 cover
// the slice's 16-byte vectors; block 0 also takes the scalar ends.
template <typename T, bool kDrop, int kUnroll, int kBatch>
__device__ __forceinline__ void ring_slice(const void* const* bufs, const RingJob& J, int c, int bx,
                                           RingShared& S) {
  using E = Elem<T>;
  constexpr int V = E::kVec;
  const int n = J.n;
  const int cnt = n - J.k;
  const int start = ((c + J.k - J.o) % n + n) % n;
  const int holder = ((c - 1 - J.o) % n + n) % n;
  const int nd = J.rs_only ? 1 : n;
  for (int t = threadIdx.x; t < n; t += blockDim.x) {
    int r = start + t;
    if (r >= n) r -= n;
    S.src[t] = bufs[J.ptr_base + r];
    S.dst[t] = const_cast<void*>(bufs[J.ptr_base + (J.rs_only ? holder : t)]);
    if (kDrop) S.stream[t] = splitmix_output(J.drop_seed, J.drop_step * 64ull + (uint64_t)r);
  }
  __syncthreads();

  const int64_t lo = (int64_t)c * J.chunk;
  const int64_t hi = min(lo + J.chunk, J.m);
  if (lo >= hi) return;
  int64_t vlo = (lo + V - 1) / V;
  int64_t vhi = hi / V;
  if (vlo > vhi) vhi = vlo;  // the whole slice sits inside one vector

  // Scalar ends: [lo, vlo*V) and [vhi*V, hi), each fewer than V elements
  // (or the whole short slice).
  if (bx == 0) {
    int64_t a0 = lo, a1 = min(vlo * V, hi);
    int64_t b0 = max(vhi * V, a1), b1 = hi;
    int64_t na = a1 - a0;
    int64_t tot = na + max((int64_t)0, b1 - b0);
    for (int64_t i = threadIdx.x; i < tot; i += blockDim.x) {
      int64_t e = (i < na) ? a0 + i : b0 + (i - na);
      float acc = E::load1(S.src[0], e);
      for (int t = 1; t < cnt; ++t) {
        const float x = E::load1(S.src[t], e);
        if (!kDrop || (uint64_t)drop_draw(S.stream[t], e) >= J.drop_thr) acc = __fadd_rn(acc, x);
      }
      acc = apply_div(acc, J);
      for (int r = 0; r < nd; ++r) E::store1(S.dst[r], e, acc);
    }
  }

  // Aligned vectors: each thread takes kUnroll vectors a block apart and
  // issues the loads of both (up to kUnroll x kBatch 16-byte loads) before
  // folding either, so many bytes are in flight per SM.
  const int64_t stride = (int64_t)J.bps * blockDim.x * kUnroll;
  for (int64_t j0 = vlo + (int64_t)bx * blockDim.x * kUnroll + threadIdx.x; j0 < vhi;
       j0 += stride) {
    float acc[kUnroll][V];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t j = j0 + (int64_t)u * blockDim.x;
      if (j < vhi) E::unpack(__ldcs(static_cast<const uint4*>(S.src[0]) + j), acc[u]);
    }
    for (int t = 1; t < cnt; t += kBatch) {
      uint4 w[kUnroll][kBatch];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t j = j0 + (int64_t)u * blockDim.x;
#pragma unroll
        for (int b = 0; b < kBatch; ++b)
          if (t + b < cnt && j < vhi) w[u][b] = __ldcs(static_cast<const uint4*>(S.src[t + b]) + j);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t j = j0 + (int64_t)u * blockDim.x;
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          if (t + b < cnt) {
            float f[V];
            E::unpack(w[u][b], f);
            // the vector's V elements start at an even index: their draws are
            // the two halves of V / 2 consecutive outputs
            uint32_t d[V];
            if (kDrop) {
#pragma unroll
              for (int i = 0; i < V / 2; ++i) {
                const uint64_t o = splitmix_output(S.stream[t + b], (uint64_t)(j * (V / 2) + i));
                d[2 * i] = (uint32_t)(o >> 32);
                d[2 * i + 1] = (uint32_t)o;
              }
            }
#pragma unroll
            for (int q = 0; q < V; ++q) {
              if (kDrop && (uint64_t)d[q] < J.drop_thr) continue;
              acc[u][q] = __fadd_rn(acc[u][q], f[q]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t j = j0 + (int64_t)u * blockDim.x;
      if (j < vhi) {
#pragma unroll
        for (int q = 0; q < V; ++q) acc[u][q] = apply_div(acc[u][q], J);
        const uint4 out = E::pack(acc[u]);
        for (int r = 0; r < nd; ++r) __stcs(static_cast<uint4*>(S.dst[r]) + j, out);
      }
    }
  }
}

// One job: blockIdx.y is the slice, blockIdx.x the block inside it.
template <typename T, bool kDrop, int kU = kUnroll, int kB = kBatch>
__global__ void __launch_bounds__(kThreads)
ring_fused_kernel(const __grid_constant__ RingParams P) {
  __shared__ RingShared S;
  ring_slice<T, kDrop, kU, kB>(P.bufs, P.job, blockIdx.y, blockIdx.x, S);
}

// Many jobs (buckets) in one launch: block i belongs to the job whose block
// range holds it, then to slice (i - start) / bps of that job.
template <typename T>
__global__ void __launch_bounds__(kThreads)
ring_buckets_kernel(const __grid_constant__ BucketParams P) {
  __shared__ RingShared S;
  const int i = blockIdx.x;
  int lo = 0, hi = P.n_jobs - 1;
  while (lo < hi) {  // last job whose start <= i
    const int mid = (lo + hi + 1) >> 1;
    if (P.block_start[mid] <= i) lo = mid;
    else hi = mid - 1;
  }
  const RingJob& J = P.jobs[lo];
  const int local = i - P.block_start[lo];
  ring_slice<T, false, kUnroll, kBatch>(P.bufs, J, local / J.bps, local % J.bps, S);
}

// Grid: blockIdx.y is the slice; blockIdx.x covers the slice's vectors with
// about 1.25 passes of kUnroll vectors per thread.  Measured on GB300 for the
// C2 shape, covering the whole slice with short-lived blocks moves more bytes
// than a one-wave persistent grid (consecutive blocks sweep consecutive
// addresses), and evict-first stores beat write-back stores by a wide margin.
template <typename T>
int blocks_per_slice(int64_t chunk, int unroll = kUnroll) {
  constexpr int V = Elem<T>::kVec;
  const int64_t vecs_per_chunk = (chunk + V - 1) / V;
  const int64_t per_block = (int64_t)kThreads * unroll;
  int64_t gx = (vecs_per_chunk * 4 + per_block * 5 - 1) / (per_block * 5);
  if (gx > 0x7fffffff) gx = 0x7fffffff;
  if (gx < 1) gx = 1;
  return (int)gx;
}

// Fills a job from validated arguments.
RingJob make_job(int n, int64_t m, int k, int mode, uint64_t seed, uint64_t step, int divisor,
                 int rs_only) {
  RingJob J = {};
  J.m = m;
  J.chunk = (m + n - 1) / n;
  J.n = n;
  J.k = k;
  J.o = (k == 0 || mode == ZR_SKIP_STATIC) ? 0 : random_offset(seed, step, n);
  int d = divisor == ZR_DIV_N ? n : (divisor == ZR_DIV_N_MINUS_K ? n - k : 1);
  J.div = (float)d;
  J.inv = 1.0f;
  if (divisor == ZR_DIV_NONE || d == 1) {
    J.div_kind = 0;
  } else if ((d & (d - 1)) == 0) {
    J.div_kind = 1;
    J.inv = 1.0f / (float)d;  // exact for a power of two
  } else {
    J.div_kind = 2;
  }
  J.rs_only = rs_only;
  return J;
}

template <typename T>
zr_status launch_one(RingParams& P, cudaStream_t stream) {
  const int fold = P.job.n - P.job.k;  // ranks folded per element
  const int shape = fold <= kTinyFold      ? 0
                    : fold <= kSmallBatch  ? 1
                    : fold <= kMediumFold  ? 2
                                           : 3;
  const bool drop = P.job.drop_thr != 0;
  // Small launches (all rank buffers together at most kOneWaveBytes): one
  // 16-byte vector per thread and a single pass, so every load of the
  // launch is issued at once; the launch is latency-bound and this shape
  // shortens it (C1, N = 4 x 2^20 fp32: 7.1 against 8.7 us).
  constexpr int V = Elem<T>::kVec;
  if (!drop && (int64_t)P.job.n * P.job.chunk * (int64_t)sizeof(T) <= kOneWaveBytes) {
    const int64_t vpc = (P.job.chunk + V - 1) / V;
    P.job.bps = (int)((vpc + kThreads - 1) / kThreads);
    const dim3 g1((unsigned)P.job.bps, (unsigned)P.job.n);
    if (fold <= kTinyFold) ring_fused_kernel<T, false, 1, kTinyBatch><<<g1, kThreads, 0, stream>>>(P);
    else if (fold <= kSmallBatch) ring_fused_kernel<T, false, 1, kSmallBatch><<<g1, kThreads, 0, stream>>>(P);
    else if (fold <= kMediumFold) ring_fused_kernel<T, false, 1, kMediumBatch><<<g1, kThreads, 0, stream>>>(P);
    else ring_fused_kernel<T, false, 1, kBatch><<<g1, kThreads, 0, stream>>>(P);
    return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
  }
  const int unroll[4] = {kTinyUnroll, kSmallUnroll, kMediumUnroll, kUnroll};
  P.job.bps = blocks_per_slice<T>(P.job.chunk, unroll[shape]);
  dim3 grid((unsigned)P.job.bps, (unsigned)P.job.n);
  switch (shape * 2 + (drop ? 1 : 0)) {
    case 0: ring_fused_kernel<T, false, kTinyUnroll, kTinyBatch><<<grid, kThreads, 0, stream>>>(P); break;
    case 1: ring_fused_kernel<T, true, kTinyUnroll, kTinyBatch><<<grid, kThreads, 0, stream>>>(P); break;
    case 2: ring_fused_kernel<T, false, kSmallUnroll, kSmallBatch><<<grid, kThreads, 0, stream>>>(P); break;
    case 3: ring_fused_kernel<T, true, kSmallUnroll, kSmallBatch><<<grid, kThreads, 0, stream>>>(P); break;
    case 4: ring_fused_kernel<T, false, kMediumUnroll, kMediumBatch><<<grid, kThreads, 0, stream>>>(P); break;
    case 5: ring_fused_kernel<T, true, kMediumUnroll, kMediumBatch><<<grid, kThreads, 0, stream>>>(P); break;
    case 6: ring_fused_kernel<T, false><<<grid, kThreads, 0, stream>>>(P); break;
    default: ring_fused_kernel<T, true><<<grid, kThreads, 0, stream>>>(P); break;
  }
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
}

}  // namespace

zr_status ring_launch(void* const* bufs, int n, int64_t m, zr_dtype dt, int k, int mode,
                      uint64_t seed, uint64_t step, int divisor, int rs_only, uint64_t drop_thr,
                      uint64_t drop_seed, uint64_t drop_step, cudaStream_t stream) {
  RingParams P;
  for (int r = 0; r < ZR_MAX_RANKS; ++r) P.bufs[r] = r < n ? bufs[r] : nullptr;
  P.job = make_job(n, m, k, mode, seed, step, divisor, rs_only);
  P.job.drop_thr = drop_thr;
  P.job.drop_seed = drop_seed;
  P.job.drop_step = drop_step;
  if (m == 0) return ZR_OK;
  return dt == ZR_F32 ? launch_one<float>(P, stream) : launch_one<__nv_bfloat16>(P, stream);
}

zr_status ring_buckets_launch(const zr_bucket* buckets, int n_buckets, int n, zr_dtype dt,
                              cudaStream_t stream) {
  BucketParams* P = new BucketParams();  // ~27 KB: off the host stack
  int jobs = 0;
  int64_t blocks = 0;
  for (int b = 0; b < n_buckets; ++b) {
    const zr_bucket& B = buckets[b];
    if (B.m == 0) continue;
    RingJob J = make_job(n, B.m, B.cfg.k, B.cfg.mode, B.cfg.seed, B.cfg.step, B.cfg.divisor,
                         (B.cfg.flags & ZR_SKIP_RS_ONLY) ? 1 : 0);
    J.bps = dt == ZR_F32 ? blocks_per_slice<float>(J.chunk) : blocks_per_slice<__nv_bfloat16>(J.chunk);
    J.ptr_base = jobs * n;
    for (int r = 0; r < n; ++r) P->bufs[jobs * n + r] = B.bufs[r];
    P->jobs[jobs] = J;
    P->block_start[jobs] = (int32_t)blocks;
    blocks += (int64_t)J.bps * n;
    ++jobs;
  }
  if (jobs == 0) {
    delete P;
    return ZR_OK;
  }
  if (blocks > 0x7fffffff) {
    delete P;
    return ZR_ERR_UNSUPPORTED;
  }
  P->block_start[jobs] = (int32_t)blocks;
  P->n_jobs = jobs;
  if (dt == ZR_F32) ring_buckets_kernel<float><<<(unsigned)blocks, kThreads, 0, stream>>>(*P);
  else ring_buckets_kernel<__nv_bfloat16><<<(unsigned)blocks, kThreads, 0, stream>>>(*P);
  delete P;
  return cudaGetLastError() == cudaSuccess ? ZR_OK : ZR_ERR_CUDA;
}

}  // namespace zr
