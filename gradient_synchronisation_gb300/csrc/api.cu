// libzr C ABI: argument validation, status mapping and dispatch to the
// kernels in ring.cu, sparse.cu, partition.cu and hashbitmap.cu.  Every check here runs on the host before
// anything is enqueued; a failed check returns without touching any buffer.

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <utility>
#include <atomic>
#include <vector>

#include "zr.h"
#include "zr_internal.h"

namespace zr {

int sm_count() {
  static std::atomic<int> cached[64];  // 0 until first asked; any thread may fill it
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  const int c = cached[dev].load(std::memory_order_relaxed);
  if (c > 0) return c;
  int s = 0;
  if (cudaDeviceGetAttribute(&s, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || s <= 0)
    s = 148;
  cached[dev].store(s, std::memory_order_relaxed);
  return s;
}

namespace {

size_t elem_size(zr_dtype dt) { return dt == ZR_F32 ? 4 : 2; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Dense rank buffers: present, aligned, pairwise disjoint.
zr_status check_dense(void* const* bufs, int32_t n, int64_t m, zr_dtype dt) {
  if (!bufs || n < 1 || n > ZR_MAX_RANKS || m < 0) return ZR_ERR_INVALID_ARG;
  if (dt != ZR_F32 && dt != ZR_BF16) return ZR_ERR_INVALID_ARG;
  if (m > (INT64_MAX / 16)) return ZR_ERR_INVALID_ARG;
  if (m == 0) return ZR_OK;
  const uint64_t bytes = (uint64_t)m * elem_size(dt);
  std::vector<std::pair<uintptr_t, int>> spans;
  for (int r = 0; r < n; ++r) {
    if (!bufs[r]) return ZR_ERR_INVALID_ARG;
    if (!aligned16(bufs[r])) return ZR_ERR_ALIGNMENT;
    spans.emplace_back(reinterpret_cast<uintptr_t>(bufs[r]), r);
  }
  std::sort(spans.begin(), spans.end());
  for (size_t i = 1; i < spans.size(); ++i)
    if (spans[i].first - spans[i - 1].first < bytes) return ZR_ERR_INVALID_ARG;  // overlap
  return ZR_OK;
}

zr_status check_cfg(const zr_skip_cfg* cfg, int32_t n) {
  if (!cfg) return ZR_ERR_INVALID_ARG;
  if (cfg->mode != ZR_SKIP_STATIC && cfg->mode != ZR_SKIP_RANDOM) return ZR_ERR_INVALID_ARG;
  if (cfg->k < 0 || cfg->k > n - 1) return ZR_ERR_INVALID_ARG;
  if (cfg->divisor != ZR_DIV_N && cfg->divisor != ZR_DIV_N_MINUS_K && cfg->divisor != ZR_DIV_NONE)
    return ZR_ERR_INVALID_ARG;
  if ((cfg->flags & ~ZR_SKIP_RS_ONLY) != 0) return ZR_ERR_INVALID_ARG;
  return ZR_OK;
}

zr_status check_ws(const void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return ZR_ERR_INVALID_ARG;
  if (!aligned16(ws)) return ZR_ERR_ALIGNMENT;
  return ws_bytes >= need ? ZR_OK : ZR_ERR_CAPACITY;
}

}  // namespace
}  // namespace zr

extern "C" {

zr_status zr_ring_allreduce(void* const* bufs, int32_t n, int64_t m, zr_dtype dt,
                            int32_t average, void* stream) {
  zr_status st = zr::check_dense(bufs, n, m, dt);
  if (st != ZR_OK) return st;
  if (average != 0 && average != 1) return ZR_ERR_INVALID_ARG;
  if (m == 0) return ZR_OK;
  return zr::ring_launch(bufs, n, m, dt, 0, ZR_SKIP_STATIC, 0, 0,
                         average ? ZR_DIV_N : ZR_DIV_NONE, 0, 0, 0, 0,
                         static_cast<cudaStream_t>(stream));
}

zr_status zr_skipreduce(void* const* bufs, int32_t n, int64_t m, zr_dtype dt,
                        const zr_skip_cfg* cfg, void* stream) {
  zr_status st = zr::check_dense(bufs, n, m, dt);
  if (st != ZR_OK) return st;
  st = zr::check_cfg(cfg, n);
  if (st != ZR_OK) return st;
  if (m == 0) return ZR_OK;
  return zr::ring_launch(bufs, n, m, dt, cfg->k, cfg->mode, cfg->seed, cfg->step, cfg->divisor,
                         (cfg->flags & ZR_SKIP_RS_ONLY) ? 1 : 0, 0, 0, 0,
                         static_cast<cudaStream_t>(stream));
}

zr_status zr_skipreduce_buckets(const zr_bucket* buckets, int32_t n_buckets, int32_t n,
                                zr_dtype dt, void* stream) {
  if (!buckets || n_buckets < 1 || n_buckets > ZR_MAX_BUCKETS) return ZR_ERR_INVALID_ARG;
  if (n < 1 || n > ZR_MAX_RANKS || (int64_t)n_buckets * n > ZR_MAX_BUCKET_BUFS)
    return ZR_ERR_INVALID_ARG;
  // Every bucket as zr_skipreduce would check it, then no overlap between
  // the buffers of different buckets (one launch writes them all).
  std::vector<std::pair<uintptr_t, uintptr_t>> spans;
  for (int b = 0; b < n_buckets; ++b) {
    const zr_bucket& B = buckets[b];
    zr_status st = zr::check_dense(B.bufs, n, B.m, dt);
    if (st != ZR_OK) return st;
    st = zr::check_cfg(&B.cfg, n);
    if (st != ZR_OK) return st;
    if (B.m == 0) continue;
    const uintptr_t bytes = (uintptr_t)B.m * zr::elem_size(dt);
    for (int r = 0; r < n; ++r) {
      const uintptr_t a = reinterpret_cast<uintptr_t>(B.bufs[r]);
      spans.emplace_back(a, a + bytes);
    }
  }
  std::sort(spans.begin(), spans.end());
  for (size_t i = 1; i < spans.size(); ++i)
    if (spans[i].first < spans[i - 1].second) return ZR_ERR_INVALID_ARG;  // overlap
  return zr::ring_buckets_launch(buckets, n_buckets, n, dt, static_cast<cudaStream_t>(stream));
}

zr_status zr_allreduce_dropout(void* const* bufs, int32_t n, int64_t m, zr_dtype dt,
                               uint64_t threshold, uint64_t seed, uint64_t step,
                               int32_t average, void* stream) {
  zr_status st = zr::check_dense(bufs, n, m, dt);
  if (st != ZR_OK) return st;
  if (average != 0 && average != 1) return ZR_ERR_INVALID_ARG;
  if (threshold > (1ull << 32)) return ZR_ERR_INVALID_ARG;
  if (m == 0) return ZR_OK;
  return zr::ring_launch(bufs, n, m, dt, 0, ZR_SKIP_STATIC, 0, 0,
                         average ? ZR_DIV_N : ZR_DIV_NONE, 0, threshold, seed, step,
                         static_cast<cudaStream_t>(stream));
}

zr_status zr_hash_index_sets(int64_t dense_size, int32_t n_parts, uint64_t part_seed,
                             int32_t* out_sets, int64_t* d_offsets, void* ws, size_t ws_bytes,
                             void* stream) {
  if (dense_size < 1 || dense_size > INT32_MAX) return ZR_ERR_INVALID_ARG;
  if (n_parts < 1 || n_parts > ZR_MAX_PARTS || !out_sets || !d_offsets) return ZR_ERR_INVALID_ARG;
  zr_status st = zr::check_ws(ws, ws_bytes, zr::partition_workspace_bytes(dense_size, n_parts));
  if (st != ZR_OK) return st;
  return zr::index_sets_launch(dense_size, n_parts, part_seed, out_sets, d_offsets, ws,
                               static_cast<cudaStream_t>(stream));
}

size_t zr_hash_directory_size(int64_t dense_size, int32_t n_parts) {
  if (dense_size < 1 || dense_size > INT32_MAX || n_parts < 1 || n_parts > ZR_MAX_PARTS) return 0;
  return zr::hash_directory_bytes(dense_size, n_parts);
}

zr_status zr_hash_directory(int64_t dense_size, int32_t n_parts, uint64_t part_seed,
                            int32_t* d_dir, size_t dir_bytes, void* stream) {
  if (dense_size < 1 || dense_size > INT32_MAX || n_parts < 1 || n_parts > ZR_MAX_PARTS || !d_dir)
    return ZR_ERR_INVALID_ARG;
  zr_status st = zr::check_ws(d_dir, dir_bytes, zr::hash_directory_bytes(dense_size, n_parts));
  if (st != ZR_OK) return st;
  return zr::hash_directory_launch(dense_size, n_parts, part_seed, d_dir,
                                   static_cast<cudaStream_t>(stream));
}

size_t zr_hash_bitmap_workspace_size(int64_t dense_size, int32_t n_parts) {
  if (dense_size < 1 || dense_size > INT32_MAX || n_parts < 1 || n_parts > ZR_MAX_PARTS) return 0;
  return zr::hash_bitmap_workspace_bytes(dense_size, n_parts);
}

zr_status zr_hash_bitmap_encode(const int32_t* d_dir, int64_t dense_size, int32_t n_parts,
                                uint64_t part_seed, const int32_t* keys, int64_t n_keys,
                                uint32_t* out_bits, int64_t out_cap_words,
                                int64_t* d_word_offsets, void* ws, size_t ws_bytes, void* stream) {
  if (dense_size < 1 || dense_size > INT32_MAX || n_parts < 1 || n_parts > ZR_MAX_PARTS)
    return ZR_ERR_INVALID_ARG;
  if (!d_dir || !out_bits || !d_word_offsets || n_keys < 0 || (n_keys > 0 && !keys))
    return ZR_ERR_INVALID_ARG;
  if (out_cap_words < (dense_size + 31) / 32 + n_parts) return ZR_ERR_CAPACITY;
  zr_status st = zr::check_ws(ws, ws_bytes, zr::hash_bitmap_workspace_bytes(dense_size, n_parts));
  if (st != ZR_OK) return st;
  return zr::hash_bitmap_encode_launch(d_dir, dense_size, n_parts, part_seed, keys, n_keys,
                                       out_bits, out_cap_words, d_word_offsets, ws,
                                       static_cast<cudaStream_t>(stream));
}

zr_status zr_hash_bitmap_decode(const int32_t* d_dir, int64_t dense_size, int32_t n_parts,
                                uint64_t part_seed, const uint32_t* bits, int32_t* out_keys,
                                int64_t out_cap, int64_t* d_key_offsets, void* ws,
                                size_t ws_bytes, void* stream) {
  if (dense_size < 1 || dense_size > INT32_MAX || n_parts < 1 || n_parts > ZR_MAX_PARTS)
    return ZR_ERR_INVALID_ARG;
  if (!d_dir || !bits || !d_key_offsets || out_cap < 0 || (out_cap > 0 && !out_keys))
    return ZR_ERR_INVALID_ARG;
  zr_status st = zr::check_ws(ws, ws_bytes, zr::hash_bitmap_workspace_bytes(dense_size, n_parts));
  if (st != ZR_OK) return st;
  return zr::hash_bitmap_decode_launch(d_dir, dense_size, n_parts, part_seed, bits, out_keys,
                                       out_cap, d_key_offsets, ws,
                                       static_cast<cudaStream_t>(stream));
}

size_t zr_densification_workspace_size(int32_t n, int64_t dense_size) {
  if (n < 1 || n > ZR_MAX_RANKS || (n & (n - 1)) != 0 || dense_size < 1 || dense_size > INT32_MAX)
    return 0;
  return zr::densify_workspace_bytes(n, dense_size);
}

zr_status zr_densification(const int32_t* const* idx, const int64_t* nnz, int32_t n,
                           int64_t dense_size, int64_t* d_union_counts, void* ws,
                           size_t ws_bytes, void* stream) {
  if (!idx || !nnz || !d_union_counts) return ZR_ERR_INVALID_ARG;
  if (n < 1 || n > ZR_MAX_RANKS || (n & (n - 1)) != 0) return ZR_ERR_INVALID_ARG;
  if (dense_size < 1 || dense_size > INT32_MAX) return ZR_ERR_INVALID_ARG;
  for (int r = 0; r < n; ++r) {
    if (nnz[r] < 0 || nnz[r] > dense_size) return ZR_ERR_INVALID_ARG;
    if (nnz[r] > 0 && !idx[r]) return ZR_ERR_INVALID_ARG;
  }
  zr_status st = zr::check_ws(ws, ws_bytes, zr::densify_workspace_bytes(n, dense_size));
  if (st != ZR_OK) return st;
  return zr::densify_launch(idx, nnz, n, dense_size, d_union_counts, ws,
                            static_cast<cudaStream_t>(stream));
}

int32_t zr_choose_scheme(const int64_t* union_counts, int32_t n, double* gammas, double* t_bp,
                         double* t_hc) {
  if (!union_counts || n < 2 || n > ZR_MAX_RANKS || (n & (n - 1)) != 0) return -1;
  int logn = 0;
  while ((1 << logn) < n) ++logn;
  if (union_counts[0] <= 0) return -1;
  double g[7];
  for (int level = 0; level <= logn; ++level) {
    if (union_counts[level] < 0) return -1;
    g[level] = (double)union_counts[level] * (double)(1 << level) / (double)union_counts[0];
    if (gammas) gammas[level] = g[level];
  }
  const double bp = 2.0 * (n - 1) * (g[logn] + 1.0) / n;
  double hc = 0.0;
  for (int i = 1; i <= logn; ++i) hc += g[i - 1];
  hc *= 2.0;
  if (t_bp) *t_bp = bp;
  if (t_hc) *t_hc = hc;
  return bp <= hc ? ZR_SCHEME_BALANCED : ZR_SCHEME_HIERARCHICAL;
}

size_t zr_sparse_workspace_size(int32_t n, int64_t dense_size, int32_t n_parts) {
  if (n < 1 || n > ZR_MAX_RANKS || dense_size < 1 || dense_size > INT32_MAX || n_parts < 0 ||
      n_parts > ZR_MAX_PARTS)
    return 0;
  return zr::sparse_workspace_bytes(n, dense_size, n_parts);
}

zr_status zr_sparse_aggregate(const int32_t* const* idx, const float* const* val,
                              const int64_t* nnz, int32_t n, int64_t dense_size,
                              int32_t n_parts, uint64_t part_seed, int32_t average,
                              int32_t* out_idx, float* out_val, int64_t out_cap,
                              int64_t* d_out_nnz, int64_t* d_offsets, void* ws, size_t ws_bytes,
                              void* stream) {
  if (!idx || !val || !nnz || n < 1 || n > ZR_MAX_RANKS) return ZR_ERR_INVALID_ARG;
  if (dense_size < 1 || dense_size > INT32_MAX) return ZR_ERR_INVALID_ARG;
  if (n_parts < 0 || n_parts > ZR_MAX_PARTS) return ZR_ERR_INVALID_ARG;
  if (average != 0 && average != 1) return ZR_ERR_INVALID_ARG;
  if (!d_out_nnz || (n_parts > 0 && !d_offsets)) return ZR_ERR_INVALID_ARG;
  int64_t total = 0;
  for (int r = 0; r < n; ++r) {
    if (nnz[r] < 0 || nnz[r] > INT32_MAX - 1) return ZR_ERR_INVALID_ARG;
    if (nnz[r] > 0 && (!idx[r] || !val[r])) return ZR_ERR_INVALID_ARG;
    total += nnz[r];
  }
  if (total > 0 && (!out_idx || !out_val)) return ZR_ERR_INVALID_ARG;
  if (out_cap < total) return ZR_ERR_CAPACITY;
  zr_status st = zr::check_ws(ws, ws_bytes, zr::sparse_workspace_bytes(n, dense_size, n_parts));
  if (st != ZR_OK) return st;
  return zr::sparse_launch(idx, val, nnz, n, dense_size, n_parts, part_seed, average, out_idx,
                           out_val, out_cap, d_out_nnz, d_offsets, ws,
                           static_cast<cudaStream_t>(stream));
}

size_t zr_partition_workspace_size(int64_t nnz, int32_t n_parts) {
  if (nnz < 0 || nnz > INT32_MAX || n_parts < 1 || n_parts > ZR_MAX_PARTS) return 0;
  return zr::partition_workspace_bytes(nnz, n_parts);
}

zr_status zr_partition(const int32_t* idx, const float* val, int64_t nnz, int32_t n_parts,
                       uint64_t part_seed, int32_t* out_idx, float* out_val, int64_t* d_offsets,
                       void* ws, size_t ws_bytes, void* stream) {
  if (nnz < 0 || nnz > INT32_MAX || n_parts < 1 || n_parts > ZR_MAX_PARTS || !d_offsets)
    return ZR_ERR_INVALID_ARG;
  if (nnz > 0 && (!idx || !val || !out_idx || !out_val)) return ZR_ERR_INVALID_ARG;
  zr_status st = zr::check_ws(ws, ws_bytes, zr::partition_workspace_bytes(nnz, n_parts));
  if (st != ZR_OK) return st;
  return zr::partition_launch(idx, val, nnz, n_parts, part_seed, out_idx, out_val, d_offsets, ws,
                              static_cast<cudaStream_t>(stream));
}

zr_status zr_query_status(const void* ws, void* stream, int32_t* status) {
  if (!ws || !status) return ZR_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(status, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return ZR_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return ZR_ERR_CUDA;
  return ZR_OK;
}

const char* zr_status_string(zr_status s) {
  switch (s) {
    case ZR_OK: return "ok";
    case ZR_ERR_INVALID_ARG: return "invalid argument";
    case ZR_ERR_UNSUPPORTED: return "unsupported";
    case ZR_ERR_ALIGNMENT: return "buffer not 16-byte aligned";
    case ZR_ERR_CAPACITY: return "output or workspace too small";
    case ZR_ERR_INPUT_UNSORTED: return "sparse indices not strictly ascending or out of range";
    case ZR_ERR_TIMEOUT: return "device wait timed out";
    case ZR_ERR_CUDA: return "CUDA error";
    case ZR_ERR_INTERNAL: return "internal consistency check failed on the device";
  }
  return "unknown status";
}

const char* zr_version(void) { return "zr 0.1.0 sm_103a"; }

}  // extern "C"
