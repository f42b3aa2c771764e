// Internal declarations shared by the libzr translation units (not part of
// the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "zr.h"

namespace zr {

// Streaming multiprocessors on the current device (cached per device).
int sm_count();

// Dense ring all-reduce / SkipReduce launch; arguments already validated.
zr_status ring_launch(void* const* bufs, int n, int64_t m, zr_dtype dt, int k, int mode,
                      uint64_t seed, uint64_t step, int divisor, int rs_only, uint64_t drop_thr,
                      uint64_t drop_seed, uint64_t drop_step, cudaStream_t stream);

// Multi-bucket SkipReduce in one launch; arguments already validated.
zr_status ring_buckets_launch(const zr_bucket* buckets, int n_buckets, int n, zr_dtype dt,
                              cudaStream_t stream);

// Sparse aggregation; arguments already validated.
size_t sparse_workspace_bytes(int n, int64_t dense_size, int n_parts);
zr_status sparse_launch(const int32_t* const* idx, const float* const* val, const int64_t* nnz,
                        int n, int64_t dense_size, int n_parts, uint64_t part_seed, int average,
                        int32_t* out_idx, float* out_val, int64_t out_cap, int64_t* d_out_nnz,
                        int64_t* d_offsets, void* ws, cudaStream_t stream);

// Push-side partition; arguments already validated.
size_t partition_workspace_bytes(int64_t nnz, int n_parts);
zr_status partition_launch(const int32_t* idx, const float* val, int64_t nnz, int n_parts,
                           uint64_t part_seed, int32_t* out_idx, float* out_val,
                           int64_t* d_offsets, void* ws, cudaStream_t stream);

}  // namespace zr
