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

// Union sizes of groups of 2^L consecutive ranks; arguments already validated.
size_t densify_workspace_bytes(int n, int64_t dense_size);
zr_status densify_launch(const int32_t* const* idx, const int64_t* nnz, int n, int64_t dense_size,
                         int64_t* d_union_counts, void* ws, cudaStream_t stream);

// Zen's index sets I_p (the partition of [0, m) by h0); same workspace as a
// partition of m entries.
zr_status index_sets_launch(int64_t m, int n_parts, uint64_t part_seed, int32_t* out_sets,
                            int64_t* d_offsets, void* ws, cudaStream_t stream);

// Zen's directory of index-set counts and the hash bitmap encode / decode;
// arguments already validated.
size_t hash_directory_bytes(int64_t m, int n_parts);
zr_status hash_directory_launch(int64_t m, int n_parts, uint64_t part_seed, int32_t* d_dir,
                                cudaStream_t stream);
size_t hash_bitmap_workspace_bytes(int64_t m, int n_parts);
zr_status hash_bitmap_encode_launch(const int32_t* d_dir, int64_t m, int n_parts,
                                    uint64_t part_seed, const int32_t* keys, int64_t n_keys,
                                    uint32_t* out_bits, int64_t out_cap_words,
                                    int64_t* d_word_offsets, void* ws, cudaStream_t stream);
zr_status hash_bitmap_decode_launch(const int32_t* d_dir, int64_t m, int n_parts,
                                    uint64_t part_seed, const uint32_t* bits, int32_t* out_keys,
                                    int64_t out_cap, int64_t* d_key_offsets, void* ws,
                                    cudaStream_t stream);

// Push-side partition; arguments already validated.
size_t partition_workspace_bytes(int64_t nnz, int n_parts);
zr_status partition_launch(const int32_t* idx, const float* val, int64_t nnz, int n_parts,
                           uint64_t part_seed, int32_t* out_idx, float* out_val,
                           int64_t* d_offsets, void* ws, cudaStream_t stream);

}  // namespace zr
