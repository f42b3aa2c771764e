/*
 * zr.h -- C ABI of libzr: gradient aggregation across N data-parallel ranks
 * whose buffers all live in one GPU's memory.
 *
 * Pages the operations follow (cited by title and section):
 *   [SR]  "SkipReduce: (Interconnection) Network Sparsity to Accelerate
 *         Distributed Machine Learning" (MICRO'25 digest)
 *   [ZEN] "Zen: Empowering Distributed Training with Sparsity-driven Data
 *         Synchronization" (OSDI'25 digest)
 *   [CMU] "15642 Machine Learning Systems: Distributed Training and
 *         Parallelization" (CMU course notes)
 *
 * Conventions for every entry point:
 *   - Pointers named d_* / device buffers are CUDA device pointers; arrays of
 *     pointers (bufs, idx, val) and count arrays (nnz) are HOST arrays.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call is stream-ordered and asynchronous: it validates
 *     its arguments on the host, enqueues its kernels and returns.  Nothing
 *     is copied back to the host and nothing synchronises.
 *   - The caller owns every buffer, including the workspace `ws`; the library
 *     allocates no device or host memory.
 *   - The return value reports argument errors (checked before anything is
 *     enqueued; on error nothing is enqueued and no buffer is touched) and
 *     launch errors (ZR_ERR_CUDA).  Errors found by a kernel on the device
 *     (an unsorted or out-of-range sparse index) are written to a status
 *     word inside `ws`; read it with zr_query_status after the stream work.
 *   - zr_partition, zr_partition_static and zr_hash_index_sets are each one
 *     cooperative launch whose CTAs wait for one another once.  That wait is
 *     bounded: if the CTAs cannot all run at once (for example while another
 *     cooperative grid holds the device from a stream that is not ordered
 *     with this one) it gives up after about a second, the status word
 *     becomes ZR_ERR_TIMEOUT and the outputs are unspecified.  Order such
 *     calls on one stream, or with events.  No other kernel waits on
 *     another CTA.
 *   - No C++ exception crosses this interface.
 */
#ifndef ZR_H
#define ZR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum zr_status {
  ZR_OK = 0,
  ZR_ERR_INVALID_ARG = 1,    /* a size, count, pointer or flag is out of range */
  ZR_ERR_UNSUPPORTED = 2,    /* a valid request this build does not implement */
  ZR_ERR_ALIGNMENT = 3,      /* a dense rank buffer or a workspace is not
                                16-byte aligned */
  ZR_ERR_CAPACITY = 4,       /* an output or workspace buffer is too small */
  ZR_ERR_INPUT_UNSORTED = 5, /* device-detected: sparse indices not strictly
                                ascending or outside [0, dense_size) */
  ZR_ERR_TIMEOUT = 6,        /* device-detected: a bounded wait gave up */
  ZR_ERR_CUDA = 7,           /* a CUDA runtime call or launch failed */
  ZR_ERR_INTERNAL = 8        /* device-detected: an internal consistency check
                                failed (the access was skipped) */
} zr_status;

typedef enum zr_dtype {
  ZR_F32 = 0,  /* IEEE binary32 */
  ZR_BF16 = 1  /* bfloat16: widened exactly to fp32, accumulated in fp32,
                  rounded once (round-to-nearest-even) on output */
} zr_dtype;

#define ZR_MAX_RANKS 64
#define ZR_MAX_PARTS 256

/* SkipReduce slice choice [SR section 4.2 (Static), section 4.3 (Random)]. */
typedef enum zr_skip_mode {
  ZR_SKIP_STATIC = 0, /* offset o = 0: slice c omits ranks c .. c+k-1 */
  ZR_SKIP_RANDOM = 1  /* offset o drawn from (seed, step), see zr_skip_cfg */
} zr_skip_mode;

/* What the reduced slice is divided by [SR section 4.1, and section 5's
 * SkipReduce vs DropReduce comparison]. */
typedef enum zr_divisor {
  ZR_DIV_N = 0,         /* SkipReduce average: skipped slices count as zero */
  ZR_DIV_N_MINUS_K = 1, /* DropReduce: skipped slices are removed */
  ZR_DIV_NONE = 2       /* plain sum */
} zr_divisor;

/*
 * SkipReduce configuration.
 *   mode     ZR_SKIP_STATIC or ZR_SKIP_RANDOM.
 *   k        Reduce-Scatter steps skipped, 0 <= k <= n-1 [SR Algorithm 2:
 *            the loop runs s = k .. N-2].  A skip fraction p maps to k = p*N.
 *   seed     Random mode: generator seed shared by every rank.
 *   step     Random mode: the iteration count [SR section 4.3].
 *   divisor  a zr_divisor value.
 * Random offset: o = floor(hi32(x) * n / 2^32), where x is output number
 * `step` (0-based) of SplitMix64 seeded with `seed` (Steele, Lea and Flood,
 * OOPSLA 2014): x = mix(seed + (step + 1) * 0x9E3779B97F4A7C15 mod 2^64),
 * mix(z) = z ^= z>>30; z *= 0xBF58476D1CE4E5B9; z ^= z>>27;
 *          z *= 0x94D049BB133111EB; z ^= z>>31.
 * With k = 0 the offset is 0 in both modes (p = 0 is exactly the plain ring).
 *   flags    0, or ZR_SKIP_RS_ONLY: run the Reduce-Scatter only [15-642
 *            notes, "ZeRO Stage 2": Reduce-Scatter replaces AllReduce and
 *            each GPU keeps only its own partition].  Slice c is then written
 *            only to its holder, rank (c - 1 - o) mod n, the rank where the
 *            Reduce-Scatter ends; every other element of every buffer keeps
 *            its input value.
 */
#define ZR_SKIP_RS_ONLY 1

typedef struct zr_skip_cfg {
  int32_t mode;
  int32_t k;
  uint64_t seed;
  uint64_t step;
  int32_t divisor;
  int32_t flags; /* 0 or ZR_SKIP_RS_ONLY */
} zr_skip_cfg;

/*
 * Ring all-reduce, in place [CMU "Ring AllReduce"; SR section 2 and
 * Algorithm 1 with p = 0].
 *
 * bufs     host array of n device pointers; bufs[r] is rank r's buffer of m
 *          elements of type dt, 16-byte aligned, pairwise non-overlapping.
 * n        ranks, 1 <= n <= ZR_MAX_RANKS.   m: elements per rank, >= 0.
 * average  0: every rank ends with the sum; 1: with the sum / n.
 *
 * Result, bit for bit: the tensor is cut into n slices of C = ceil(m/n)
 * elements (the last ones may be short or empty).  Element e of slice c ends,
 * on every rank, as fl(...fl(fl(g_c[e] + g_{c+1}[e]) + g_{c+2}[e]) ... +
 * g_{c+n-1}[e]) (ranks mod n; each + one fp32 RNE addition) -- the order in
 * which the Reduce-Scatter accumulates slice c, starting at the rank that
 * first sends it -- then divided by n with one fp32 RNE division when
 * average = 1, then (bf16) rounded once to bf16.  AllGather copies it to all
 * ranks.  m = 0 or n = 1 with average = 0 changes nothing.
 */
zr_status zr_ring_allreduce(void* const* bufs, int32_t n, int64_t m, zr_dtype dt,
                            int32_t average, void* stream);

/*
 * SkipReduce all-reduce, in place [SR section 4.2 Algorithm 2, section 4.3].
 *
 * Arguments as zr_ring_allreduce, plus cfg (host pointer, see zr_skip_cfg).
 * Result: slice c is folded as above but starting at rank
 * s_c = (c + k - o) mod n and over the n - k ranks s_c .. s_c+n-k-1 only;
 * the k skipped ranks' values are not read.  The divisor is n, n - k or none.
 * With k = 0 and divisor ZR_DIV_N the result equals
 * zr_ring_allreduce(average = 1) bit for bit.
 */
zr_status zr_skipreduce(void* const* bufs, int32_t n, int64_t m, zr_dtype dt,
                        const zr_skip_cfg* cfg, void* stream);

/*
 * Selective SkipReduce: several gradient buckets in one launch [SR section
 * 4.4: gradients are communicated in buckets, each its own AllReduce, so
 * each bucket can take its own skip rate -- aggressive for unimportant
 * layers, k = 0 for protected ones].
 *
 * buckets    host array of n_buckets entries, 1 <= n_buckets <=
 *            ZR_MAX_BUCKETS and n_buckets * n <= ZR_MAX_BUCKET_BUFS.
 *            Bucket b is bufs (host array of n device pointers, each
 *            16-byte aligned), m elements per rank buffer (>= 0) and its own
 *            zr_skip_cfg (mode, k, seed, step, divisor, flags), validated as
 *            for zr_skipreduce.  No two buffers of any buckets may overlap.
 * n, dt      ranks and element type, shared by every bucket.
 * Result: every bucket ends exactly as zr_skipreduce(bucket.bufs, n,
 * bucket.m, dt, &bucket.cfg) would leave it, bit for bit.  The caller gives
 * each bucket its own seed or step when buckets should skip different
 * slices.
 */
#define ZR_MAX_BUCKETS 128
#define ZR_MAX_BUCKET_BUFS 2048

typedef struct zr_bucket {
  void* const* bufs;
  int64_t m;
  zr_skip_cfg cfg;
} zr_bucket;

zr_status zr_skipreduce_buckets(const zr_bucket* buckets, int32_t n_buckets, int32_t n,
                                zr_dtype dt, void* stream);

/*
 * AllReduce_Dropout, in place [SR section 4.2, Algorithm 1 "AllReduce with
 * Fine-Grained Skipping": at every Reduce-Scatter step the receiving rank
 * skips its local gradient element with probability p, forwarding what it
 * received unchanged; the AllGather is the baseline one].
 *
 * Arguments as zr_ring_allreduce, plus:
 * threshold  T in [0, 2^32]: an element is skipped when its 32-bit draw is
 *            below T; T = ceil(p * 2^32) gives skip probability p (T = 0
 *            never skips, T = 2^32 always does).
 * seed, step generator seed shared by every rank, and the iteration count.
 * Draw of receiving rank r for element e (its index in the buffer): one
 * 32-bit half of output number floor(e / 2) of SplitMix64 seeded with
 * s_r = (output number step * 64 + r of SplitMix64 seeded with seed), the
 * high half for even e and the low half for odd e.
 * Result: slice c (as in zr_ring_allreduce) is folded from its first sender,
 * rank c, whose value is always kept; rank c + t (t = 1 .. n-1, mod n) adds
 * its value unless its draw for e is below T.  Then divided by n when
 * average = 1, (bf16) rounded once, and written to every rank.  Every rank's
 * element is read (skipping saves no traffic, as the pages note).
 */
zr_status zr_allreduce_dropout(void* const* bufs, int32_t n, int64_t m, zr_dtype dt,
                               uint64_t threshold, uint64_t seed, uint64_t step,
                               int32_t average, void* stream);

/*
 * Sparse (COO) aggregation with partitioning [ZEN section 2.1 (COO), Problem
 * 1, section 3.2 Technique #3 and Algorithm 1's first-level hash h0].
 *
 * idx, val, nnz  host arrays of n entries: rank r's list is nnz[r] entries at
 *                device pointers idx[r] (int32, strictly ascending, each in
 *                [0, dense_size)) and val[r] (fp32).  nnz[r] may be 0 (its
 *                pointers are then ignored).
 * n              ranks, 1 <= n <= ZR_MAX_RANKS.
 * dense_size     M, the dense tensor size, 1 <= M <= 2^31 - 1.
 * n_parts        partitions (servers), 0 <= n_parts <= ZR_MAX_PARTS;
 *                0 = no partitioning (plain ascending union).
 * part_seed      seed of h0.
 * average        0: sums; 1: sums divided once by n (fp32 RNE).
 * out_idx, out_val  device outputs of out_cap entries; out_cap must be at
 *                least sum(nnz) (checked here, so the kernels cannot write
 *                past it).
 * d_out_nnz      device int64: receives U, the union size.
 * d_offsets      device int64[n_parts + 1]: partition j is
 *                [d_offsets[j], d_offsets[j+1]); may be NULL if n_parts = 0.
 * ws, ws_bytes   device workspace of at least
 *                zr_sparse_workspace_size(n, dense_size, n_parts) bytes,
 *                16-byte aligned.  Its first 4 bytes are the status word.
 *
 * Result: one entry per index in the union of the n lists.  Its value is the
 * left fold, in ascending rank order, of the values of the ranks that hold
 * the index, starting from the first holder's value (fp32 RNE additions).
 * Partition of index x: h(x) = ((a*x + b) mod 2^64) >> 32,
 * p(x) = (h(x) * n_parts) >> 32, with a = (SplitMix64(part_seed) output 0) | 1
 * and b = output 1.  Entries are written partition-major, ascending index
 * inside each partition.
 * If an input list is not strictly ascending or holds an index outside
 * [0, dense_size), the status word becomes ZR_ERR_INPUT_UNSORTED and the
 * outputs are unspecified (every access still stays inside the buffers).
 */
zr_status zr_sparse_aggregate(const int32_t* const* idx, const float* const* val,
                              const int64_t* nnz, int32_t n, int64_t dense_size,
                              int32_t n_parts, uint64_t part_seed, int32_t average,
                              int32_t* out_idx, float* out_val, int64_t out_cap,
                              int64_t* d_out_nnz, int64_t* d_offsets,
                              void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes zr_sparse_aggregate needs (0 on invalid arguments).  The
 * kernels keep per-bin tables over the key range (bins of 1024 keys, wider
 * for very large dense sizes): bin starts per rank and per-bin counts and
 * positions per partition, so the size grows with dense_size * (n +
 * n_parts), not with the entry count. */
size_t zr_sparse_workspace_size(int32_t n, int64_t dense_size, int32_t n_parts);

/*
 * Push-side partition of one rank's COO list [ZEN Problem 1, requirement 1:
 * each worker splits its nonzeros into n parts with the shared h0].
 *
 * idx, val   device inputs of nnz entries (any order; indices need not be
 *            unique).  out_idx, out_val: device outputs of nnz entries.
 * d_offsets  device int64[n_parts + 1].   1 <= n_parts <= ZR_MAX_PARTS.
 * ws         device workspace of zr_partition_workspace_size(nnz, n_parts)
 *            bytes, 16-byte aligned.
 * Result: entries grouped by p(idx) (same h0 as above), partition-major; inside
 * a partition entries keep their input order (a stable split).
 */
zr_status zr_partition(const int32_t* idx, const float* val, int64_t nnz,
                       int32_t n_parts, uint64_t part_seed, int32_t* out_idx,
                       float* out_val, int64_t* d_offsets, void* ws,
                       size_t ws_bytes, void* stream);

/* Workspace bytes zr_partition needs (0 on invalid arguments); like the
 * union's, it does not grow with nnz (about 4 KB per partition). */
size_t zr_partition_workspace_size(int64_t nnz, int32_t n_parts);

/*
 * Zen's index sets [ZEN section 3.3.2 "Hash bitmap": the indices a worker
 * pushes to server p are I_p = {x in [0, M) : h0(x) = p}, computed once,
 * offline, and sorted].
 *
 * dense_size M, 1 <= M <= 2^31 - 1.   n_parts: 1 <= n_parts <= ZR_MAX_PARTS.
 * out_sets   device int32[M]: every I_p, ascending, concatenated in
 *            partition order (a permutation of 0 .. M-1).
 * d_offsets  device int64[n_parts + 1]: I_p = out_sets[d_offsets[p] ..
 *            d_offsets[p+1]).
 * ws         device workspace of zr_partition_workspace_size(M, n_parts)
 *            bytes, 16-byte aligned.
 * h0 is the partition hash of zr_sparse_aggregate (same part_seed).
 */
zr_status zr_hash_index_sets(int64_t dense_size, int32_t n_parts, uint64_t part_seed,
                             int32_t* out_sets, int64_t* d_offsets, void* ws, size_t ws_bytes,
                             void* stream);

/*
 * Zen's index sets as a directory [ZEN section 3.3.2 "Hash bitmap":
 * I_p = {x in [0, M) : h0(x) = p}, ascending, fixed for the whole run].  The
 * hash bitmap calls below use this directory instead of the index sets; it
 * is built once per (M, n_parts, part_seed), in two launches, and holds
 * NB = ceil(log2 n_parts) bits per index instead of the index sets' 32.
 *
 * dense_size M, 1 <= M <= 2^31 - 1.   n_parts: 1 <= n_parts <= ZR_MAX_PARTS.
 * d_dir      device buffer of zr_hash_directory_size(M, n_parts) bytes,
 *            16-byte aligned.  With R = ceil(M / ZR_HASH_RANGE) and S = R + 1
 *            rounded up to a multiple of 4, it holds
 *            header  256 bytes: int64 magic, M, n_parts, part_seed;
 *            counts  int32, from byte 256: entry [p S + r], r <= R, is
 *                    |{x < min(r ZR_HASH_RANGE, M) : h0(x) = p}|, so entry
 *                    [p S + R] is |I_p|;
 *            slices  uint64, from byte 256 + ceil(n_parts S 4 / 256) 256:
 *                    word [(r NB + b) 32 + l] has bit k set iff bit b of
 *                    h0(r ZR_HASH_RANGE + 64 l + k) is set (bits of indices
 *                    at or past M unspecified).
 *            The encode and decode calls read it; they report
 *            ZR_ERR_INVALID_ARG, and write nothing, for a directory built
 *            for another (M, n_parts, part_seed), and they check every
 *            range's counts against the slices.
 * h0 is the partition hash of zr_sparse_aggregate (same part_seed).
 */
#define ZR_HASH_RANGE 2048
size_t zr_hash_directory_size(int64_t dense_size, int32_t n_parts);
zr_status zr_hash_directory(int64_t dense_size, int32_t n_parts, uint64_t part_seed,
                            int32_t* d_dir, size_t dir_bytes, void* stream);

/*
 * Hash bitmap encode [ZEN section 3.3.2, Figure 10, Algorithm 2
 * hash_bitmap_encode: a server marks which elements of I_p are nonzero,
 * one bit each, so that all servers' bitmaps total |G| bits].
 *
 * d_dir                 the directory of (dense_size, n_parts, part_seed).
 * keys, n_keys   device int32: the nonzero indices (any order, each in
 *                [0, M)), e.g. the out_idx of zr_sparse_aggregate.
 * out_bits       device uint32[out_cap_words], out_cap_words >=
 *                ceil(M / 32) + n_parts.  Partition p's bitmap is
 *                ceil(|I_p| / 32) words from word d_word_offsets[p]; bit j
 *                (bit j mod 32 of word j / 32, least significant first) is 1
 *                iff I_p[j] is one of the keys; padding bits are 0.
 * d_word_offsets device int64[n_parts + 1] (output).
 * ws             device workspace of zr_hash_bitmap_workspace_size(M,
 *                n_parts) bytes, 16-byte aligned; its first 4 bytes are the
 *                status word (ZR_ERR_INPUT_UNSORTED: a key outside [0, M);
 *                ZR_ERR_INVALID_ARG: a directory that does not match h0).
 * Four launches: two memsets, the membership marks, the encode.
 */
zr_status zr_hash_bitmap_encode(const int32_t* d_dir, int64_t dense_size, int32_t n_parts,
                                uint64_t part_seed, const int32_t* keys, int64_t n_keys,
                                uint32_t* out_bits, int64_t out_cap_words,
                                int64_t* d_word_offsets, void* ws, size_t ws_bytes, void* stream);

/*
 * Hash bitmap decode [ZEN section 3.3.2, Algorithm 2 hash_bitmap_decode: a
 * worker maps the set bits j of server p's bitmap back to the indices
 * I_p[j]].
 *
 * d_dir          the directory of (dense_size, n_parts, part_seed).
 * bits           device uint32 bitmaps laid out as zr_hash_bitmap_encode
 *                writes them (partition p from word sum_{q<p} ceil(|I_q|/32));
 *                the buffer holds at least the sum_q ceil(|I_q|/32) words the
 *                directory gives (ceil(M / 32) + n_parts always suffices).
 * out_keys       device int32[out_cap]: partition-major, ascending inside a
 *                partition (the indices I_p[j] of the set bits j).
 * d_key_offsets  device int64[n_parts + 1] (output): partition p's keys are
 *                out_keys[d_key_offsets[p] .. d_key_offsets[p+1]).
 * ws             as for encode.  Status: ZR_ERR_CAPACITY if more keys than
 *                out_cap (nothing is written past it), ZR_ERR_INVALID_ARG if a
 *                padding bit is set or the directory does not match h0.
 * Four launches: the status memset, the segment counts, their scan, the
 * decode.
 */
zr_status zr_hash_bitmap_decode(const int32_t* d_dir, int64_t dense_size, int32_t n_parts,
                                uint64_t part_seed, const uint32_t* bits, int32_t* out_keys,
                                int64_t out_cap, int64_t* d_key_offsets, void* ws,
                                size_t ws_bytes, void* stream);

/* Workspace bytes zr_hash_bitmap_encode / _decode need (0 on invalid
 * arguments): the status word, an M-bit membership map and 4 bytes per
 * partition per ZR_HASH_RANGE indices. */
size_t zr_hash_bitmap_workspace_size(int64_t dense_size, int32_t n_parts);

/*
 * Densification of rank groups, measured on the device [ZEN Definition 4
 * and section 2.3: the densification ratio gamma_k of aggregating k sparse
 * tensors decides between the two optimal schemes].
 *
 * idx, nnz, n, dense_size  as zr_sparse_aggregate (values are not needed);
 *                n must be a power of two, 1 <= n <= ZR_MAX_RANKS.
 * d_union_counts device int64[log2(n) + 1] (output): entry L is the sum,
 *                over the n / 2^L groups of 2^L consecutive ranks
 *                (ranks i*2^L .. (i+1)*2^L - 1), of the size of the union of
 *                the group's index lists.  Entry 0 is sum(nnz); entry log2(n)
 *                is the size of the whole union.
 * ws, ws_bytes   device workspace of zr_densification_workspace_size(n,
 *                dense_size) bytes, 16-byte aligned; status word first
 *                (ZR_ERR_INPUT_UNSORTED as for zr_sparse_aggregate).
 */
zr_status zr_densification(const int32_t* const* idx, const int64_t* nnz, int32_t n,
                           int64_t dense_size, int64_t* d_union_counts, void* ws,
                           size_t ws_bytes, void* stream);

size_t zr_densification_workspace_size(int32_t n, int64_t dense_size);

/*
 * Zen's scheme choice [ZEN Theorem 1 and Equations (1), (2)], on the host.
 *
 * union_counts  host int64[log2(n) + 1], as zr_densification writes them.
 * gamma_k = union_counts[L] * k / union_counts[0] for k = 2^L (the mean
 * union of a k-group over the mean per-rank count).  Balanced parallelism
 * costs t_bp = 2 (n-1) (gamma_n + 1) / n, hierarchical centralisation
 * t_hc = 2 sum_{i=1}^{log2 n} gamma_{2^(i-1)} (both in units of d_G M / b).
 * gammas, t_bp, t_hc  optional host outputs (gammas has log2(n) + 1 slots).
 * Returns ZR_SCHEME_BALANCED (also on a tie) or ZR_SCHEME_HIERARCHICAL, or
 * -1 on invalid arguments (n not a power of two in [2, 64], a count < 0, or
 * union_counts[0] = 0).
 */
#define ZR_SCHEME_BALANCED 0
#define ZR_SCHEME_HIERARCHICAL 1

int32_t zr_choose_scheme(const int64_t* union_counts, int32_t n, double* gammas, double* t_bp,
                         double* t_hc);

/*
 * zr_partition without a workspace argument, for callers that cannot
 * allocate device memory (for example a gradient hook running inside a
 * framework whose caching allocator owns the device, or a service that
 * reserves all device memory at start-up).  The pages have no counterpart:
 * it exists only for such callers.
 *
 * Arguments and result are those of zr_partition minus ws / ws_bytes.  The
 * scratch is a fixed array of ZR_STATIC_SCRATCH_BYTES inside the library on
 * every device that loads it.  It holds what zr_partition_workspace_size
 * asks for at every valid nnz and n_parts (at most about 1 MiB), so every
 * valid request fits; a request that did not would return ZR_ERR_CAPACITY
 * and enqueue nothing.  The library never calls cudaMalloc or cudaFree
 * here.  The first call on a device (with that device current) looks up the
 * array's device address and keeps it for the process; make that first call
 * before any stream capture, and do not call this entry point on a device
 * after cudaDeviceReset, which can move the array.  All calls on a device
 * share the array (each call clears what must start at zero), so calls that
 * overlap on the GPU race.
 */
#define ZR_STATIC_SCRATCH_BYTES (2u << 20)
zr_status zr_partition_static(const int32_t* idx, const float* val, int64_t nnz,
                              int32_t n_parts, uint64_t part_seed, int32_t* out_idx,
                              float* out_val, int64_t* d_offsets, void* stream);

/*
 * Testing only: makes the CTA with index `cta` skip its arrival at the grid
 * wait of the next cooperative launches (zr_partition, zr_partition_static,
 * zr_hash_index_sets), so that every other CTA's
 * bounded wait runs out and the status word becomes ZR_ERR_TIMEOUT; -1 (the
 * default) turns it off.  A process-wide setting, for tests of the timeout
 * path; no GPU faults or hangs because of it.
 */
void zr_test_barrier_skip(int32_t cta);

/*
 * Read the device status word at the start of a sparse workspace: waits for
 * `stream`, copies the word to *status.  Returns ZR_ERR_CUDA if the copy
 * fails, ZR_ERR_INVALID_ARG for NULL pointers, else ZR_OK.
 */
zr_status zr_query_status(const void* ws, void* stream, int32_t* status);

/* Static English description of a status code (never NULL). */
const char* zr_status_string(zr_status s);

/* Library version string, e.g. "zr 0.1.0 sm_103a". */
const char* zr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ZR_H */
