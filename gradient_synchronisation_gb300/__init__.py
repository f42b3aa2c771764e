"""gradient_synchronisation_gb300 -- Python binding of libzr (``include/zr.h``).

Gradient aggregation across N data-parallel ranks whose buffers all live in
one GPU's memory: the ring all-reduce with SkipReduce slice skipping and the
fused average (dense), and the Zen-style COO union with rank-ordered sums and
the h0 partition (sparse).  Every step runs in the library's CUDA kernels;
this module only marshals arguments (pointers, sizes, the stream handle) into
the C ABI.  There is no CPU fallback: the library is loaded on the first call,
and if ``libzr.so`` has not been built that call raises ImportError.  (Loading
lazily lets ``gradient_synchronisation_gb300._build`` run before the library
exists.)

Two layers:

* ``zr_ring_allreduce``, ``zr_skipreduce``, ``zr_skipreduce_buckets``,
  ``zr_allreduce_dropout``, ``zr_sparse_aggregate``, ``zr_partition``,
  ``zr_query_status`` ... -- the C entry points under their own names, taking
  integers for pointers and streams; they return the ``zr_status`` code.
* ``ring_allreduce``, ``skipreduce``, ``skipreduce_buckets``,
  ``allreduce_dropout``, ``sparse_aggregate``, ``partition`` -- the same calls
  taking torch CUDA tensors, raising ``ZrError`` on a non-OK status.  PyTorch
  supplies device memory and the current stream only.
"""

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libzr.so")

ZR_OK = 0
ZR_ERR_INVALID_ARG = 1
ZR_ERR_UNSUPPORTED = 2
ZR_ERR_ALIGNMENT = 3
ZR_ERR_CAPACITY = 4
ZR_ERR_INPUT_UNSORTED = 5
ZR_ERR_TIMEOUT = 6
ZR_ERR_CUDA = 7
ZR_ERR_INTERNAL = 8

ZR_F32 = 0
ZR_BF16 = 1
ZR_SKIP_STATIC = 0
ZR_SKIP_RANDOM = 1
ZR_DIV_N = 0
ZR_DIV_N_MINUS_K = 1
ZR_DIV_NONE = 2
ZR_MAX_RANKS = 64
ZR_MAX_PARTS = 256
ZR_HASH_RANGE = 2048
ZR_SKIP_RS_ONLY = 1
ZR_MAX_BUCKETS = 128
ZR_MAX_BUCKET_BUFS = 2048

EXPORTS = (
    "zr_ring_allreduce", "zr_skipreduce", "zr_sparse_aggregate", "zr_sparse_workspace_size",
    "zr_partition", "zr_partition_workspace_size", "zr_query_status", "zr_status_string",
    "zr_version", "zr_partition_static", "zr_skipreduce_buckets", "zr_allreduce_dropout",
    "zr_hash_index_sets", "zr_hash_directory", "zr_hash_directory_size",
    "zr_hash_bitmap_encode", "zr_hash_bitmap_decode",
    "zr_hash_bitmap_workspace_size", "zr_densification", "zr_densification_workspace_size",
    "zr_choose_scheme", "zr_test_barrier_skip",
)
ZR_SCHEME_BALANCED = 0
ZR_SCHEME_HIERARCHICAL = 1
ZR_STATIC_SCRATCH_BYTES = 2 << 20


class ZrError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, status_string(status), status))


class SkipCfg(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("k", ctypes.c_int32), ("seed", ctypes.c_uint64),
                ("step", ctypes.c_uint64), ("divisor", ctypes.c_int32),
                ("flags", ctypes.c_int32)]


class Bucket(ctypes.Structure):
    _fields_ = [("bufs", ctypes.POINTER(ctypes.c_void_p)), ("m", ctypes.c_int64),
                ("cfg", SkipCfg)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libzr.so is not built (%s); run gradient_synchronisation_gb300._build.build()"
                          % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    i32, i64, u64, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
    PP = ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "zr_ring_allreduce": (i32, [PP, i32, i64, i32, i32, P]),
        "zr_skipreduce": (i32, [PP, i32, i64, i32, ctypes.POINTER(SkipCfg), P]),
        "zr_sparse_aggregate": (i32, [PP, PP, ctypes.POINTER(i64), i32, i64, i32, u64, i32, P, P,
                                      i64, P, P, P, sz, P]),
        "zr_sparse_workspace_size": (sz, [i32, i64, i32]),
        "zr_partition": (i32, [P, P, i64, i32, u64, P, P, P, P, sz, P]),
        "zr_partition_workspace_size": (sz, [i64, i32]),
        "zr_query_status": (i32, [P, P, ctypes.POINTER(i32)]),
        "zr_status_string": (ctypes.c_char_p, [i32]),
        "zr_version": (ctypes.c_char_p, []),
        "zr_partition_static": (i32, [P, P, i64, i32, u64, P, P, P, P]),
        "zr_skipreduce_buckets": (i32, [ctypes.POINTER(Bucket), i32, i32, i32, P]),
        "zr_allreduce_dropout": (i32, [PP, i32, i64, i32, u64, u64, u64, i32, P]),
        "zr_hash_index_sets": (i32, [i64, i32, u64, P, P, P, sz, P]),
        "zr_hash_directory": (i32, [i64, i32, u64, P, sz, P]),
        "zr_hash_directory_size": (sz, [i64, i32]),
        "zr_hash_bitmap_encode": (i32, [P, i64, i32, u64, P, i64, P, i64, P, P, sz, P]),
        "zr_hash_bitmap_decode": (i32, [P, i64, i32, u64, P, P, i64, P, P, sz, P]),
        "zr_hash_bitmap_workspace_size": (sz, [i64, i32]),
        "zr_densification": (i32, [PP, ctypes.POINTER(i64), i32, i64, P, P, sz, P]),
        "zr_densification_workspace_size": (sz, [i32, i64]),
        "zr_test_barrier_skip": (None, [i32]),
        "zr_choose_scheme": (i32, [ctypes.POINTER(i64), i32, ctypes.POINTER(ctypes.c_double),
                                   ctypes.POINTER(ctypes.c_double),
                                   ctypes.POINTER(ctypes.c_double)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib_handle = None


def lib():
    """The loaded libzr (ctypes.CDLL); loads it on first use."""
    global _lib_handle
    if _lib_handle is None:
        _lib_handle = _load()
    return _lib_handle


def _ptrs(values):
    arr = (ctypes.c_void_p * max(1, len(values)))()
    for i, v in enumerate(values):
        arr[i] = v
    return arr


# ------------------------------------------------------------ C entry points
def zr_ring_allreduce(bufs, n, m, dtype, average, stream):
    return lib().zr_ring_allreduce(_ptrs(bufs), n, m, dtype, average, stream)


def zr_skipreduce(bufs, n, m, dtype, cfg, stream):
    return lib().zr_skipreduce(_ptrs(bufs), n, m, dtype, ctypes.byref(cfg), stream)


def zr_skipreduce_buckets(buckets, n, dtype, stream):
    """``buckets``: list of (list of n pointers, m, SkipCfg)."""
    arr = (Bucket * max(1, len(buckets)))()
    keep = []
    for i, (bufs, m, cfg) in enumerate(buckets):
        p = _ptrs(bufs)
        keep.append(p)
        arr[i].bufs = ctypes.cast(p, ctypes.POINTER(ctypes.c_void_p))
        arr[i].m = m
        arr[i].cfg = cfg
    return lib().zr_skipreduce_buckets(arr, len(buckets), n, dtype, stream)


def zr_allreduce_dropout(bufs, n, m, dtype, threshold, seed, step, average, stream):
    return lib().zr_allreduce_dropout(_ptrs(bufs), n, m, dtype, threshold, seed, step, average,
                                      stream)


def zr_hash_index_sets(dense_size, n_parts, part_seed, out_sets, d_offsets, ws, ws_bytes, stream):
    return lib().zr_hash_index_sets(dense_size, n_parts, part_seed, out_sets, d_offsets, ws,
                                    ws_bytes, stream)


def zr_hash_directory_size(dense_size, n_parts):
    return lib().zr_hash_directory_size(dense_size, n_parts)


def zr_hash_directory(dense_size, n_parts, part_seed, d_dir, dir_bytes, stream):
    return lib().zr_hash_directory(dense_size, n_parts, part_seed, d_dir, dir_bytes, stream)


def zr_hash_bitmap_workspace_size(dense_size, n_parts):
    return lib().zr_hash_bitmap_workspace_size(dense_size, n_parts)


def zr_hash_bitmap_encode(d_dir, dense_size, n_parts, part_seed, keys, n_keys, out_bits,
                          out_cap_words, d_word_offsets, ws, ws_bytes, stream):
    return lib().zr_hash_bitmap_encode(d_dir, dense_size, n_parts, part_seed, keys, n_keys,
                                       out_bits, out_cap_words, d_word_offsets, ws, ws_bytes,
                                       stream)


def zr_hash_bitmap_decode(d_dir, dense_size, n_parts, part_seed, bits, out_keys, out_cap,
                          d_key_offsets, ws, ws_bytes, stream):
    return lib().zr_hash_bitmap_decode(d_dir, dense_size, n_parts, part_seed, bits, out_keys,
                                       out_cap, d_key_offsets, ws, ws_bytes, stream)


def zr_densification(idx, nnz, n, dense_size, d_union_counts, ws, ws_bytes, stream):
    nnz_arr = (ctypes.c_int64 * max(1, len(nnz)))(*nnz)
    return lib().zr_densification(_ptrs(idx), nnz_arr, n, dense_size, d_union_counts, ws,
                                  ws_bytes, stream)


def zr_densification_workspace_size(n, dense_size):
    return lib().zr_densification_workspace_size(n, dense_size)


def zr_choose_scheme(union_counts, n):
    """Host call: returns (choice, gammas, t_bp, t_hc); choice -1 on invalid
    arguments."""
    levels = max(1, len(union_counts))
    uc = (ctypes.c_int64 * levels)(*union_counts)
    g = (ctypes.c_double * 8)()
    bp, hc = ctypes.c_double(0), ctypes.c_double(0)
    choice = lib().zr_choose_scheme(uc, n, g, ctypes.byref(bp), ctypes.byref(hc))
    return choice, list(g)[:len(union_counts)], bp.value, hc.value


def zr_sparse_aggregate(idx, val, nnz, n, dense_size, n_parts, part_seed, average, out_idx,
                        out_val, out_cap, d_out_nnz, d_offsets, ws, ws_bytes, stream):
    nnz_arr = (ctypes.c_int64 * max(1, len(nnz)))(*nnz)
    return lib().zr_sparse_aggregate(_ptrs(idx), _ptrs(val), nnz_arr, n, dense_size, n_parts,
                                    part_seed, average, out_idx, out_val, out_cap, d_out_nnz,
                                    d_offsets, ws, ws_bytes, stream)


def zr_sparse_workspace_size(n, dense_size, n_parts):
    return lib().zr_sparse_workspace_size(n, dense_size, n_parts)


def zr_test_barrier_skip(cta):
    """Testing only: the CTA ``cta`` skips its grid-wait arrival (-1: off)."""
    lib().zr_test_barrier_skip(cta)


def zr_partition(idx, val, nnz, n_parts, part_seed, out_idx, out_val, d_offsets, ws, ws_bytes,
                 stream):
    return lib().zr_partition(idx, val, nnz, n_parts, part_seed, out_idx, out_val, d_offsets, ws,
                             ws_bytes, stream)


def zr_partition_static(idx, val, nnz, n_parts, part_seed, out_idx, out_val, d_offsets, stream):
    """zr_partition with the library's own fixed scratch (no workspace)."""
    return lib().zr_partition_static(idx, val, nnz, n_parts, part_seed, out_idx, out_val,
                                     d_offsets, stream)


def zr_partition_workspace_size(nnz, n_parts):
    return lib().zr_partition_workspace_size(nnz, n_parts)


def zr_query_status(ws, stream):
    out = ctypes.c_int32(-1)
    st = lib().zr_query_status(ws, stream, ctypes.byref(out))
    if st != ZR_OK:
        raise ZrError(st, "zr_query_status")
    return out.value


def status_string(status):
    return lib().zr_status_string(status).decode()


def version():
    return lib().zr_version().decode()


# ------------------------------------------------------------ torch wrappers
def _stream(stream):
    import torch

    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _dtype_code(t):
    import torch

    if t.dtype == torch.float32:
        return ZR_F32
    if t.dtype == torch.bfloat16:
        return ZR_BF16
    raise TypeError("dense buffers must be float32 or bfloat16, got %s" % t.dtype)


def _check(st, where):
    if st != ZR_OK:
        raise ZrError(st, where)


def _dense_args(bufs):
    if len(bufs) == 0:
        raise ValueError("need at least one rank buffer")
    m = bufs[0].numel()
    dt = _dtype_code(bufs[0])
    for b in bufs:
        if not b.is_cuda or not b.is_contiguous() or b.numel() != m or _dtype_code(b) != dt:
            raise ValueError("rank buffers must be contiguous CUDA tensors of one size and dtype")
    return [b.data_ptr() for b in bufs], len(bufs), m, dt


def ring_allreduce(bufs, average=True, stream=None):
    """In-place ring all-reduce of the rank buffers ``bufs`` (list of tensors)."""
    ptrs, n, m, dt = _dense_args(bufs)
    _check(zr_ring_allreduce(ptrs, n, m, dt, 1 if average else 0, _stream(stream)),
           "zr_ring_allreduce")


def skipreduce(bufs, k, mode=ZR_SKIP_RANDOM, seed=0, step=0, divisor=ZR_DIV_N, rs_only=False,
               stream=None):
    """In-place SkipReduce all-reduce skipping ``k`` Reduce-Scatter steps
    (``rs_only``: Reduce-Scatter only, each slice written to its holder)."""
    ptrs, n, m, dt = _dense_args(bufs)
    cfg = SkipCfg(mode, k, seed, step, divisor, ZR_SKIP_RS_ONLY if rs_only else 0)
    _check(zr_skipreduce(ptrs, n, m, dt, cfg, _stream(stream)), "zr_skipreduce")


def skipreduce_buckets(buckets, stream=None):
    """Selective SkipReduce over several buckets in one launch.

    ``buckets``: list of dicts with ``bufs`` (list of rank tensors) and the
    ``skipreduce`` keywords ``k``, ``mode``, ``seed``, ``step``, ``divisor``,
    ``rs_only`` (k = 0 protects a bucket).  All buckets share N and dtype.
    """
    args, n, dt = [], None, None
    for b in buckets:
        ptrs, bn, m, bdt = _dense_args(b["bufs"])
        if n is None:
            n, dt = bn, bdt
        elif bn != n or bdt != dt:
            raise ValueError("every bucket needs the same number of ranks and dtype")
        cfg = SkipCfg(b.get("mode", ZR_SKIP_RANDOM), b.get("k", 0), b.get("seed", 0),
                      b.get("step", 0), b.get("divisor", ZR_DIV_N),
                      ZR_SKIP_RS_ONLY if b.get("rs_only", False) else 0)
        args.append((ptrs, m, cfg))
    _check(zr_skipreduce_buckets(args, n, dt, _stream(stream)), "zr_skipreduce_buckets")


def dropout_threshold(p):
    """Integer threshold T = ceil(p * 2^32) for skip probability p in [0, 1]."""
    from fractions import Fraction

    q = Fraction(p)
    if not (0 <= q <= 1):
        raise ValueError("p must be in [0, 1]")
    t = q * (1 << 32)
    return -(-t.numerator // t.denominator)


def allreduce_dropout(bufs, p, seed=0, step=0, average=True, stream=None):
    """In-place AllReduce_Dropout: each receiving rank skips its local element
    with probability ``p`` (SkipReduce's ReduceOrSkip)."""
    ptrs, n, m, dt = _dense_args(bufs)
    _check(zr_allreduce_dropout(ptrs, n, m, dt, dropout_threshold(p), seed, step,
                                1 if average else 0, _stream(stream)), "zr_allreduce_dropout")


def skip_fraction_to_k(p, n):
    """SkipReduce skip fraction p -> number of skipped steps k = p*N (the pages:
    skipping k Reduce-Scatter steps skips k/N of the gradients)."""
    k = p * n
    if abs(k - round(k)) > 1e-9 or not (0 <= round(k) <= n - 1):
        raise ValueError("skip fraction %r needs p*N to be an integer in [0, N-1]" % (p,))
    return int(round(k))


class SparseWorkspace:
    """Device workspace and outputs for ``sparse_aggregate`` (torch-allocated)."""

    def __init__(self, n, dense_size, n_parts, capacity, device):
        import torch

        ws_bytes = zr_sparse_workspace_size(n, dense_size, n_parts)
        if ws_bytes == 0:
            raise ValueError("invalid sparse workspace request")
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
        self.out_idx = torch.empty(max(1, capacity), dtype=torch.int32, device=device)
        self.out_val = torch.empty(max(1, capacity), dtype=torch.float32, device=device)
        self.out_nnz = torch.zeros(1, dtype=torch.int64, device=device)
        self.offsets = torch.zeros(max(n_parts, 1) + 1, dtype=torch.int64, device=device)
        self.capacity = capacity
        self.n_parts = n_parts


def sparse_aggregate(idx_list, val_list, dense_size, n_parts, part_seed=0, average=False,
                     work=None, stream=None):
    """Union with rank-ordered sums, partitioned by h0.  Returns the workspace
    object whose ``out_idx``/``out_val``/``out_nnz``/``offsets`` hold the result
    (device tensors; nothing is copied to the host)."""
    n = len(idx_list)
    nnz = [int(a.numel()) for a in idx_list]
    for a, v in zip(idx_list, val_list):
        if a.dtype.itemsize != 4 or not a.is_cuda or not v.is_cuda or a.numel() != v.numel():
            raise ValueError("idx must be int32 and val float32 CUDA tensors of equal length")
    if work is None:
        work = SparseWorkspace(n, dense_size, n_parts, sum(nnz), idx_list[0].device)
    st = zr_sparse_aggregate([a.data_ptr() for a in idx_list], [v.data_ptr() for v in val_list],
                             nnz, n, dense_size, n_parts, part_seed, 1 if average else 0,
                             work.out_idx.data_ptr(), work.out_val.data_ptr(), work.capacity,
                             work.out_nnz.data_ptr(), work.offsets.data_ptr(), work.ws.data_ptr(),
                             work.ws.numel(), _stream(stream))
    _check(st, "zr_sparse_aggregate")
    return work


def partition(idx, val, n_parts, part_seed=0, out_idx=None, out_val=None, offsets=None, ws=None,
              stream=None):
    """Stable h0 partition of one COO list; returns (out_idx, out_val, offsets)."""
    import torch

    nnz = int(idx.numel())
    dev = idx.device
    out_idx = torch.empty(max(1, nnz), dtype=torch.int32, device=dev) if out_idx is None else out_idx
    out_val = torch.empty(max(1, nnz), dtype=torch.float32, device=dev) if out_val is None else out_val
    offsets = torch.empty(n_parts + 1, dtype=torch.int64, device=dev) if offsets is None else offsets
    if ws is None:
        ws = torch.empty(max(16, zr_partition_workspace_size(nnz, n_parts)), dtype=torch.uint8,
                         device=dev)
    st = zr_partition(idx.data_ptr(), val.data_ptr(), nnz, n_parts, part_seed, out_idx.data_ptr(),
                      out_val.data_ptr(), offsets.data_ptr(), ws.data_ptr(), ws.numel(),
                      _stream(stream))
    _check(st, "zr_partition")
    return out_idx, out_val, offsets


# ------------------------------------------------------------ hash bitmap
class HashBitmap:
    """Zen's hash bitmaps of a dense size, partition count and h0 seed: the
    directory of index-set counts built once on the device, and the encode /
    decode calls that use it.  ``bits`` and ``keys`` results are torch
    tensors (bitmap words stored as int32)."""

    def __init__(self, dense_size, n_parts, part_seed=0, device="cuda", stream=None):
        import torch

        self.m, self.parts, self.seed = dense_size, n_parts, part_seed
        n_dir = zr_hash_directory_size(dense_size, n_parts)
        n_ws = zr_hash_bitmap_workspace_size(dense_size, n_parts)
        if n_dir == 0 or n_ws == 0:
            raise ValueError("invalid hash bitmap request")
        self.directory = torch.empty(n_dir // 4, dtype=torch.int32, device=device)
        _check(zr_hash_directory(dense_size, n_parts, part_seed, self.directory.data_ptr(), n_dir,
                                 _stream(stream)), "zr_hash_directory")
        self.ws = torch.empty(n_ws, dtype=torch.uint8, device=device)
        self.cap_words = (dense_size + 31) // 32 + n_parts
        self.bits = torch.empty(self.cap_words, dtype=torch.int32, device=device)
        self.word_offsets = torch.empty(n_parts + 1, dtype=torch.int64, device=device)

    def encode(self, keys, stream=None):
        """Bitmaps of the nonzero indices ``keys`` (int32 CUDA tensor)."""
        _check(zr_hash_bitmap_encode(self.directory.data_ptr(), self.m, self.parts, self.seed,
                                     keys.data_ptr() if keys.numel() else None, keys.numel(),
                                     self.bits.data_ptr(), self.cap_words,
                                     self.word_offsets.data_ptr(), self.ws.data_ptr(),
                                     self.ws.numel(), _stream(stream)), "zr_hash_bitmap_encode")
        return self.bits, self.word_offsets

    def decode(self, bits, out_keys, key_offsets, stream=None):
        """Indices of the set bits of ``bits`` (laid out as ``encode``
        writes them) into ``out_keys``; partition offsets into
        ``key_offsets``."""
        _check(zr_hash_bitmap_decode(self.directory.data_ptr(), self.m, self.parts, self.seed,
                                     bits.data_ptr(), out_keys.data_ptr(), out_keys.numel(),
                                     key_offsets.data_ptr(), self.ws.data_ptr(), self.ws.numel(),
                                     _stream(stream)), "zr_hash_bitmap_decode")
        return out_keys, key_offsets

    def status(self, stream=None):
        return zr_query_status(self.ws.data_ptr(), _stream(stream))


def hash_index_sets(dense_size, n_parts, part_seed=0, device="cuda", stream=None):
    """Zen's index sets I_p of [0, dense_size) on the device: (sets, offsets)
    with I_p = sets[offsets[p]:offsets[p+1]], each ascending."""
    import torch

    sets = torch.empty(dense_size, dtype=torch.int32, device=device)
    offsets = torch.empty(n_parts + 1, dtype=torch.int64, device=device)
    ws = torch.empty(max(16, zr_partition_workspace_size(dense_size, n_parts)),
                     dtype=torch.uint8, device=device)
    _check(zr_hash_index_sets(dense_size, n_parts, part_seed, sets.data_ptr(), offsets.data_ptr(),
                              ws.data_ptr(), ws.numel(), _stream(stream)), "zr_hash_index_sets")
    torch.cuda.synchronize()  # one-time build; the workspace is freed on return
    return sets, offsets


def densification(idx_list, dense_size, stream=None):
    """Union sizes of groups of 2^L consecutive ranks (int64 CUDA tensor of
    log2(n) + 1 entries), measured on the device."""
    import torch

    n = len(idx_list)
    nnz = [int(a.numel()) for a in idx_list]
    dev = idx_list[0].device
    ws_bytes = zr_densification_workspace_size(n, dense_size)
    if ws_bytes == 0:
        raise ValueError("densification needs a power-of-two rank count and a valid dense size")
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty(n.bit_length(), dtype=torch.int64, device=dev)
    _check(zr_densification([a.data_ptr() for a in idx_list], nnz, n, dense_size, out.data_ptr(),
                            ws.data_ptr(), ws_bytes, _stream(stream)), "zr_densification")
    return out, ws


def choose_scheme(union_counts, n):
    """Zen's choice between balanced parallelism and hierarchical
    centralisation from measured union sizes (host)."""
    choice, g, bp, hc = zr_choose_scheme([int(v) for v in union_counts], n)
    if choice < 0:
        raise ValueError("invalid union counts or rank count")
    return choice, g, bp, hc
