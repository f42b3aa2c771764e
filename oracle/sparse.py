"""COO union with rank-ordered sums, and the h0 partition -- oracle side.

Test infrastructure only.

* Sparse tensors are COO lists: ascending unique int32 indices with float32
  values (Zen, section 2.1, Definitions 1 and 2 and the COO paragraph).
  Indices are 0-based here (the page numbers them from 1).
* Aggregation: the result has one entry for every index in the union
  I = I_1 u ... u I_n (Zen, Problem 1), and its value is the same sum a dense
  AllReduce would give (Zen, section 3.2, "no effect on per-iteration
  accuracy").  The order of the sum is fixed here as a left fold over the
  ranks that hold the index, in ascending rank order, starting from the first
  such rank's value (so a lone -0.0 stays -0.0).  With ``average`` the folded
  sum is divided once by the number of ranks N (IEEE float32 division).
* Partition: Zen's consistent first-level hash h0 decides which of the n
  servers owns an index (section 3.2, Technique #3, and Algorithm 1, where
  p <- h0(idx)).  The page asks only for a universal hash (its implementation
  uses seeded MurmurHash 2.0, whose constants are not on the pages).  Reading
  used here: Dietzfelbinger's multiply-add-shift family on 32-bit keys,
  h(x) = ((a*x + b) mod 2**64) >> 32 with a odd and (a, b) drawn from the
  partition seed by SplitMix64, then range reduction
  p(x) = floor(h(x) * n / 2**32).  The key x is the index's 32-bit pattern
  (indices of a sparse list are non-negative; a push-side list handed to the
  partition alone may hold any int32).
* Output order: Algorithm 1 says the order inside a partition does not
  matter; a canonical one is chosen: partition-major, and inside each
  partition the order of the input (ascending index for a union or any
  sorted list).  ``offsets[j]`` is where partition j starts; offsets[n] is
  the total.
"""

import heapq

import numpy as np

from . import splitmix


def union_heap(idx_lists, val_lists, average=False):
    """Union by an explicit N-way heap merge keyed (index, rank).

    Pure Python; for small and medium inputs.  Returns (idx int32, val float32).
    """
    n = len(idx_lists)
    heap = []
    for r in range(n):
        if len(idx_lists[r]):
            heap.append((int(idx_lists[r][0]), r, 0))
    heapq.heapify(heap)
    out_idx = []
    out_val = []
    while heap:
        key, r, pos = heapq.heappop(heap)
        v = np.float32(val_lists[r][pos])
        if out_idx and out_idx[-1] == key:
            out_val[-1] = np.float32(out_val[-1] + v)
        else:
            out_idx.append(key)
            out_val.append(v)
        if pos + 1 < len(idx_lists[r]):
            heapq.heappush(heap, (int(idx_lists[r][pos + 1]), r, pos + 1))
    vals = np.array(out_val, dtype=np.float32)
    if average:
        vals = vals / np.float32(n)
    return np.array(out_idx, dtype=np.int32), vals


def union_sort(idx_lists, val_lists, average=False):
    """Union by a stable sort of the rank-major concatenation.

    Equal indices stay in ascending rank order (stable sort of a rank-major
    list); the values of each run are then folded left one depth at a time,
    so the association order is the same left fold as ``union_heap``.
    """
    n = len(idx_lists)
    if n == 0:
        return np.zeros(0, np.int32), np.zeros(0, np.float32)
    idx = np.concatenate([np.asarray(a, dtype=np.int64) for a in idx_lists])
    val = np.concatenate([np.asarray(a, dtype=np.float32) for a in val_lists])
    if idx.size == 0:
        return np.zeros(0, np.int32), np.zeros(0, np.float32)
    order = np.argsort(idx, kind="stable")
    idx = idx[order]
    val = val[order]
    starts = np.flatnonzero(np.concatenate(([True], idx[1:] != idx[:-1])))
    lengths = np.diff(np.concatenate((starts, [idx.size])))
    acc = val[starts].copy()
    for depth in range(1, int(lengths.max())):
        sel = lengths > depth
        acc[sel] = acc[sel] + val[starts[sel] + depth]
    if average:
        acc = acc / np.float32(n)
    return idx[starts].astype(np.int32), acc


def h0(idx, n_parts, seed):
    """Partition of each index: floor(h(x) * n / 2**32), h multiply-add-shift."""
    a, b = splitmix.h0_params(seed)
    x = (np.asarray(idx, dtype=np.int64) & 0xFFFFFFFF).astype(np.uint64)
    h = (np.uint64(a) * x + np.uint64(b)) >> np.uint64(32)
    return ((h * np.uint64(n_parts)) >> np.uint64(32)).astype(np.int64)


def h0_scalar(x, n_parts, seed):
    """The same map on one index, with Python integers."""
    a, b = splitmix.h0_params(seed)
    h = ((a * (int(x) & 0xFFFFFFFF) + b) & splitmix.MASK64) >> 32
    return (h * n_parts) >> 32


def partition(idx, val, n_parts, seed):
    """Stable partition of one COO list by h0.

    Returns (out_idx, out_val, offsets) with offsets of length n_parts + 1.
    """
    idx = np.asarray(idx, dtype=np.int32)
    val = np.asarray(val, dtype=np.float32)
    p = h0(idx, n_parts, seed)
    order = np.argsort(p, kind="stable")
    counts = np.bincount(p, minlength=n_parts)
    offsets = np.zeros(n_parts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    return idx[order], val[order], offsets


def aggregate(idx_lists, val_lists, n_parts, seed, average=False):
    """Union with rank-ordered sums, then (if n_parts > 0) the h0 partition.

    With n_parts == 0 the union is returned in ascending index order and
    offsets is [0, U].
    """
    u_idx, u_val = union_sort(idx_lists, val_lists, average=average)
    if n_parts == 0:
        return u_idx, u_val, np.array([0, u_idx.size], dtype=np.int64)
    return partition(u_idx, u_val, n_parts, seed)
