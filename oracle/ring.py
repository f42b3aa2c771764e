"""Literal ring all-reduce with SkipReduce -- oracle side (test infrastructure).

What it executes, step by step, on N simulated workers:

* Reduce-Scatter (SkipReduce, section 4.2, Algorithms 1 and 2; 15-642 notes,
  "Ring AllReduce", aggregation phase): for s = k .. N-2, every rank r sends
  its slice (r - s + o) mod N to rank r+1 and, having received the slice
  (r - s - 1 + o) mod N from rank r-1, sets that slice to op(local, received).
  All sends of a step are taken before any receive is applied, as on a real
  ring where every worker sends and receives at once.  k = 0, o = 0 is the
  plain ring; k > 0 is Static SkipReduce (k Reduce-Scatter steps skipped);
  o != 0 is Random SkipReduce (section 4.3: every rank shifts its slice
  indices by the same per-iteration offset).
* Average: after the last Reduce-Scatter step rank r holds the fully reduced
  slice (r + 1 + o) mod N.  The holder divides it by the divisor: N for the
  SkipReduce average (section 5, "skipped gradients count as zero, the divisor
  stays N"), N - k for DropReduce (section 4.1 and the DropReduce comparison
  in section 5), or nothing for a plain sum.  Division is one IEEE
  round-to-nearest float32 division.
* AllGather (SkipReduce, Algorithm 2, "same as baseline AllReduce"; 15-642
  notes, broadcast phase): N - 1 steps; at step t rank r sends the finished
  slice (r + 1 + o - t) mod N to rank r+1, which REPLACES its own copy.

Arithmetic is elementwise numpy float32: every "+" is one IEEE binary32
addition with round-to-nearest-even, nothing is reassociated.  The functions
are written without fixing the element type, so a test can run them on object
arrays whose "+" records the fold order symbolically.

Slices ("chunks"): the pages cut the tensor into N slices, one per worker
("slices = #GPUs"); they do not say how when N does not divide M.  Reading
used here: slice c covers elements [c*C, min((c+1)*C, M)) with C = ceil(M/N),
so the last slices may be short or empty.  ``chunk_ids`` gives that mapping;
the ring functions also accept any explicit per-element slice id, which lets a
test run the literal ring on a sample of elements.

Traffic counters record the number of elements each rank sends in each phase
(15-642 notes, "communication cost": 2(N-1) steps of M/N each per worker).
"""

import numpy as np

from . import bf16 as _bf16
from . import splitmix

SKIP_STATIC = 0
SKIP_RANDOM = 1
DIV_N = 0
DIV_N_MINUS_K = 1
DIV_NONE = 2


def chunk_size(m, n):
    """Slice length C = ceil(M / N) (0 for an empty tensor)."""
    return -(-m // n) if m > 0 else 0


def chunk_ids(m, n):
    """Slice id of every element: floor(e / C)."""
    c = chunk_size(m, n)
    if m == 0:
        return np.zeros(0, dtype=np.int64)
    return np.arange(m, dtype=np.int64) // c


def skip_offset(mode, k, seed, step, n):
    """Slice offset o for one iteration.

    Static SkipReduce uses o = 0.  Random SkipReduce draws o in [0, N) from the
    seed and the iteration count (SkipReduce, section 4.3).  With k = 0 nothing
    is skipped and o is forced to 0, so that "skip fraction 0" is exactly the
    plain ring.
    """
    if k == 0 or mode == SKIP_STATIC:
        return 0
    if mode != SKIP_RANDOM:
        raise ValueError("unknown skip mode %r" % (mode,))
    return splitmix.random_offset(seed, step, n)


def ring_allreduce(x, k=0, o=0, divisor=DIV_NONE, chunk=None, counters=None):
    """Run the literal ring on ``x`` (shape (N, L)), in place, and return it.

    ``x[r]`` is rank r's buffer.  ``chunk`` gives each of the L elements its
    slice id in [0, N) (default: ``chunk_ids(L, N)``).  ``k`` Reduce-Scatter
    steps are skipped (0 <= k <= N-1), ``o`` is the slice offset, ``divisor``
    one of DIV_N, DIV_N_MINUS_K, DIV_NONE.  If ``counters`` is a dict it
    receives 'rs_sent' and 'ag_sent': per-rank element counts.
    """
    n = x.shape[0]
    length = x.shape[1]
    if not (0 <= k <= n - 1):
        raise ValueError("k must be in [0, N-1]")
    if chunk is None:
        chunk = chunk_ids(length, n)
    chunk = np.asarray(chunk)
    members = [np.nonzero(chunk == c)[0] for c in range(n)]
    rs_sent = [0] * n
    ag_sent = [0] * n

    # Reduce-Scatter: N-1-k steps, s = k .. N-2.
    for s in range(k, n - 1):
        messages = []
        for r in range(n):
            send = (r - s + o) % n
            messages.append(x[r, members[send]].copy())
            rs_sent[r] += len(members[send])
        for r in range(n):
            recv = (r - s - 1 + o) % n
            prev = (r - 1) % n
            x[r, members[recv]] = x[r, members[recv]] + messages[prev]

    # The holder of slice c is rank (c - 1 - o) mod N; it applies the average.
    if divisor != DIV_NONE:
        d = n if divisor == DIV_N else n - k
        for c in range(n):
            holder = (c - 1 - o) % n
            x[holder, members[c]] = x[holder, members[c]] / np.float32(d)

    # AllGather: N-1 steps of replacing copies.
    for t in range(n - 1):
        messages = []
        for r in range(n):
            send = (r + 1 + o - t) % n
            messages.append((send, x[r, members[send]].copy()))
            ag_sent[r] += len(members[send])
        for r in range(n):
            c, payload = messages[(r - 1) % n]
            x[r, members[c]] = payload

    if counters is not None:
        counters["rs_sent"] = rs_sent
        counters["ag_sent"] = ag_sent
    return x


def allreduce_f32(ranks, k=0, o=0, divisor=DIV_NONE, chunk=None, counters=None):
    """Ring all-reduce of float32 rank buffers; returns a new (N, L) array."""
    x = np.array(ranks, dtype=np.float32, copy=True)
    return ring_allreduce(x, k=k, o=o, divisor=divisor, chunk=chunk, counters=counters)


def allreduce_bf16(ranks_bits, k=0, o=0, divisor=DIV_NONE, chunk=None, counters=None):
    """Ring all-reduce of bf16 rank buffers (uint16 bit patterns).

    Inputs are widened exactly to float32, every message and partial sum stays
    float32, and the finished value is rounded once to bf16 (RNE).  Returns the
    (N, L) uint16 bit patterns every rank ends with.
    """
    x = _bf16.widen(np.asarray(ranks_bits, dtype=np.uint16)).copy()
    ring_allreduce(x, k=k, o=o, divisor=divisor, chunk=chunk, counters=counters)
    return _bf16.round_rne(x)


def naive_allreduce(ranks, order):
    """Naive all-reduce (15-642 notes, "Naive AllReduce"): every worker
    receives all other workers' full tensors and sums them.  ``order`` is the
    list of ranks in the order the receiver adds them; the sum is a left fold
    in float32.  Returns one (L,) array (every worker computes the same one).
    """
    x = np.asarray(ranks, dtype=np.float32)
    acc = x[order[0]].copy()
    for r in order[1:]:
        acc = acc + x[r]
    return acc


def traffic_naive(n, m):
    """Total elements moved by the naive all-reduce: N(N-1)M."""
    return n * (n - 1) * m
