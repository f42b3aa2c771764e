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

AllReduce_Dropout (SkipReduce, section 4.2, Algorithm 1 "AllReduce with
Fine-Grained Skipping", ReduceOrSkip): at every Reduce-Scatter step the
receiving rank draws, per element, whether to skip its local gradient; a
skipped element forwards the received value unchanged, otherwise it forwards
local + received.  The rank that first sends a slice is never asked, so its
value is always in the sum.  The pages draw from cuRAND; here the draw of
receiving rank r for element e (its index in the tensor) in iteration
``step`` is one 32-bit half of output number e // 2 of SplitMix64 seeded
with ``dropout_stream(seed, step, r)`` (output number step*64 + r of
SplitMix64(seed)): the high half for even e, the low half for odd e.  The
element is skipped when the draw is below the integer threshold T (T = ceil(p * 2**32) for skip probability p, so T = 0
never skips and T = 2**32 always does).

RS-only (15-642 notes, "ZeRO Stage 2": the AllReduce is replaced by a
Reduce-Scatter and every GPU keeps only the partition it owns): the
AllGather is not run, and only the holder's slice is a result.
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


def dropout_stream(seed, step, r):
    """Seed of receiving rank r's draw stream in iteration ``step``."""
    return splitmix.output(seed, step * 64 + r)


def dropout_skips(seed, step, r, elems, threshold):
    """Boolean array: does rank r skip each element index in ``elems``?

    The element's draw is one 32-bit half of output number e // 2 of
    SplitMix64(dropout_stream(seed, step, r)): the high half for even e, the
    low half for odd e.  The element is skipped when the draw is below
    ``threshold`` (an integer in [0, 2**32]).
    """
    s = dropout_stream(seed, step, r)
    e = np.asarray(elems, dtype=np.int64)
    out = splitmix.outputs(s, e >> 1)
    draws = np.where((e & 1) == 1, out & np.uint64(0xFFFFFFFF), out >> np.uint64(32))
    return draws.astype(np.int64) < threshold


def ring_allreduce(x, k=0, o=0, divisor=DIV_NONE, chunk=None, counters=None, dropout=None,
                   elem=None, rs_only=False):
    """Run the literal ring on ``x`` (shape (N, L)), in place, and return it.

    ``x[r]`` is rank r's buffer.  ``chunk`` gives each of the L elements its
    slice id in [0, N) (default: ``chunk_ids(L, N)``).  ``k`` Reduce-Scatter
    steps are skipped (0 <= k <= N-1), ``o`` is the slice offset, ``divisor``
    one of DIV_N, DIV_N_MINUS_K, DIV_NONE.  If ``counters`` is a dict it
    receives 'rs_sent' and 'ag_sent': per-rank element counts.

    ``dropout = (threshold, seed, step)`` turns on AllReduce_Dropout's
    ReduceOrSkip at every receive; ``elem`` gives each of the L elements its
    index in the tensor (default 0 .. L-1), which keys its draw.  With
    ``rs_only`` the AllGather is not run (the holder of slice c keeps the
    result; every other position holds what the Reduce-Scatter left there).
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
            summed = x[r, members[recv]] + messages[prev]
            if dropout is not None:
                threshold, dseed, dstep = dropout
                ids = (np.arange(length) if elem is None else np.asarray(elem))[members[recv]]
                skip = dropout_skips(dseed, dstep, r, ids, threshold)
                summed = np.where(skip, messages[prev], summed)
            x[r, members[recv]] = summed

    # The holder of slice c is rank (c - 1 - o) mod N; it applies the average.
    if divisor != DIV_NONE:
        d = n if divisor == DIV_N else n - k
        for c in range(n):
            holder = (c - 1 - o) % n
            x[holder, members[c]] = x[holder, members[c]] / np.float32(d)

    # AllGather: N-1 steps of replacing copies.
    for t in range(0 if rs_only else n - 1):
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


def allreduce_f32(ranks, k=0, o=0, divisor=DIV_NONE, chunk=None, counters=None, dropout=None,
                  elem=None, rs_only=False):
    """Ring all-reduce of float32 rank buffers; returns a new (N, L) array."""
    x = np.array(ranks, dtype=np.float32, copy=True)
    return ring_allreduce(x, k=k, o=o, divisor=divisor, chunk=chunk, counters=counters,
                          dropout=dropout, elem=elem, rs_only=rs_only)


def allreduce_bf16(ranks_bits, k=0, o=0, divisor=DIV_NONE, chunk=None, counters=None,
                   dropout=None, elem=None, rs_only=False):
    """Ring all-reduce of bf16 rank buffers (uint16 bit patterns).

    Inputs are widened exactly to float32, every message and partial sum stays
    float32, and the finished value is rounded once to bf16 (RNE).  Returns the
    (N, L) uint16 bit patterns every rank ends with.
    """
    x = _bf16.widen(np.asarray(ranks_bits, dtype=np.uint16)).copy()
    ring_allreduce(x, k=k, o=o, divisor=divisor, chunk=chunk, counters=counters, dropout=dropout,
                   elem=elem, rs_only=rs_only)
    return _bf16.round_rne(x)


def holder_of(c, n, o=0):
    """The rank that holds slice c, fully reduced, after the Reduce-Scatter."""
    return (c - 1 - o) % n


def dropout_threshold(p):
    """Integer threshold T = ceil(p * 2**32) for a skip probability p in [0, 1]
    (exact: p is taken as the binary fraction a Python float holds)."""
    from fractions import Fraction

    q = Fraction(p)
    if not (0 <= q <= 1):
        raise ValueError("p must be in [0, 1]")
    t = q * (1 << 32)
    return int(-(-t.numerator // t.denominator))


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
