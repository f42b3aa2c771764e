"""Pins for the literal-ring oracle (CPU only).

Each test checks the oracle against something other than its own code:
symbolic fold trees, exact integer arithmetic, exact rational sums with the
textbook floating-point error bound, and the closed-form traffic counts of
the 15-642 notes ("Ring AllReduce": 2(N-1) steps of M/N elements per worker)
and of SkipReduce (section 4.2: skipping k Reduce-Scatter steps removes
k/(2(N-1)) of the communication and k/N of the gradients).
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import ring, splitmix


# ---------------------------------------------------------------- symbolic
class Sym:
    """Expression node: leaves ('g', rank, elem); '+' and '/' record the tree."""

    __slots__ = ("t",)

    def __init__(self, t):
        self.t = t

    def __add__(self, other):
        return Sym(("+", self.t, other.t))

    def __truediv__(self, d):
        return Sym(("/", self.t, float(d)))


def comm_equal(a, b):
    """Tree equality up to swapping the two operands of a '+' (IEEE addition
    is commutative, so operand order never changes a result)."""
    if a[0] != b[0]:
        return False
    if a[0] == "g":
        return a == b
    if a[0] == "/":
        return a[2] == b[2] and comm_equal(a[1], b[1])
    return (comm_equal(a[1], b[1]) and comm_equal(a[2], b[2])) or (
        comm_equal(a[1], b[2]) and comm_equal(a[2], b[1]))


def leaves(t):
    if t[0] == "g":
        return [t[1]]
    if t[0] == "/":
        return leaves(t[1])
    return leaves(t[1]) + leaves(t[2])


def symbolic_ranks(n, m):
    x = np.empty((n, m), dtype=object)
    for r in range(n):
        for e in range(m):
            x[r, e] = Sym(("g", r, e))
    return x


def expected_tree(n, e, start, count, divide):
    # What the receiver in the Reduce-Scatter computes for one element: the
    # first sender's own value, then each next rank on the ring adds its local
    # value to what it received.
    acc = ("g", start % n, e)
    for t in range(1, count):
        acc = ("+", ("g", (start + t) % n, e), acc)
    if divide is not None:
        acc = ("/", acc, float(divide))
    return acc


@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_fold_order_every_k_and_offset(n):
    m = 2 * n + 1  # ragged: the last slice is short
    c_of = ring.chunk_ids(m, n)
    for k in range(n):
        for o in range(n):
            for div in (ring.DIV_NONE, ring.DIV_N, ring.DIV_N_MINUS_K):
                x = ring.ring_allreduce(symbolic_ranks(n, m), k=k, o=o, divisor=div)
                d = {ring.DIV_NONE: None, ring.DIV_N: n, ring.DIV_N_MINUS_K: n - k}[div]
                for e in range(m):
                    c = int(c_of[e])
                    want = expected_tree(n, e, c + k - o, n - k, d)
                    for r in range(n):
                        assert comm_equal(x[r, e].t, want), (n, k, o, r, e)


@pytest.mark.parametrize("n", [2, 3, 4, 6])
def test_skipped_ranks_static_fig5(n):
    # Static SkipReduce (o = 0): slice c omits exactly ranks c .. c+k-1, and
    # every rank is left out of exactly k slices ("one full slice per GPU is
    # skipped" per skipped step, SkipReduce Figure 5).
    m = n
    for k in range(n):
        x = ring.ring_allreduce(symbolic_ranks(n, m), k=k, o=0)
        omitted_per_rank = [0] * n
        for c in range(n):
            got = set(leaves(x[0, c].t))
            want_omit = {(c + j) % n for j in range(k)}
            assert got == set(range(n)) - want_omit
            for r in want_omit:
                omitted_per_rank[r] += 1
        assert omitted_per_rank == [k] * n


@pytest.mark.parametrize("n", [3, 4, 5])
def test_random_offsets_rotate_fairly_fig6(n):
    # Random SkipReduce (Figure 6): over all offsets o in [0, N) every rank is
    # skipped from every slice exactly k times.
    for k in range(1, n):
        counts = np.zeros((n, n), dtype=int)  # [slice, rank]
        for o in range(n):
            x = ring.ring_allreduce(symbolic_ranks(n, n), k=k, o=o)
            for c in range(n):
                for r in set(range(n)) - set(leaves(x[0, c].t)):
                    counts[c, r] += 1
        assert (counts == k).all()


# ---------------------------------------------------------------- numeric
@pytest.mark.parametrize("n", [1, 2, 3, 4, 7, 8, 16])
def test_integer_inputs_ring_equals_naive_equals_sum(n):
    rng = np.random.default_rng(n)
    m = 5 * n + 3
    x = rng.integers(-1024, 1025, size=(n, m)).astype(np.float32)
    got = ring.allreduce_f32(x)
    naive = ring.naive_allreduce(x, list(range(n))[::-1])
    exact = x.astype(np.float64).sum(axis=0)
    for r in range(n):
        np.testing.assert_array_equal(got[r], exact.astype(np.float32))
    np.testing.assert_array_equal(naive, exact.astype(np.float32))


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16])
def test_power_of_two_average_is_exact(n):
    rng = np.random.default_rng(100 + n)
    m = 3 * n
    x = rng.integers(-1024, 1025, size=(n, m)).astype(np.float32)
    got = ring.allreduce_f32(x, divisor=ring.DIV_N)
    np.testing.assert_array_equal(got[0] * np.float32(n), x.astype(np.float64).sum(axis=0))


def gamma(k):
    u = Fraction(1, 1 << 24)
    return k * u / (1 - k * u)


@pytest.mark.parametrize("n,k,o", [(5, 0, 0), (5, 2, 0), (5, 2, 3), (4, 3, 1), (8, 4, 5)])
def test_error_bound_against_exact_rational_sum(n, k, o):
    # |fl(sum) - sum| <= gamma_{n-k-1} * sum |g| for a recursive sum of n-k
    # terms (Higham, Accuracy and Stability of Numerical Algorithms, 4.2).
    # The exact sum runs over the ranks that SkipReduce keeps for the slice.
    rng = np.random.default_rng(7 * n + k)
    m = 3 * n + 2
    x = (rng.standard_normal((n, m)) * 10.0 ** rng.integers(-3, 3, size=(n, m))).astype(np.float32)
    got = ring.allreduce_f32(x, k=k, o=o)
    c_of = ring.chunk_ids(m, n)
    for e in range(m):
        kept = [(int(c_of[e]) - o + k + t) % n for t in range(n - k)]
        exact = sum(Fraction(float(x[r, e])) for r in kept)
        mag = sum(abs(Fraction(float(x[r, e]))) for r in kept)
        err = abs(Fraction(float(got[0, e])) - exact)
        assert err <= gamma(n - k - 1) * mag, (e, float(err))
        # a dropped or doubled term would be far outside the bound
        assert len(kept) == n - k


@pytest.mark.parametrize("n", [1, 2, 3, 8])
def test_allgather_replicates(n):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((n, 4 * n + 1)).astype(np.float32)
    got = ring.allreduce_f32(x, divisor=ring.DIV_N)
    for r in range(1, n):
        np.testing.assert_array_equal(got[r].view(np.uint32), got[0].view(np.uint32))


def test_n1_is_identity():
    x = np.random.default_rng(0).standard_normal((1, 37)).astype(np.float32)
    x[0, 5] = -0.0
    for div in (ring.DIV_NONE, ring.DIV_N):
        got = ring.allreduce_f32(x, divisor=div)
        np.testing.assert_array_equal(got.view(np.uint32), x.view(np.uint32))


def test_negative_zero_survives_when_single_contributor():
    # With k = N-1 a slice has one contributor: its value passes through
    # unchanged (no "0 +" in front of the fold), so -0.0 stays -0.0.
    n = 4
    x = np.ones((n, n), dtype=np.float32)
    x[:, :] = -0.0
    got = ring.allreduce_f32(x, k=n - 1)
    assert np.all(np.signbit(got))


# ---------------------------------------------------------------- traffic
@pytest.mark.parametrize("n", [2, 3, 4, 5, 8])
def test_traffic_closed_forms(n):
    m = 6 * n
    full = None
    for k in range(n):
        cnt = {}
        ring.allreduce_f32(np.zeros((n, m), np.float32), k=k, counters=cnt)
        per_worker = [a + b for a, b in zip(cnt["rs_sent"], cnt["ag_sent"])]
        assert per_worker == [(2 * (n - 1) - k) * m // n] * n
        if k == 0:
            full = per_worker[0]
            assert sum(per_worker) == 2 * (n - 1) * m
            assert cnt["rs_sent"] == [(n - 1) * m // n] * n
        else:
            saved = Fraction(full - per_worker[0], full)
            assert saved == Fraction(k, 2 * (n - 1))
    assert ring.traffic_naive(n, m) == n * (n - 1) * m


def test_random_offset_forced_zero_without_skip():
    for seed in range(5):
        for step in range(5):
            assert ring.skip_offset(ring.SKIP_RANDOM, 0, seed, step, 8) == 0
            o = ring.skip_offset(ring.SKIP_RANDOM, 3, seed, step, 8)
            assert o == splitmix.random_offset(seed, step, 8)
            assert 0 <= o < 8


def test_random_offset_is_roughly_uniform():
    n = 8
    hist = np.bincount([splitmix.random_offset(0, s, n) for s in range(8000)], minlength=n)
    assert hist.min() > 850 and hist.max() < 1150


def test_chunking_ceil_rule():
    assert ring.chunk_size(10, 4) == 3
    np.testing.assert_array_equal(ring.chunk_ids(10, 4), [0, 0, 0, 1, 1, 1, 2, 2, 2, 3])
    np.testing.assert_array_equal(ring.chunk_ids(2, 4), [0, 1])
    assert ring.chunk_ids(0, 4).size == 0


# ------------------------------------------------------- AllReduce_Dropout
def test_dropout_threshold_exact():
    # T = ceil(p * 2^32) with p taken exactly as the binary fraction a float
    # holds: 0.1 is 0x3FB999999999999A, so p * 2^32 = 429496729.600000...
    assert ring.dropout_threshold(0.0) == 0
    assert ring.dropout_threshold(0.5) == 1 << 31
    assert ring.dropout_threshold(1.0) == 1 << 32
    assert ring.dropout_threshold(0.1) == 429496730
    assert ring.dropout_threshold(2.0 ** -32) == 1


@pytest.mark.parametrize("n", [2, 3, 4, 5])
def test_dropout_fold_order(n):
    # SkipReduce Algorithm 1 (ReduceOrSkip): slice c starts with its first
    # sender's value (never skipped); each next rank on the ring either adds
    # its local value or forwards what it received unchanged.
    m = 3 * n + 2
    c_of = ring.chunk_ids(m, n)
    thr, seed, step = 1 << 31, 7, 3
    x = ring.ring_allreduce(symbolic_ranks(n, m), dropout=(thr, seed, step), divisor=ring.DIV_N)
    for e in range(m):
        c = int(c_of[e])
        acc = ("g", c, e)
        for t in range(1, n):
            r = (c + t) % n
            if not ring.dropout_skips(seed, step, r, [e], thr)[0]:
                acc = ("+", ("g", r, e), acc)
        want = ("/", acc, float(n))
        for r in range(n):
            assert comm_equal(x[r, e].t, want), (n, r, e)


def test_dropout_extremes():
    rng = np.random.default_rng(11)
    n, m = 5, 53
    x = rng.standard_normal((n, m)).astype(np.float32)
    plain = ring.allreduce_f32(x, divisor=ring.DIV_N)
    none = ring.allreduce_f32(x, divisor=ring.DIV_N, dropout=(0, 1, 2))
    assert np.array_equal(plain.view(np.uint32), none.view(np.uint32))
    # T = 2^32 skips every receiving rank: slice c keeps its start rank's value
    allskip = ring.allreduce_f32(x, divisor=ring.DIV_N, dropout=(1 << 32, 1, 2))
    c_of = ring.chunk_ids(m, n)
    want = np.array([x[c_of[e], e] / np.float32(n) for e in range(m)], dtype=np.float32)
    for r in range(n):
        assert np.array_equal(allskip[r].view(np.uint32), want.view(np.uint32))


def test_dropout_integer_inputs_equal_masked_sum():
    # Small integers add exactly in fp32, so the result is the exact sum of
    # the start rank's value and every non-skipped rank's value.
    rng = np.random.default_rng(12)
    n, m = 6, 97
    x = rng.integers(-512, 512, size=(n, m)).astype(np.float32)
    thr, seed, step = ring.dropout_threshold(0.3), 5, 9
    got = ring.allreduce_f32(x, dropout=(thr, seed, step))
    c_of = ring.chunk_ids(m, n)
    for e in range(m):
        c = int(c_of[e])
        total = int(x[c, e])
        for t in range(1, n):
            r = (c + t) % n
            if not ring.dropout_skips(seed, step, r, [e], thr)[0]:
                total += int(x[r, e])
        assert got[0, e] == total


def test_dropout_skip_rate_matches_probability():
    # Bernoulli(p) per (rank, element): over 8 ranks x 20000 elements the
    # observed rate is within 5 sigma of p, for every rank and overall.
    n, m, p = 8, 20000, 0.25
    thr = ring.dropout_threshold(p)
    sigma = (p * (1 - p) / m) ** 0.5
    rates = []
    for r in range(n):
        rate = ring.dropout_skips(3, 4, r, np.arange(m), thr).mean()
        assert abs(rate - p) < 5 * sigma, (r, rate)
        rates.append(rate)
    assert abs(np.mean(rates) - p) < 5 * sigma / n ** 0.5
    # ranks draw from different streams: their skip patterns are not equal
    a = ring.dropout_skips(3, 4, 0, np.arange(512), thr)
    b = ring.dropout_skips(3, 4, 1, np.arange(512), thr)
    assert not np.array_equal(a, b)


@pytest.mark.parametrize("p", [0.5, 0.3])
def test_dropout_neighbour_draws_independent(p):
    # Two neighbouring elements share one 64-bit generator output (its two
    # halves); their skips must still be independent: the joint skip rate of
    # each pair (2i, 2i+1), and of the pairs straddling two outputs
    # (2i+1, 2i+2), is p^2 within 5 sigma.  Drawing both elements from the
    # same half would give p; the two halves swapped or taken from
    # different outputs would fail the element-by-element pins above.
    m = 1 << 16
    thr = ring.dropout_threshold(p)
    s = ring.dropout_skips(11, 2, 3, np.arange(m), thr)
    q = p * p
    sigma = (q * (1 - q) / (m // 2)) ** 0.5
    same = (s[0::2] & s[1::2]).mean()
    straddle = (s[1:-1:2] & s[2::2]).mean()
    assert abs(same - q) < 5 * sigma, same
    assert abs(straddle - q) < 5 * sigma, straddle
    # the even element's draw is the high half of output e / 2, the odd
    # element's the low half (the generator itself is pinned by its
    # published known-answer vectors)
    from oracle import splitmix
    st = ring.dropout_stream(11, 2, 3)
    for e in (0, 1, 6, 7, 1001):
        o = splitmix.output(st, e // 2)
        draw = (o & 0xFFFFFFFF) if e % 2 else (o >> 32)
        assert bool(ring.dropout_skips(11, 2, 3, [e], thr)[0]) == (draw < thr)


# ----------------------------------------------------------------- RS-only
@pytest.mark.parametrize("n,k,o", [(2, 0, 0), (4, 1, 2), (5, 3, 1), (8, 4, 7)])
def test_rs_only_holder_slices_equal_full_ring(n, k, o):
    rng = np.random.default_rng(13)
    m = 4 * n + 3
    x = rng.standard_normal((n, m)).astype(np.float32)
    full = ring.allreduce_f32(x, k=k, o=o, divisor=ring.DIV_N)
    counters = {}
    rs = ring.allreduce_f32(x, k=k, o=o, divisor=ring.DIV_N, rs_only=True, counters=counters)
    c_of = ring.chunk_ids(m, n)
    for c in range(n):
        h = ring.holder_of(c, n, o)
        cols = np.nonzero(c_of == c)[0]
        assert np.array_equal(rs[h, cols].view(np.uint32), full[0, cols].view(np.uint32))
    # no AllGather traffic; the Reduce-Scatter sends N-1-k slices per rank
    assert counters["ag_sent"] == [0] * n
    per = ring.chunk_size(m, n)
    assert sum(counters["rs_sent"]) <= n * (n - 1 - k) * per
