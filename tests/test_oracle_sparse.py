"""Pins for the sparse oracle: union, partition and the statistics (CPU only).

* union: brute force with a Python dict on tiny random supports; the two
  independent union implementations (heap merge and stable-sort fold) agree
  bit for bit; the special cases of full overlap (densification 1) and
  disjoint supports (densification N).
* partition: offsets count what they bound, partitions are in input order,
  every index lands in the partition h0 gives it, and the Push / Pull
  imbalance stays inside Zen's Theorem 2 bound.
* statistics: Zen Figure 7's worked example, Definition 5 on a hand case, and
  the C4 generator's skew (4.8 exactly), pairwise overlap and densification
  (closed forms for sampling without replacement).
"""

import math

import numpy as np
import pytest

import workloads
from oracle import sparse, stats


def brute_union(idx_lists, val_lists):
    acc = {}
    for r in range(len(idx_lists)):  # ascending rank order
        for i, v in zip(idx_lists[r], val_lists[r]):
            i = int(i)
            acc[i] = np.float32(acc[i] + np.float32(v)) if i in acc else np.float32(v)
    keys = sorted(acc)
    return np.array(keys, np.int32), np.array([acc[k] for k in keys], np.float32)


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_union_brute_force(n):
    rng = np.random.default_rng(n)
    for trial in range(30):
        m = int(rng.integers(1, 65))
        lists_i, lists_v = [], []
        for r in range(n):
            k = int(rng.integers(0, m + 1))
            idx = np.sort(rng.choice(m, size=k, replace=False)).astype(np.int32)
            lists_i.append(idx)
            lists_v.append(rng.standard_normal(k).astype(np.float32))
        bi, bv = brute_union(lists_i, lists_v)
        for fn in (sparse.union_heap, sparse.union_sort):
            gi, gv = fn(lists_i, lists_v)
            np.testing.assert_array_equal(gi, bi)
            np.testing.assert_array_equal(gv.view(np.uint32), bv.view(np.uint32))


def test_heap_and_sort_agree_medium():
    idx_l, val_l = workloads.random_coo(8, 100_000, 5_000, seed=11, shared=2_000)
    hi, hv = sparse.union_heap(idx_l, val_l)
    si, sv = sparse.union_sort(idx_l, val_l)
    np.testing.assert_array_equal(hi, si)
    np.testing.assert_array_equal(hv.view(np.uint32), sv.view(np.uint32))
    hi, hv = sparse.union_heap(idx_l, val_l, average=True)
    si, sv = sparse.union_sort(idx_l, val_l, average=True)
    np.testing.assert_array_equal(hv.view(np.uint32), sv.view(np.uint32))


def test_full_overlap_and_disjoint():
    rng = np.random.default_rng(5)
    n, m = 4, 1000
    idx = np.sort(rng.choice(m, 100, replace=False)).astype(np.int32)
    vals = [rng.integers(-50, 50, idx.size).astype(np.float32) for _ in range(n)]
    ui, uv = sparse.union_sort([idx] * n, vals)
    np.testing.assert_array_equal(ui, idx)
    np.testing.assert_array_equal(uv, np.sum(vals, axis=0, dtype=np.float64).astype(np.float32))
    assert stats.densification_ratio([idx] * n, m) == pytest.approx(1.0)
    perm = rng.permutation(m)[: n * 50]
    parts = [np.sort(perm[r * 50:(r + 1) * 50]).astype(np.int32) for r in range(n)]
    pv = [rng.standard_normal(50).astype(np.float32) for _ in range(n)]
    ui, uv = sparse.union_sort(parts, pv)
    np.testing.assert_array_equal(ui, np.sort(perm[: n * 50]))
    lookup = {int(i): v for p, vv in zip(parts, pv) for i, v in zip(p, vv)}
    np.testing.assert_array_equal(uv, np.array([lookup[int(i)] for i in ui], np.float32))
    assert stats.densification_ratio(parts, m) == pytest.approx(n)


def test_negative_zero_kept_for_single_holder():
    ui, uv = sparse.union_sort([np.array([3], np.int32), np.array([4], np.int32)],
                               [np.array([-0.0], np.float32), np.array([1.0], np.float32)])
    assert np.signbit(uv[0]) and uv[1] == 1.0


def test_partition_structure():
    rng = np.random.default_rng(9)
    idx = np.sort(rng.choice(1 << 24, 50_000, replace=False)).astype(np.int32)
    val = rng.standard_normal(idx.size).astype(np.float32)
    for n_parts in (1, 3, 8, 16, 64):
        oi, ov, off = sparse.partition(idx, val, n_parts, seed=7)
        assert off[0] == 0 and off[-1] == idx.size and (np.diff(off) >= 0).all()
        p_sample = rng.choice(idx.size, 200, replace=False)
        for j in range(n_parts):
            seg = oi[off[j]:off[j + 1]]
            assert (np.diff(seg) > 0).all()
        for pos in p_sample:
            j = int(np.searchsorted(off, pos, side="right") - 1)
            assert sparse.h0_scalar(int(oi[pos]), n_parts, 7) == j
        # values travel with their indices
        lookup = dict(zip(idx.tolist(), val.view(np.uint32).tolist()))
        assert all(lookup[i] == v for i, v in zip(oi[:500].tolist(), ov[:500].view(np.uint32).tolist()))


def theorem2_bound(n, size, density, c=3.0):
    # Zen, Theorem 2: imbalance <= 1 + Theta(sqrt(n log n / (|G| d))) w.p. >= 1 - 1/n.
    return 1.0 + c * math.sqrt(n * math.log(n) / (size * density))


def test_theorem2_worked_example():
    # Zen, Theorem 2 remark: n = 128, |G| = 1e7, d = 0.5 gives a term below 0.02.
    assert math.sqrt(128 * math.log(128) / (1e7 * 0.5)) < 0.02


def test_push_pull_imbalance_within_theorem2():
    idx_l, val_l = workloads.random_coo(8, 1 << 22, 40_000, seed=3, shared=10_000)
    n = 8
    part_of = lambda a: sparse.h0(a, n, 0)  # noqa: E731
    push = stats.push_imbalance(idx_l, part_of, n)
    ui, _ = sparse.union_sort(idx_l, val_l)
    pull = stats.pull_imbalance(ui, part_of, n)
    assert push <= theorem2_bound(n, 1 << 22, 40_000 / (1 << 22))
    assert pull <= theorem2_bound(n, 1 << 22, ui.size / (1 << 22))
    # The contiguous split (the naive mapping Zen argues against) is badly
    # skewed on skewed inputs; h0 is not.
    c4_i, c4_v = workloads.sparse_c4(n=2)
    contiguous = lambda a: np.asarray(a, np.int64) // ((1 << 25) // n)  # noqa: E731
    assert stats.push_imbalance(c4_i, contiguous, n) > 4.0
    assert stats.push_imbalance(c4_i, part_of, n) < 1.1


def test_fig7_worked_example():
    # Zen, Figure 7: 15 gradients, 6 nonzeros, 3 GPUs, contiguous partitions
    # of 5; the middle one holds 4 nonzeros, so GPU 1 receives 4x the others.
    nz = np.array([1, 5, 6, 8, 9, 13])
    contiguous = lambda a: np.asarray(a) // 5  # noqa: E731
    counts = np.bincount(contiguous(nz), minlength=3)
    assert list(counts) == [1, 4, 1]
    assert stats.pull_imbalance(nz, contiguous, 3) == pytest.approx(2.0)


def test_definitions_on_hand_cases():
    assert stats.overlap_ratio([1, 2, 3, 4], [3, 4, 5]) == pytest.approx(2 / 3)
    assert stats.skew_ratio([0, 1, 2, 9], 12, 3) == pytest.approx((3 / 4) / (4 / 12))
    assert stats.densification_ratio([[0, 1], [1, 2]], 10) == pytest.approx(1.5)


@pytest.mark.slow
def test_c4_generator_statistics():
    idx_l, _ = workloads.sparse_c4()
    c = workloads.SPARSE_C4
    m, n = c["m"], c["n"]
    assert all(a.size == 335_544 for a in idx_l)
    assert all((np.diff(a) > 0).all() and a[0] >= 0 and a[-1] < m for a in idx_l)
    # Definition 5 with 8 partitions: 60 % of entries in 1/8 of the range.
    assert stats.skew_ratio(idx_l[0], m, 8) == pytest.approx(0.6 * 8, abs=1e-5)
    # Definition 3: shared pool + chance overlap of two private draws.
    hot, cold = m // 8, m - m // 8
    pool = 100_663 + 67_109
    chance = 100_663 ** 2 / (hot - 100_663) + 67_109 ** 2 / (cold - 67_109)
    assert stats.overlap_ratio(idx_l[0], idx_l[1]) == pytest.approx((pool + chance) / 335_544, abs=2e-3)
    # Definition 4: the union of 8 private draws without replacement.
    u_hot = (hot - 100_663) * (1 - (1 - 100_663 / (hot - 100_663)) ** n)
    u_cold = (cold - 67_109) * (1 - (1 - 67_109 / (cold - 67_109)) ** n)
    gamma = (pool + u_hot + u_cold) / 335_544
    assert stats.densification_ratio(idx_l, m) == pytest.approx(gamma, rel=2e-3)


# --------------------------------------------------------- scheme choice
def test_group_union_counts_brute_force():
    from oracle import stats

    rng = np.random.default_rng(31)
    for n in (1, 2, 4, 8):
        lists = [np.unique(rng.integers(0, 200, size=rng.integers(0, 60))) for _ in range(n)]
        counts = stats.group_union_counts(lists)
        assert counts[0] == sum(len(a) for a in lists)
        assert counts[-1] == len(set().union(*[set(a.tolist()) for a in lists]))
        # each level: sum over groups, recomputed by hand
        for level, c in enumerate(counts):
            g = 1 << level
            want = sum(len(set(np.concatenate(lists[s:s + g]).tolist())) for s in range(0, n, g))
            assert c == want


@pytest.mark.parametrize("n", [4, 8, 16, 64])
def test_scheme_choice_extreme_cases(n):
    # Zen section 2.3: with full overlap (gamma_k = 1) the hierarchical sum
    # is log n while the balanced term is 2(n-1)/n < 2, so balanced
    # parallelism wins; with no overlap (gamma_k = k) the sum is n - 1 and
    # the balanced term (n-1)(1 + 1/n) is larger, so the hierarchy wins.
    from oracle import stats

    logn = n.bit_length() - 1
    full = [1.0] * (logn + 1)
    choice, t_bp, t_hc = stats.choose_scheme(full, n)
    assert t_hc == pytest.approx(2 * logn) and t_bp == pytest.approx(4 * (n - 1) / n)
    assert choice == stats.BALANCED_PARALLELISM
    disjoint = [float(1 << level) for level in range(logn + 1)]
    choice, t_bp, t_hc = stats.choose_scheme(disjoint, n)
    assert t_hc == pytest.approx(2 * (n - 1)) and t_bp == pytest.approx(2 * (n - 1) * (1 + 1 / n))
    assert choice == stats.HIERARCHICAL_CENTRALISATION


def test_gammas_of_identical_and_disjoint_lists():
    from oracle import stats

    same = [np.arange(0, 100, 3)] * 8
    g = stats.gammas_from_counts(stats.group_union_counts(same), 8 * 34, 8)
    assert g == pytest.approx([1.0, 1.0, 1.0, 1.0])
    disjoint = [np.arange(r * 50, r * 50 + 50) for r in range(8)]
    g = stats.gammas_from_counts(stats.group_union_counts(disjoint), 400, 8)
    assert g == pytest.approx([1.0, 2.0, 4.0, 8.0])
    # gamma_n equals Definition 4's densification ratio
    m = 1000
    assert g[-1] == pytest.approx(stats.densification_ratio(disjoint, m))
