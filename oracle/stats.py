"""Sparsity statistics straight from their definitions -- oracle side.

Test infrastructure only.  All from "Zen: Empowering Distributed Training
with Sparsity-driven Data Synchronization":

* overlap ratio, Definition 3: |I1 n I2| / min(|I1|, |I2|);
* densification ratio, Definition 4: gamma_n = d_n / d_G, the density after
  aggregating n tensors over the density of one tensor (with unequal per-rank
  counts, d_G is read as the mean per-rank density);
* skew ratio, Definition 5: max_i d_{G_i} / d_G over n uniform contiguous
  partitions of the dense index range (partition i covers
  [i*ceil(M/n), (i+1)*ceil(M/n)));
* Push and Pull imbalance ratios, Definition 8:
  max_{i,j} n*|I_i^j| / |I_i| and max_j n*|I'_j| / |I|.
* the scheme choice of section 2.3 (Theorem 1, Equations (1) and (2)):
  balanced parallelism moves 2(n-1)(gamma_n + 1) d_G M / n per GPU,
  hierarchical centralisation 2 sum_{i=1}^{log n} gamma_{2^(i-1)} d_G M.
  The pages take n a power of two and one average densification ratio per
  group size; here gamma_k is the mean over the n/k groups of k consecutive
  ranks (the groups the hierarchy merges), over the mean per-rank count.
"""

import numpy as np


def overlap_ratio(i1, i2):
    s1 = set(int(v) for v in i1)
    s2 = set(int(v) for v in i2)
    return len(s1 & s2) / min(len(s1), len(s2))


def densification_ratio(idx_lists, m):
    union = set()
    for a in idx_lists:
        union.update(int(v) for v in a)
    d_n = len(union) / m
    d_g = sum(len(a) for a in idx_lists) / len(idx_lists) / m
    return d_n / d_g


def skew_ratio(idx, m, n):
    width = -(-m // n)
    counts = [0] * n
    for v in idx:
        counts[int(v) // width] += 1
    d_g = len(idx) / m
    best = 0.0
    for i in range(n):
        size = min((i + 1) * width, m) - i * width
        if size > 0:
            best = max(best, (counts[i] / size) / d_g)
    return best


def push_imbalance(idx_lists, part_of, n):
    """``part_of`` maps an array of indices to their partitions in [0, n)."""
    worst = 0.0
    for a in idx_lists:
        if len(a) == 0:
            continue
        counts = np.bincount(part_of(np.asarray(a)), minlength=n)
        worst = max(worst, n * counts.max() / len(a))
    return worst


def pull_imbalance(union_idx, part_of, n):
    counts = np.bincount(part_of(np.asarray(union_idx)), minlength=n)
    return n * counts.max() / len(union_idx)


def group_union_counts(idx_lists):
    """For L = 0 .. log2(n): the sum over the n / 2^L groups of 2^L
    consecutive ranks of the size of the group's union (Python sets)."""
    n = len(idx_lists)
    if n & (n - 1):
        raise ValueError("n must be a power of two")
    lists = [np.unique(np.asarray(a, dtype=np.int64)) for a in idx_lists]
    out = []
    g = 1
    while g <= n:
        total = 0
        for start in range(0, n, g):
            total += np.unique(np.concatenate(lists[start:start + g])).size
        out.append(int(total))
        g *= 2
    return out


def gammas_from_counts(union_counts, total_nnz, n):
    """gamma_{2^L} = (mean union of a 2^L group) / (mean per-rank count)."""
    return [union_counts[level] * (1 << level) / total_nnz for level in range(len(union_counts))]


BALANCED_PARALLELISM = 0
HIERARCHICAL_CENTRALISATION = 1


def choose_scheme(gammas, n):
    """Equations (1) and (2) without the common factor d_G M / b; the
    balanced scheme is kept on a tie.  Returns (choice, t_bp, t_hc)."""
    logn = n.bit_length() - 1
    t_bp = 2 * (n - 1) * (gammas[logn] + 1) / n
    t_hc = 2 * sum(gammas[i - 1] for i in range(1, logn + 1))
    return (BALANCED_PARALLELISM if t_bp <= t_hc else HIERARCHICAL_CENTRALISATION), t_bp, t_hc
