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
