"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module only draws inputs: it holds none of the aggregation arithmetic
(no ring, no skip mask, no union, no hash, no rounding rule of its own -- the
bf16 inputs are made by torch's CPU float32 -> bfloat16 cast).  Both the CUDA
path and the CPU oracle consume what it returns.

The shapes and distributions stand in for the pages' workloads (the real
models, datasets and trained weights are not available):

* DENSE_C1  -- ring all-reduce, N=4, M=2**20 fp32, N(0, 1e-3) from one PCG64
  stream seeded 0, drawn rank-major.
* DENSE_C2  -- N=8, M=25,557,032 fp32 (a ResNet-50-sized flat gradient), rank
  r drawn from PCG64 seed 200+r, N(0, 1e-3); plain, and Random SkipReduce
  with skip fraction 0.5 (k = 4), seed 0.
* DENSE_C3  -- N=8, M=143,667,240 bf16 (VGG-19-sized), rank r from seed 300+r,
  N(0, 1e-2) cast to bf16; skip fractions 0, 0.25, 0.5 (k = 0, 2, 4).
* SPARSE_C4 -- N=8 COO lists over a dense size of 262,144 x 128 = 33,554,432
  (an embedding gradient), 1 % density (335,544 entries per rank), 60 % of
  each rank's entries in the first 1/8 of the index range (Zen, Figure 3a:
  over 60 % of nonzeros in the first of 8 partitions) and the rest uniform
  over the other 7/8; a shared pool of 100,663 hot + 67,109 cold indices is
  in every rank (pairwise overlap ratio about 0.51), each rank adds a private
  draw of the same sizes; values N(0, 1).  8 partitions, partition seed 0.
* SWEEP     -- dense fp32, N in {2, 4, 8, 16} x M in {2**10, 2**14, 2**18,
  2**22, 2**26, 2**28}, N(0, 1e-3).
* DGC_C5B   -- N=16 ranks, each a dense N(0, 1) fp32 tensor of
  4096 x 11008 = 45,088,768 (rank r from seed 510+r), keeping its top 5 % by
  magnitude (2,254,438 entries; ties broken by smaller index), ascending.
  16 partitions.  Stands in for the pages' DGC top-5 % LLM gradients.

"N(0, s)" means standard deviation s.
"""

import numpy as np

DENSE_C1 = dict(name="dense_c1", n=4, m=1 << 20, sigma=1e-3, dtype="f32")
DENSE_C2 = dict(name="dense_c2", n=8, m=25_557_032, sigma=1e-3, dtype="f32",
                skip_k=4, skip_seed=0)
DENSE_C3 = dict(name="dense_c3", n=8, m=143_667_240, sigma=1e-2, dtype="bf16",
                skip_ks=(0, 2, 4))
SPARSE_C4 = dict(name="sparse_c4", n=8, m=262_144 * 128, density=0.01,
                 hot_fraction=0.6, n_parts=8, part_seed=0)
SWEEP_NS = (2, 4, 8, 16)
SWEEP_MS = (1 << 10, 1 << 14, 1 << 18, 1 << 22, 1 << 26, 1 << 28)
DGC_C5B = dict(name="dgc_c5b", n=16, m=4096 * 11008, keep=0.05, n_parts=16,
               part_seed=0)


def dense_f32_single_stream(n, m, sigma, seed):
    """(n, m) float32, one PCG64 stream drawn rank-major (DENSE_C1)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, m), dtype=np.float32)
    x *= np.float32(sigma)
    return x


def dense_f32_per_rank(n, m, sigma, seed_base):
    """(n, m) float32, rank r drawn from PCG64 seed seed_base + r."""
    x = np.empty((n, m), dtype=np.float32)
    for r in range(n):
        rng = np.random.default_rng(seed_base + r)
        x[r] = rng.standard_normal(m, dtype=np.float32)
        x[r] *= np.float32(sigma)
    return x


def dense_bf16_per_rank(n, m, sigma, seed_base):
    """(n, m) uint16 bf16 bit patterns: float32 draws cast by torch (CPU)."""
    import torch

    out = np.empty((n, m), dtype=np.uint16)
    for r in range(n):
        rng = np.random.default_rng(seed_base + r)
        v = rng.standard_normal(m, dtype=np.float32)
        v *= np.float32(sigma)
        out[r] = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return out


def dense_c1():
    c = DENSE_C1
    return dense_f32_single_stream(c["n"], c["m"], c["sigma"], 0)


def dense_c2():
    c = DENSE_C2
    return dense_f32_per_rank(c["n"], c["m"], c["sigma"], 200)


def dense_c3():
    c = DENSE_C3
    return dense_bf16_per_rank(c["n"], c["m"], c["sigma"], 300)


def dense_device(n, m, sigma, seed, device):
    """(n, m) float32 drawn on a CUDA device by torch's seeded generator
    (used for the largest sweep points, which are slow to draw on the host)."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn((n, m), generator=g, device=device, dtype=torch.float32)
    x.mul_(sigma)
    return x


def _complement(lo, hi, taken):
    mask = np.ones(hi - lo, dtype=bool)
    mask[np.asarray(taken, dtype=np.int64) - lo] = False
    return np.flatnonzero(mask).astype(np.int64) + lo


def sparse_c4(n=None, m=None, density=None, hot_fraction=None, seed=400):
    """N COO lists (idx int32 ascending unique, val float32) of the C4 shape.

    Counts are exact: nnz = floor(density*M); hot = round(hot_fraction*nnz)
    entries in [0, M/8), the rest in [M/8, M).  Half of each part (rounded
    down) is a pool shared by every rank, drawn once from PCG64(seed); the rest
    is private, drawn from PCG64(seed + 1 + r) without replacement from what
    the pool left.  Values are N(0, 1) from the rank's stream.
    """
    c = SPARSE_C4
    n = c["n"] if n is None else n
    m = c["m"] if m is None else m
    density = c["density"] if density is None else density
    hot_fraction = c["hot_fraction"] if hot_fraction is None else hot_fraction
    nnz = int(density * m)
    hot = int(round(hot_fraction * nnz))
    cold = nnz - hot
    hot_hi = m // 8
    pool_hot_n = hot // 2
    pool_cold_n = cold // 2
    rng = np.random.default_rng(seed)
    pool_hot = rng.choice(hot_hi, size=pool_hot_n, replace=False).astype(np.int64)
    pool_cold = rng.choice(m - hot_hi, size=pool_cold_n, replace=False).astype(np.int64) + hot_hi
    free_hot = _complement(0, hot_hi, pool_hot)
    free_cold = _complement(hot_hi, m, pool_cold)
    idx_lists, val_lists = [], []
    for r in range(n):
        rr = np.random.default_rng(seed + 1 + r)
        ph = free_hot[rr.choice(free_hot.size, size=hot - pool_hot_n, replace=False)]
        pc = free_cold[rr.choice(free_cold.size, size=cold - pool_cold_n, replace=False)]
        idx = np.sort(np.concatenate((pool_hot, pool_cold, ph, pc)))
        idx_lists.append(idx.astype(np.int32))
        val_lists.append(rr.standard_normal(idx.size, dtype=np.float32))
    return idx_lists, val_lists


def random_coo(n, m, nnz_per_rank, seed, shared=0):
    """Small random COO lists for parity cases: rank r holds ``shared`` common
    indices plus private ones, uniform over [0, m), values N(0, 1)."""
    rng = np.random.default_rng(seed)
    common = rng.choice(m, size=shared, replace=False) if shared else np.zeros(0, np.int64)
    idx_lists, val_lists = [], []
    for r in range(n):
        rest = _complement(0, m, common)
        k = max(0, min(nnz_per_rank - shared, rest.size))
        own = rest[rng.choice(rest.size, size=k, replace=False)] if k else np.zeros(0, np.int64)
        idx = np.sort(np.concatenate((common, own)))
        idx_lists.append(idx.astype(np.int32))
        val_lists.append(rng.standard_normal(idx.size, dtype=np.float32))
    return idx_lists, val_lists


def dgc_topk(dense, keep):
    """Indices (ascending) and values of the top ``keep`` fraction of |dense|,
    ties broken by the smaller index."""
    m = dense.size
    k = int(keep * m)
    mag = np.abs(dense)
    part = np.argpartition(-mag, k - 1)[:k]
    thresh = mag[part].min()
    above = np.flatnonzero(mag > thresh)
    at = np.flatnonzero(mag == thresh)
    idx = np.concatenate((above, at[: k - above.size]))
    idx.sort()
    return idx.astype(np.int32), dense[idx].astype(np.float32)


def dgc_c5b(n=None, m=None, keep=None):
    c = DGC_C5B
    n = c["n"] if n is None else n
    m = c["m"] if m is None else m
    keep = c["keep"] if keep is None else keep
    idx_lists, val_lists = [], []
    for r in range(n):
        rng = np.random.default_rng(510 + r)
        dense = rng.standard_normal(m, dtype=np.float32)
        i, v = dgc_topk(dense, keep)
        idx_lists.append(i)
        val_lists.append(v)
    return idx_lists, val_lists
