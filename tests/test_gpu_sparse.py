"""GPU parity: sparse COO aggregation and the push-side partition (through the
C ABI) against the CPU oracle -- indices, values (bitwise), the union size and
the partition offsets must all be identical.

Small cases cover 1..64 ranks, empty lists, full overlap, disjoint supports,
keys at 0 and M-1, a dense size that is not a multiple of the bin width,
0 / 1 / 8 / 256 partitions and the average flag.  The full-size workloads are
the skewed embedding gradient (C4) and the DGC top-5 % lists (C5b), compared
whole.  Malformed input (unsorted or out-of-range indices, made on the host)
must raise the device status word without touching memory outside the
buffers.
"""

import numpy as np
import pytest

import workloads
from oracle import sparse as osparse
from tests.gpu_util import require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return require_cuda()


def run_sparse(torch, zr, idx_l, val_l, m, n_parts, seed=0, average=False):
    dev = "cuda"
    d_idx = [torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev) for a in idx_l]
    d_val = [torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(dev) for v in val_l]
    work = zr.sparse_aggregate(d_idx, d_val, m, n_parts, part_seed=seed, average=average)
    status = zr.zr_query_status(work.ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    u = int(work.out_nnz.item())
    return (status, u, work.out_idx[:u].cpu().numpy(), work.out_val[:u].cpu().numpy(),
            work.offsets.cpu().numpy())


def check(torch, zr, idx_l, val_l, m, n_parts, seed=0, average=False):
    status, u, gi, gv, goff = run_sparse(torch, zr, idx_l, val_l, m, n_parts, seed, average)
    assert status == zr.ZR_OK
    wi, wv, woff = osparse.aggregate(idx_l, val_l, n_parts, seed, average=average)
    assert u == wi.size
    np.testing.assert_array_equal(gi, wi)
    np.testing.assert_array_equal(gv.view(np.uint32), wv.view(np.uint32))
    if n_parts > 0:
        np.testing.assert_array_equal(goff, woff)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 8, 16, 64])
def test_random_small(env, n):
    torch, zr = env
    for m, nnz, shared in ((100, 30, 10), (8192, 500, 100), (8193, 2000, 1000), (50_000, 3000, 0),
                           (1 << 20, 20_000, 5_000), (3, 3, 3)):
        idx_l, val_l = workloads.random_coo(n, m, nnz, seed=n * 7 + m, shared=min(shared, nnz))
        for n_parts in (0, 1, 8, 256):
            check(torch, zr, idx_l, val_l, m, n_parts, seed=n_parts)
        # the 1/N average on the per-lane and the sort placements
        check(torch, zr, idx_l, val_l, m, 8, seed=5, average=True)
        check(torch, zr, idx_l, val_l, m, 256, seed=6, average=True)


def test_edge_cases(env):
    torch, zr = env
    empty = np.zeros(0, np.int32)
    ev = np.zeros(0, np.float32)
    # all lists empty
    check(torch, zr, [empty, empty], [ev, ev], 1000, 4)
    # some lists empty
    a = np.array([0, 5, 999], np.int32)
    av = np.array([1.0, -0.0, 3.0], np.float32)
    check(torch, zr, [empty, a, empty], [ev, av, ev], 1000, 4)
    # extremes of the key range, dense size one past a bin boundary, M = 1
    m = (1 << 13) * 3 + 1
    b = np.array([0, 8191, 8192, m - 1], np.int32)
    check(torch, zr, [b, b[::2].copy()], [np.arange(4, dtype=np.float32), np.ones(2, np.float32)], m, 3)
    check(torch, zr, [np.array([0], np.int32)] * 4, [np.array([v], np.float32) for v in (1, 2, 3, 4)], 1, 2)
    # full overlap and disjoint
    rng = np.random.default_rng(1)
    idx = np.sort(rng.choice(100_000, 4000, replace=False)).astype(np.int32)
    check(torch, zr, [idx] * 6, [rng.standard_normal(4000).astype(np.float32) for _ in range(6)], 100_000, 16)
    perm = rng.permutation(100_000)[:6000]
    parts = [np.sort(perm[r * 1000:(r + 1) * 1000]).astype(np.int32) for r in range(6)]
    check(torch, zr, parts, [rng.standard_normal(1000).astype(np.float32) for _ in range(6)], 100_000, 16)
    # special values fold like the oracle (NaN by class through bitwise equal
    # is fine here: no NaN payload arithmetic)
    s = np.array([1, 2, 3, 4], np.int32)
    vals = [np.array([np.inf, 1.0, -0.0, 3e38], np.float32), np.array([-np.inf, 1e-42, -0.0, 3e38], np.float32)]
    status, u, gi, gv, _ = run_sparse(torch, zr, [s, s], vals, 10, 2)
    wi, wv, _ = osparse.aggregate([s, s], vals, 2, 0)
    assert np.array_equal(gi, wi)
    assert np.isnan(gv[np.searchsorted(wi, 1)]) and np.isnan(wv[np.searchsorted(wi, 1)])
    ok = ~np.isnan(wv)
    assert np.array_equal(gv[ok].view(np.uint32), wv[ok].view(np.uint32))


def test_wide_key_range_many_partitions(env):
    # A dense size large enough that the per-warp partition counts do not
    # fit their workspace budget, so the writer recounts them itself.
    torch, zr = env
    rng = np.random.default_rng(12)
    m = 1 << 27
    idx_l = [np.unique(rng.integers(0, m, size=3000)).astype(np.int32) for _ in range(3)]
    idx_l[1] = np.union1d(idx_l[1], idx_l[0][::3]).astype(np.int32)
    val_l = [rng.standard_normal(a.size).astype(np.float32) for a in idx_l]
    for n_parts in (256, 3, 0):
        check(torch, zr, idx_l, val_l, m, n_parts, seed=1)


def test_wide_bins_few_partitions(env):
    # A key range wide enough that bins grow past 1024 keys with at most 32
    # partitions, plus dense runs of consecutive keys, so one bin's members
    # span more than 32 bitmap words per partition.
    torch, zr = env
    rng = np.random.default_rng(13)
    m = 1 << 29
    idx_l = []
    for r in range(4):
        sparse = rng.integers(0, m, size=4000)
        run = np.arange(1000 * r, 1000 * r + 6000)
        run2 = np.arange(m - 5000, m - 5000 + 2500 * (r + 1) // 2)
        idx_l.append(np.unique(np.concatenate([sparse, run, run2])).astype(np.int32))
    val_l = [rng.standard_normal(a.size).astype(np.float32) for a in idx_l]
    for n_parts in (32, 5, 1):
        check(torch, zr, idx_l, val_l, m, n_parts, seed=n_parts)
    check(torch, zr, idx_l, val_l, m, 7, seed=2, average=True)


@pytest.mark.parametrize("n", [3, 4])
def test_dense_bins(env, n):
    # Many entries per 1024-key bin (about 40 % of the keys per rank), the
    # regime where members are emitted partition by partition, with a
    # ragged last bin.
    torch, zr = env
    m = 60_000 + 37
    idx_l, val_l = workloads.random_coo(n, m, 25_000, seed=40 + n, shared=8_000)
    for n_parts in (8, 32, 5, 1, 0):
        check(torch, zr, idx_l, val_l, m, n_parts, seed=n_parts)
    check(torch, zr, idx_l, val_l, m, 16, seed=3, average=True)


def test_unsorted_input_sets_status(env):
    torch, zr = env
    good = np.array([1, 5, 9], np.int32)
    v = np.ones(3, np.float32)
    for bad in (np.array([5, 1, 9], np.int32), np.array([1, 5, 5], np.int32),
                np.array([1, 5, 1000], np.int32), np.array([-1, 5, 9], np.int32)):
        status, *_ = run_sparse(torch, zr, [good, bad], [v, v], 1000, 4)
        assert status == zr.ZR_ERR_INPUT_UNSORTED
    status, *_ = run_sparse(torch, zr, [good, good], [v, v], 1000, 4)
    assert status == zr.ZR_OK


def test_repeatable(env):
    torch, zr = env
    idx_l, val_l = workloads.random_coo(8, 1 << 20, 30_000, seed=9, shared=10_000)
    a = run_sparse(torch, zr, idx_l, val_l, 1 << 20, 8)
    b = run_sparse(torch, zr, idx_l, val_l, 1 << 20, 8)
    assert np.array_equal(a[2], b[2]) and np.array_equal(a[3].view(np.uint32), b[3].view(np.uint32))


def test_partition_entry(env):
    torch, zr = env
    rng = np.random.default_rng(4)
    for nnz in (0, 1, 31, 4096, 4097, 100_003):
        idx = rng.integers(0, 1 << 30, size=nnz).astype(np.int32)  # any order, repeats allowed
        val = rng.standard_normal(nnz).astype(np.float32)
        for n_parts in (1, 2, 3, 5, 16, 32, 33, 256):
            d_i = torch.from_numpy(idx).cuda()
            d_v = torch.from_numpy(val).cuda()
            oi, ov, off = zr.partition(d_i, d_v, n_parts, part_seed=n_parts)
            wi, wv, woff = osparse.partition(idx, val, n_parts, n_parts)
            np.testing.assert_array_equal(off.cpu().numpy(), woff)
            np.testing.assert_array_equal(oi[:nnz].cpu().numpy(), wi)
            np.testing.assert_array_equal(ov[:nnz].cpu().numpy().view(np.uint32), wv.view(np.uint32))


@pytest.mark.slow
def test_c4_embedding(env):
    torch, zr = env
    c = workloads.SPARSE_C4
    idx_l, val_l = workloads.sparse_c4()
    check(torch, zr, idx_l, val_l, c["m"], c["n_parts"], c["part_seed"])
    check(torch, zr, idx_l, val_l, c["m"], 0)


@pytest.mark.slow
def test_c5b_dgc(env):
    torch, zr = env
    c = workloads.DGC_C5B
    idx_l, val_l = workloads.dgc_c5b()
    check(torch, zr, idx_l, val_l, c["m"], c["n_parts"], c["part_seed"])
