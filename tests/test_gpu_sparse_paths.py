"""GPU parity, against the CPU oracle, for inputs the general sparse cases
reach rarely:

* ranks whose keys follow different distributions;
* a dense size of 2^31 - 1 with few entries (the widest bins);
* index lists that are not 16-byte aligned (scalar loads instead of 16-byte
  ones);
* 64 ranks with dense lists and 256 partitions;
* a push-side partition longer than the grid's resident tiles, so every CTA
  re-reads its slice after the grid-wide wait;
* the push-side partition's bounded grid-wide wait: with one CTA's arrival
  skipped (the library's test hook) every other CTA gives up after about a
  second and the status word says ZR_ERR_TIMEOUT; the next call is correct
  again.
"""

import numpy as np
import pytest

from oracle import sparse as osparse
from tests.gpu_util import require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return require_cuda()


def aggregate_raw(torch, zr, d_idx, d_val, nnz, m, n_parts, seed=0, average=0):
    """zr_sparse_aggregate through the C ABI on given device pointers."""
    n = len(nnz)
    total = int(sum(nnz))
    ws_bytes = zr.zr_sparse_workspace_size(n, m, n_parts)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out_idx = torch.full((max(1, total),), -7, dtype=torch.int32, device="cuda")
    out_val = torch.full((max(1, total),), -7.0, dtype=torch.float32, device="cuda")
    out_nnz = torch.full((1,), -7, dtype=torch.int64, device="cuda")
    offs = torch.full((max(1, n_parts) + 1,), -7, dtype=torch.int64, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = zr.zr_sparse_aggregate(d_idx, d_val, nnz, n, m, n_parts, seed, average,
                                out_idx.data_ptr(), out_val.data_ptr(), total,
                                out_nnz.data_ptr(), offs.data_ptr(), ws.data_ptr(), ws_bytes,
                                stream)
    assert st == zr.ZR_OK, zr.status_string(st)
    status = zr.zr_query_status(ws.data_ptr(), stream)
    u = int(out_nnz.item())
    return status, u, out_idx, out_val, offs


def check_lists(torch, zr, idx_l, val_l, m, n_parts, seed=0, average=False, misalign=0):
    """Device copies of the lists starting `misalign` elements into their
    allocation (misalign = 1 gives 4-byte-aligned pointers), then parity."""
    keep = []
    d_idx, d_val = [], []
    for a, v in zip(idx_l, val_l):
        ta = torch.zeros(a.size + misalign + 1, dtype=torch.int32, device="cuda")
        tv = torch.zeros(v.size + misalign + 1, dtype=torch.float32, device="cuda")
        ta[misalign:misalign + a.size] = torch.from_numpy(np.ascontiguousarray(a, np.int32))
        tv[misalign:misalign + v.size] = torch.from_numpy(np.ascontiguousarray(v, np.float32))
        keep += [ta, tv]
        d_idx.append(ta.data_ptr() + 4 * misalign)
        d_val.append(tv.data_ptr() + 4 * misalign)
    nnz = [int(a.size) for a in idx_l]
    status, u, oi, ov, offs = aggregate_raw(torch, zr, d_idx, d_val, nnz, m, n_parts, seed,
                                            1 if average else 0)
    assert status == zr.ZR_OK, zr.status_string(status)
    wi, wv, woff = osparse.aggregate(idx_l, val_l, n_parts, seed, average=average)
    assert u == wi.size
    np.testing.assert_array_equal(oi[:u].cpu().numpy(), wi)
    np.testing.assert_array_equal(ov[:u].cpu().numpy().view(np.uint32), wv.view(np.uint32))
    if n_parts > 0:
        np.testing.assert_array_equal(offs.cpu().numpy(), woff)


def test_ranks_with_different_distributions(env):
    torch, zr = env
    rng = np.random.default_rng(31)
    m = 4_000_000
    low = np.sort(rng.choice(m // 10, 60_000, replace=False)).astype(np.int32)
    high = np.sort(m - 1 - rng.choice(m // 10, 90_000, replace=False)).astype(np.int32)
    spread = np.sort(rng.choice(m, 40_000, replace=False)).astype(np.int32)
    tiny = np.array([m // 2], np.int32)
    idx_l = [low, high, spread, tiny, np.union1d(low[::7], spread[::5]).astype(np.int32)]
    val_l = [rng.standard_normal(a.size).astype(np.float32) for a in idx_l]
    for n_parts in (0, 8, 37):
        check_lists(torch, zr, idx_l, val_l, m, n_parts, seed=n_parts)


def test_full_int32_key_range_with_few_entries(env):
    torch, zr = env
    rng = np.random.default_rng(32)
    m = (1 << 31) - 1
    idx_l = []
    for r in range(3):
        a = rng.integers(0, m, size=2500)
        a = np.concatenate([a, [0, m - 1], np.arange(1 << 30, (1 << 30) + 3000)])
        idx_l.append(np.unique(a).astype(np.int32))
    val_l = [rng.standard_normal(a.size).astype(np.float32) for a in idx_l]
    for n_parts in (16, 0):
        check_lists(torch, zr, idx_l, val_l, m, n_parts, seed=3)


@pytest.mark.parametrize("n", [1, 3, 8])
def test_lists_not_16_byte_aligned(env, n):
    torch, zr = env
    rng = np.random.default_rng(33 + n)
    m = 2_000_003
    pool = rng.choice(m, 30_000, replace=False)
    idx_l = []
    for r in range(n):
        own = rng.choice(m, 50_000 + 17 * r, replace=False)
        idx_l.append(np.unique(np.concatenate([pool, own])).astype(np.int32))
    val_l = [rng.standard_normal(a.size).astype(np.float32) for a in idx_l]
    check_lists(torch, zr, idx_l, val_l, m, 8, seed=1, misalign=1)
    check_lists(torch, zr, idx_l, val_l, m, 0, misalign=3, average=True)


def test_many_ranks_dense_lists_many_partitions(env):
    torch, zr = env
    rng = np.random.default_rng(35)
    m = 300_007
    idx_l = [np.sort(rng.choice(m, int(m * (0.2 + 0.6 * (r % 5) / 4)), replace=False)).astype(np.int32)
             for r in range(64)]
    val_l = [rng.standard_normal(a.size).astype(np.float32) for a in idx_l]
    check_lists(torch, zr, idx_l, val_l, m, 256, seed=9)
    check_lists(torch, zr, idx_l, val_l, m, 33, seed=2, average=True)


def test_partition_longer_than_resident_tiles(env):
    torch, zr = env
    rng = np.random.default_rng(36)
    nnz = 3_000_017
    idx = rng.integers(0, 1 << 31, size=nnz, dtype=np.int64).astype(np.int32)
    val = rng.standard_normal(nnz).astype(np.float32)
    d_i = torch.from_numpy(idx).cuda()
    d_v = torch.from_numpy(val).cuda()
    for n_parts in (7, 256):
        oi, ov, off = zr.partition(d_i, d_v, n_parts, part_seed=n_parts)
        wi, wv, woff = osparse.partition(idx, val, n_parts, n_parts)
        np.testing.assert_array_equal(off.cpu().numpy(), woff)
        np.testing.assert_array_equal(oi[:nnz].cpu().numpy(), wi)
        np.testing.assert_array_equal(ov[:nnz].cpu().numpy().view(np.uint32), wv.view(np.uint32))


def test_grid_wait_times_out_when_a_cta_never_arrives(env):
    torch, zr = env
    rng = np.random.default_rng(37)
    nnz = 200_000
    idx = rng.integers(0, 1 << 24, size=nnz).astype(np.int32)
    val = rng.standard_normal(nnz).astype(np.float32)
    d_i = torch.from_numpy(idx).cuda()
    d_v = torch.from_numpy(val).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    ws = torch.empty(zr.zr_partition_workspace_size(nnz, 8), dtype=torch.uint8, device="cuda")
    oi = torch.empty(nnz, dtype=torch.int32, device="cuda")
    ov = torch.empty(nnz, dtype=torch.float32, device="cuda")
    off = torch.empty(9, dtype=torch.int64, device="cuda")
    try:
        zr.zr_test_barrier_skip(0)
        st = zr.zr_partition(d_i.data_ptr(), d_v.data_ptr(), nnz, 8, 0, oi.data_ptr(),
                             ov.data_ptr(), off.data_ptr(), ws.data_ptr(), ws.numel(), stream)
        assert st == zr.ZR_OK
        assert zr.zr_query_status(ws.data_ptr(), stream) == zr.ZR_ERR_TIMEOUT
    finally:
        zr.zr_test_barrier_skip(-1)
    # the context is still usable and the next call is exact
    st = zr.zr_partition(d_i.data_ptr(), d_v.data_ptr(), nnz, 8, 0, oi.data_ptr(), ov.data_ptr(),
                         off.data_ptr(), ws.data_ptr(), ws.numel(), stream)
    assert st == zr.ZR_OK
    assert zr.zr_query_status(ws.data_ptr(), stream) == zr.ZR_OK
    wi, wv, woff = osparse.partition(idx, val, 8, 0)
    np.testing.assert_array_equal(off.cpu().numpy(), woff)
    np.testing.assert_array_equal(oi.cpu().numpy(), wi)
    np.testing.assert_array_equal(ov.cpu().numpy().view(np.uint32), wv.view(np.uint32))
