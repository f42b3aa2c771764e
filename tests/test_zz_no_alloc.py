"""zr_partition_static -- the partition entry point for callers that cannot
allocate device memory (a gradient hook running under a framework's caching
allocator, or a service that reserves all device memory at start-up) -- must
give exactly what zr_partition gives with a caller-owned workspace.

Called through the C ABI (raw device pointers), twice in a row with
different inputs, because every call shares the library's one scratch array
and must clear what it needs.  The file is named so that pytest collects it
last; it also passes when run alone in a fresh process.
"""

import numpy as np
import pytest

from tests.gpu_util import require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return require_cuda()


def run_both(torch, zr, idx, val, n_parts, seed):
    nnz = idx.size
    d_idx = torch.from_numpy(idx).cuda()
    d_val = torch.from_numpy(val).cuda()
    outs = []
    for use_static in (False, True):
        o_idx = torch.full((max(1, nnz),), -7, dtype=torch.int32, device="cuda")
        o_val = torch.full((max(1, nnz),), -7.0, dtype=torch.float32, device="cuda")
        o_off = torch.full((n_parts + 1,), -7, dtype=torch.int64, device="cuda")
        stream = torch.cuda.current_stream().cuda_stream
        if use_static:
            st = zr.zr_partition_static(d_idx.data_ptr(), d_val.data_ptr(), nnz, n_parts, seed,
                                        o_idx.data_ptr(), o_val.data_ptr(), o_off.data_ptr(), stream)
        else:
            ws = torch.empty(max(16, zr.zr_partition_workspace_size(nnz, n_parts)),
                             dtype=torch.uint8, device="cuda")
            st = zr.zr_partition(d_idx.data_ptr(), d_val.data_ptr(), nnz, n_parts, seed,
                                 o_idx.data_ptr(), o_val.data_ptr(), o_off.data_ptr(),
                                 ws.data_ptr(), ws.numel(), stream)
        assert st == zr.ZR_OK, zr.status_string(st)
        torch.cuda.synchronize()
        outs.append((o_idx[:nnz].cpu().numpy(), o_val[:nnz].cpu().numpy(), o_off.cpu().numpy()))
    return outs


def test_static_scratch_matches_workspace_entry_on_two_calls(env):
    torch, zr = env
    rng = np.random.default_rng(21)
    for nnz, n_parts, seed in ((300_000, 8, 0), (123_457, 16, 3)):
        idx = np.sort(rng.choice(1 << 25, size=nnz, replace=False)).astype(np.int32)
        val = rng.standard_normal(nnz).astype(np.float32)
        (wi, wv, wo), (si, sv, so) = run_both(torch, zr, idx, val, n_parts, seed)
        np.testing.assert_array_equal(so, wo)
        np.testing.assert_array_equal(si, wi)
        np.testing.assert_array_equal(sv.view(np.uint32), wv.view(np.uint32))


def test_static_scratch_holds_the_largest_request(env):
    # The workspace grows with the partition count only; 256 partitions is
    # the largest request the fixed scratch must hold.  A long list with 256
    # partitions, twice in a row, must match the workspace entry point.
    torch, zr = env
    n_parts = zr.ZR_MAX_PARTS
    assert zr.zr_partition_workspace_size(1 << 22, n_parts) <= zr.ZR_STATIC_SCRATCH_BYTES
    rng = np.random.default_rng(22)
    for nnz, seed in ((1 << 22, 1), (700_001, 2)):
        idx = rng.integers(0, 1 << 31, size=nnz, dtype=np.int64).astype(np.int32)
        val = rng.standard_normal(nnz).astype(np.float32)
        (wi, wv, wo), (si, sv, so) = run_both(torch, zr, idx, val, n_parts, seed)
        np.testing.assert_array_equal(so, wo)
        np.testing.assert_array_equal(si, wi)
        np.testing.assert_array_equal(sv.view(np.uint32), wv.view(np.uint32))
