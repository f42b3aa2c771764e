"""GPU parity: union sizes of rank groups (Zen's densification ratios),
measured on the device through the C ABI, against the oracle, exactly; and
the scheme choice on the C4 and DGC inputs."""

import numpy as np
import pytest

import workloads
from oracle import stats
from tests.gpu_util import require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return require_cuda()


def run(torch, zr, lists, m):
    d = [torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda() for a in lists]
    counts, ws = zr.densification(d, m)
    torch.cuda.synchronize()
    assert zr.zr_query_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream) == zr.ZR_OK
    return [int(v) for v in counts.cpu().numpy()]


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64])
def test_random_lists(env, n):
    torch, zr = env
    rng = np.random.default_rng(n)
    for m in (1, 100, 5000, 1 << 20):
        lists = []
        for r in range(n):
            k = int(rng.integers(0, min(m, 3000) + 1))
            lists.append(np.sort(rng.choice(m, size=k, replace=False)))
        # overlap: half the ranks share a pool
        if m >= 100:
            pool = rng.choice(m, size=m // 20, replace=False)
            for r in range(0, n, 2):
                lists[r] = np.union1d(lists[r], pool)
        assert run(torch, zr, lists, m) == stats.group_union_counts(lists)


def test_identical_and_disjoint(env):
    torch, zr = env
    same = [np.arange(0, 100_000, 7)] * 8
    assert run(torch, zr, same, 100_000) == stats.group_union_counts(same)
    disjoint = [np.arange(r, 1 << 20, 16) for r in range(16)]
    assert run(torch, zr, disjoint, 1 << 20) == stats.group_union_counts(disjoint)


@pytest.mark.parametrize("which", ["c4", "c5b"])
def test_full_workloads_and_choice(env, which):
    torch, zr = env
    if which == "c4":
        c, (idx, _v) = workloads.SPARSE_C4, workloads.sparse_c4()
    else:
        c, (idx, _v) = workloads.DGC_C5B, workloads.dgc_c5b()
    got = run(torch, zr, idx, c["m"])
    want = stats.group_union_counts(idx)
    assert got == want
    n = len(idx)
    choice, g, bp, hc = zr.choose_scheme(got, n)
    want_choice, want_bp, want_hc = stats.choose_scheme(stats.gammas_from_counts(want, want[0], n), n)
    assert choice == want_choice
    assert bp == pytest.approx(want_bp) and hc == pytest.approx(want_hc)
