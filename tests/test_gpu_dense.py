"""GPU parity: the dense ring all-reduce / SkipReduce kernels (through the C
ABI) against the CPU oracle's literal ring, bit for bit.

Small cases cover every N from 1 to 16 plus 64, every skip count, both skip
modes, every divisor, fp32 and bf16, slice boundaries that do and do not fall
on 16-byte vectors, ragged tails, and special values.  The full-size
workloads (C1 whole; C2, C3 and the sweep on sampled elements, since every
element's result depends only on its N inputs and its slice id) run in the
launch configuration the benchmark times.
"""

import numpy as np
import pytest

import workloads
from oracle import ring as oring
from tests.gpu_util import bits_equal, require_cuda, ulp_report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return require_cuda()


def to_device(torch, x, dtype, padded=True):
    """Rank buffers as rows of one padded 2-D tensor (16-byte aligned rows) or
    as separate tensors."""
    n, m = x.shape
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    host = torch.from_numpy(x.view(np.int16) if dtype == "bf16" else x)
    if dtype == "bf16":
        host = host.view(torch.bfloat16)
    if padded:
        mp = (m + 7) // 8 * 8 + 8
        big = torch.zeros((n, mp), dtype=tdt, device="cuda")
        big[:, :m] = host.to("cuda")
        return [big[r, :m] for r in range(n)], big
    return [host[r].clone().to("cuda") for r in range(n)], None


def from_device(bufs, dtype):
    import torch

    if dtype == "f32":
        return np.stack([b.cpu().numpy() for b in bufs])
    return np.stack([b.cpu().view(torch.int16).numpy().view(np.uint16) for b in bufs])


def oracle_result(x, dtype, k, o, divisor, chunk=None):
    if dtype == "f32":
        return oring.allreduce_f32(x, k=k, o=o, divisor=divisor, chunk=chunk)
    return oring.allreduce_bf16(x, k=k, o=o, divisor=divisor, chunk=chunk)


def make_inputs(n, m, dtype, seed, special=False):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((n, m)) * 10.0 ** rng.integers(-4, 3, size=(n, m))).astype(np.float32)
    if special and m >= 8:
        x[0, 0] = np.inf
        x[-1, 1] = -np.inf
        x[n // 2, 2] = np.nan
        x[:, 3] = -0.0
        x[:, 4] = np.float32(1e-42)  # subnormal
        x[:, 5] = np.float32(3.0e38)  # overflows when summed
        x[0, 6] = -0.0
        x[1 % n, 6] = 0.0
    if dtype == "bf16":
        import torch

        return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return x


DIVS = (oring.DIV_N, oring.DIV_N_MINUS_K, oring.DIV_NONE)


def run_case(torch, zr, x, dtype, k, mode, seed, step, divisor, padded=True, use_ring_entry=False):
    n = x.shape[0]
    bufs, _keep = to_device(torch, x, dtype, padded=padded)
    if use_ring_entry:
        zr.ring_allreduce(bufs, average=(divisor == oring.DIV_N))
        o = 0
    else:
        zr.skipreduce(bufs, k=k, mode=mode, seed=seed, step=step, divisor=divisor)
        o = oring.skip_offset(mode, k, seed, step, n)
    torch.cuda.synchronize()
    got = from_device(bufs, dtype)
    want = oracle_result(x, dtype, k, o, divisor)
    return got, want


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8, 13, 16])
def test_small_all_k_modes_divisors(env, n, dtype):
    torch, zr = env
    for m in sorted({1, 5, max(1, n - 1), 4 * n + 3, 1000, 8 * n + 8, 65_537}):
        x = make_inputs(n, m, dtype, seed=1000 * n + m, special=(m >= 8))
        for avg in (oring.DIV_N, oring.DIV_NONE):
            got, want = run_case(torch, zr, x, dtype, 0, 0, 0, 0, avg, use_ring_entry=True)
            assert bits_equal(got, want), (n, m, dtype, "ring", avg)
        ks = range(n) if m <= 10_000 else sorted({k for k in (0, 1, n // 2, n - 1) if k < n})
        for k in ks:
            for mode, step in ((zr.ZR_SKIP_STATIC, 0), (zr.ZR_SKIP_RANDOM, 3), (zr.ZR_SKIP_RANDOM, 11)):
                for divisor in DIVS:
                    got, want = run_case(torch, zr, x, dtype, k, mode, 7, step, divisor,
                                         padded=(k % 2 == 0))
                    assert bits_equal(got, want), (n, m, dtype, k, mode, step, divisor)


def test_64_ranks(env):
    torch, zr = env
    n = 64
    for m, dtype in ((64 * 33 + 5, "f32"), (64 * 17 + 3, "bf16")):
        x = make_inputs(n, m, dtype, seed=m)
        for k, divisor in ((0, oring.DIV_N), (1, oring.DIV_N), (37, oring.DIV_N_MINUS_K), (63, oring.DIV_NONE)):
            got, want = run_case(torch, zr, x, dtype, k, zr.ZR_SKIP_RANDOM, 5, 9, divisor)
            assert bits_equal(got, want), (m, dtype, k)


def test_k0_skipreduce_equals_ring(env):
    torch, zr = env
    x = make_inputs(8, 100_003, "f32", seed=3)
    a, _ = run_case(torch, zr, x, "f32", 0, zr.ZR_SKIP_RANDOM, 99, 4, oring.DIV_N)
    b, _ = run_case(torch, zr, x, "f32", 0, 0, 0, 0, oring.DIV_N, use_ring_entry=True)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_repeatable_and_layout_independent(env):
    torch, zr = env
    x = make_inputs(5, 77_777, "f32", seed=4)
    a, _ = run_case(torch, zr, x, "f32", 2, zr.ZR_SKIP_RANDOM, 1, 2, oring.DIV_N, padded=True)
    b, _ = run_case(torch, zr, x, "f32", 2, zr.ZR_SKIP_RANDOM, 1, 2, oring.DIV_N, padded=False)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_empty_and_errors(env):
    torch, zr = env
    bufs = [torch.zeros(0, device="cuda") for _ in range(3)]
    zr.ring_allreduce(bufs)
    big = torch.zeros((2, 64), device="cuda")
    with pytest.raises(zr.ZrError) as e:
        zr.ring_allreduce([big[0, 1:33], big[1, 1:33]])
    assert e.value.status == zr.ZR_ERR_ALIGNMENT
    with pytest.raises(zr.ZrError) as e:
        zr.ring_allreduce([big[0, :48], big[0, 16:64]])
    assert e.value.status == zr.ZR_ERR_INVALID_ARG
    with pytest.raises(zr.ZrError) as e:
        zr.skipreduce([big[0], big[1]], k=2)
    assert e.value.status == zr.ZR_ERR_INVALID_ARG
    # nothing was written by the rejected calls
    assert float(big.abs().sum()) == 0.0


# ----------------------------------------------------------------- full size
def sample_positions(m, n, count, seed):
    """Random elements plus every slice's first and last 9 elements."""
    rng = np.random.default_rng(seed)
    c = oring.chunk_size(m, n)
    pos = set(rng.integers(0, m, size=count).tolist())
    for s in range(n):
        lo, hi = s * c, min((s + 1) * c, m)
        for e in list(range(lo, min(lo + 9, hi))) + list(range(max(lo, hi - 9), hi)):
            pos.add(e)
    pos.update(range(max(0, m - 9), m))
    return np.array(sorted(pos), dtype=np.int64)


def check_sampled(torch, bufs_dev, x_host_sampled, pos, n, m, dtype, k, o, divisor):
    """Compare the device result at ``pos`` with the oracle's literal ring run
    on just those elements (each keeps its own slice id)."""
    idx = torch.from_numpy(pos).to("cuda")
    got = np.stack([b.index_select(0, idx).cpu().view(torch.int16 if dtype == "bf16" else torch.float32)
                    .numpy() for b in bufs_dev])
    if dtype == "bf16":
        got = got.view(np.uint16)
    chunk = pos // oring.chunk_size(m, n)
    want = oracle_result(x_host_sampled, dtype, k, o, divisor, chunk=chunk)
    if not bits_equal(got, want):
        if dtype == "f32":
            raise AssertionError("mismatch: %d elements, max %d ULP" % ulp_report(got.ravel(), want.ravel()))
        raise AssertionError("bf16 mismatch")
    # every rank holds the same result everywhere
    for b in bufs_dev[1:]:
        assert torch.equal(b.view(torch.int16) if dtype == "bf16" else b.view(torch.int32),
                           bufs_dev[0].view(torch.int16) if dtype == "bf16" else bufs_dev[0].view(torch.int32))


def test_c1_whole(env):
    torch, zr = env
    x = workloads.dense_c1()
    got, want = run_case(torch, zr, x, "f32", 0, 0, 0, 0, oring.DIV_N, use_ring_entry=True)
    assert bits_equal(got, want)


@pytest.mark.slow
def test_c2_plain_and_random_skip(env):
    torch, zr = env
    c = workloads.DENSE_C2
    n, m = c["n"], c["m"]
    x = workloads.dense_c2()
    pos = sample_positions(m, n, 200_000, seed=2)
    xs = x[:, pos].copy()
    orig = torch.from_numpy(x).to("cuda")
    work = torch.empty_like(orig)
    bufs = [work[r] for r in range(n)]
    work.copy_(orig)
    zr.ring_allreduce(bufs, average=True)
    torch.cuda.synchronize()
    check_sampled(torch, bufs, xs, pos, n, m, "f32", 0, 0, oring.DIV_N)
    for step in range(10):
        work.copy_(orig)
        zr.skipreduce(bufs, k=c["skip_k"], mode=zr.ZR_SKIP_RANDOM, seed=c["skip_seed"], step=step)
        torch.cuda.synchronize()
        o = oring.skip_offset(oring.SKIP_RANDOM, c["skip_k"], c["skip_seed"], step, n)
        check_sampled(torch, bufs, xs, pos, n, m, "f32", c["skip_k"], o, oring.DIV_N)


@pytest.mark.slow
def test_c3_bf16_skip_fractions(env):
    torch, zr = env
    c = workloads.DENSE_C3
    n, m = c["n"], c["m"]
    x = workloads.dense_c3()
    pos = sample_positions(m, n, 200_000, seed=3)
    xs = x[:, pos].copy()
    orig = torch.from_numpy(x.view(np.int16)).to("cuda").view(torch.bfloat16)
    del x
    work = torch.empty_like(orig)
    bufs = [work[r] for r in range(n)]
    for k in c["skip_ks"]:
        for step in (0, 1):
            work.copy_(orig)
            zr.skipreduce(bufs, k=k, mode=zr.ZR_SKIP_RANDOM, seed=0, step=step)
            torch.cuda.synchronize()
            o = oring.skip_offset(oring.SKIP_RANDOM, k, 0, step, n)
            check_sampled(torch, bufs, xs, pos, n, m, "bf16", k, o, oring.DIV_N)


@pytest.mark.slow
@pytest.mark.parametrize("n", workloads.SWEEP_NS)
def test_sweep(env, n):
    torch, zr = env
    for m in workloads.SWEEP_MS:
        orig = workloads.dense_device(n, m, 1e-3, 500 + n, "cuda")
        work = orig.clone()
        bufs = [work[r] for r in range(n)]
        zr.ring_allreduce(bufs, average=True)
        torch.cuda.synchronize()
        if m <= (1 << 18):
            x = orig.cpu().numpy()
            got = work.cpu().numpy()
            want = oring.allreduce_f32(x, divisor=oring.DIV_N)
            assert bits_equal(got, want), (n, m)
        else:
            pos = sample_positions(m, n, 50_000, seed=n + m)
            idx = torch.from_numpy(pos).to("cuda")
            xs = orig.index_select(1, idx).cpu().numpy()
            check_sampled(torch, bufs, xs, pos, n, m, "f32", 0, 0, oring.DIV_N)
        del orig, work, bufs
        torch.cuda.empty_cache()
