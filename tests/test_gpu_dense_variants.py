"""GPU parity: AllReduce_Dropout, Reduce-Scatter-only output and the
multi-bucket (selective) SkipReduce launch, through the C ABI, against the
CPU oracle's literal ring, bit for bit.

Small cases cover N = 1 .. 16 and 64, fp32 and bf16, ragged slices, skip
probabilities 0, 1/4, 1/2 and 1, every divisor, and both skip modes per
bucket; the C2 shape runs AllReduce_Dropout at p = 1/2 on sampled elements
(each element's result depends only on its N inputs, its slice and its
index).
"""

import numpy as np
import pytest

import workloads
from oracle import ring as oring
from tests.gpu_util import bits_equal, require_cuda
from tests.test_gpu_dense import from_device, make_inputs, sample_positions, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return require_cuda()


def oracle(x, dtype, **kw):
    if dtype == "f32":
        return oring.allreduce_f32(x, **kw)
    return oring.allreduce_bf16(x, **kw)


def u32(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


# ------------------------------------------------------- AllReduce_Dropout
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [1, 2, 3, 5, 8, 16])
def test_dropout_small(env, n, dtype):
    torch, zr = env
    for m in sorted({1, 7, 4 * n + 3, 1000, 8 * n + 8, 20_011}):
        x = make_inputs(n, m, dtype, seed=77 * n + m, special=(m >= 8))
        for p in (0.0, 0.25, 0.5, 1.0):
            for avg in (True, False):
                bufs, _keep = to_device(torch, x, dtype, padded=(m % 2 == 0))
                zr.allreduce_dropout(bufs, p, seed=3, step=11, average=avg)
                torch.cuda.synchronize()
                got = from_device(bufs, dtype)
                want = oracle(x, dtype, divisor=oring.DIV_N if avg else oring.DIV_NONE,
                              dropout=(oring.dropout_threshold(p), 3, 11))
                assert bits_equal(got, want), (n, m, dtype, p, avg)


def test_dropout_zero_equals_ring_and_steps_differ(env):
    torch, zr = env
    x = make_inputs(8, 50_003, "f32", seed=9)
    a, _k1 = to_device(torch, x, "f32")
    b, _k2 = to_device(torch, x, "f32")
    zr.allreduce_dropout(a, 0.0, seed=1, step=2)
    zr.ring_allreduce(b, average=True)
    torch.cuda.synchronize()
    assert np.array_equal(u32(from_device(a, "f32")), u32(from_device(b, "f32")))
    c, _k3 = to_device(torch, x, "f32")
    d, _k4 = to_device(torch, x, "f32")
    zr.allreduce_dropout(c, 0.5, seed=1, step=2)
    zr.allreduce_dropout(d, 0.5, seed=1, step=3)
    torch.cuda.synchronize()
    assert not np.array_equal(u32(from_device(c, "f32")), u32(from_device(d, "f32")))


def test_dropout_64_ranks(env):
    torch, zr = env
    n, m = 64, 64 * 21 + 5
    x = make_inputs(n, m, "f32", seed=64)
    bufs, _keep = to_device(torch, x, "f32")
    zr.allreduce_dropout(bufs, 0.25, seed=8, step=1)
    torch.cuda.synchronize()
    want = oracle(x, "f32", divisor=oring.DIV_N, dropout=(oring.dropout_threshold(0.25), 8, 1))
    assert bits_equal(from_device(bufs, "f32"), want)


@pytest.mark.slow
def test_dropout_c2_sampled(env):
    torch, zr = env
    c = workloads.DENSE_C2
    n, m = c["n"], c["m"]
    x = workloads.dense_c2()
    pos = sample_positions(m, n, 100_000, seed=21)
    xs = x[:, pos].copy()
    work = torch.from_numpy(x).to("cuda")
    del x
    bufs = [work[r] for r in range(n)]
    zr.allreduce_dropout(bufs, 0.5, seed=0, step=4)
    torch.cuda.synchronize()
    idx = torch.from_numpy(pos).to("cuda")
    got = np.stack([b.index_select(0, idx).cpu().numpy() for b in bufs])
    want = oring.allreduce_f32(xs, divisor=oring.DIV_N, chunk=pos // oring.chunk_size(m, n),
                               elem=pos, dropout=(oring.dropout_threshold(0.5), 0, 4))
    assert bits_equal(got, want)


# ---------------------------------------------------------------- RS-only
def check_rs_only(got, x, want_full, n, m, o, dtype):
    c_of = oring.chunk_ids(m, n)
    for c in range(n):
        cols = np.nonzero(c_of == c)[0]
        if cols.size == 0:
            continue
        h = oring.holder_of(c, n, o)
        for r in range(n):
            if r == h:
                assert np.array_equal(u32(got[r, cols]), u32(want_full[0, cols])), (c, r)
            else:  # untouched
                assert np.array_equal(u32(got[r, cols]), u32(x[r, cols])), (c, r)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [1, 2, 4, 7, 8])
def test_rs_only(env, n, dtype):
    torch, zr = env
    for m in (5, 4 * n + 3, 30_001):
        x = make_inputs(n, m, dtype, seed=5 * n + m)
        for k in sorted({0, n // 2, n - 1}):
            for mode, step in ((zr.ZR_SKIP_STATIC, 0), (zr.ZR_SKIP_RANDOM, 6)):
                bufs, _keep = to_device(torch, x, dtype)
                zr.skipreduce(bufs, k=k, mode=mode, seed=2, step=step, divisor=zr.ZR_DIV_N,
                              rs_only=True)
                torch.cuda.synchronize()
                o = oring.skip_offset(mode, k, 2, step, n)
                full = oracle(x, dtype, k=k, o=o, divisor=oring.DIV_N)
                check_rs_only(from_device(bufs, dtype), x, full, n, m, o, dtype)


# ----------------------------------------------------------------- buckets
def bucket_specs(zr, n):
    specs = []
    rng = np.random.default_rng(n)
    for b, m in enumerate((1, 4 * n + 3, 1000, 65_537, 8 * n, 300_001)):
        k = int(rng.integers(0, n))
        if b == 2:
            k = 0  # a protected bucket
        specs.append(dict(m=m, k=k, mode=[zr.ZR_SKIP_STATIC, zr.ZR_SKIP_RANDOM][b % 2], seed=b,
                          step=7 + b, divisor=[zr.ZR_DIV_N, zr.ZR_DIV_N_MINUS_K, zr.ZR_DIV_NONE][b % 3],
                          rs_only=(b == 4)))
    return specs


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [1, 3, 8, 16])
def test_buckets_match_oracle_and_single_calls(env, n, dtype):
    torch, zr = env
    specs = bucket_specs(zr, n)
    xs = [make_inputs(n, s["m"], dtype, seed=1000 + i) for i, s in enumerate(specs)]
    dev = [to_device(torch, x, dtype, padded=(i % 2 == 0)) for i, x in enumerate(xs)]
    zr.skipreduce_buckets([dict(bufs=d[0], **{k: v for k, v in s.items() if k != "m"})
                           for d, s in zip(dev, specs)])
    torch.cuda.synchronize()
    for i, (x, s, d) in enumerate(zip(xs, specs, dev)):
        got = from_device(d[0], dtype)
        o = oring.skip_offset(s["mode"], s["k"], s["seed"], s["step"], n)
        full = oracle(x, dtype, k=s["k"], o=o, divisor=s["divisor"])
        if s["rs_only"]:
            check_rs_only(got, x, full, n, s["m"], o, dtype)
        else:
            assert bits_equal(got, full), (i, s)
        # the same bucket through the single-call entry gives the same bits
        single, _keep = to_device(torch, x, dtype)
        zr.skipreduce(single, k=s["k"], mode=s["mode"], seed=s["seed"], step=s["step"],
                      divisor=s["divisor"], rs_only=s["rs_only"])
        torch.cuda.synchronize()
        assert np.array_equal(u32(from_device(single, dtype)), u32(got)), i


def test_many_buckets_64_ranks(env):
    torch, zr = env
    n, nb = 64, 32  # 2048 rank buffers: the whole pointer table
    big = torch.zeros((nb, n, 72), dtype=torch.float32, device="cuda")
    rng = np.random.default_rng(3)
    host = rng.standard_normal((nb, n, 72)).astype(np.float32)
    big.copy_(torch.from_numpy(host))
    zr.skipreduce_buckets([dict(bufs=[big[b, r, :67] for r in range(n)], k=b % n, mode=zr.ZR_SKIP_RANDOM,
                                seed=b, step=1) for b in range(nb)])
    torch.cuda.synchronize()
    got = big.cpu().numpy()
    for b in range(nb):
        o = oring.skip_offset(oring.SKIP_RANDOM, b % n, b, 1, n)
        want = oring.allreduce_f32(host[b, :, :67], k=b % n, o=o, divisor=oring.DIV_N)
        assert bits_equal(got[b, :, :67], want), b
        assert np.array_equal(got[b, :, 67:], host[b, :, 67:])  # padding untouched
