"""GPU parity: Zen's hash bitmap encode / decode and the directory of
index-set counts they use (through the C ABI) against the CPU oracle, bit
for bit; the index sets themselves; the C4 union at full size."""

import numpy as np
import pytest

import workloads
from oracle import hash_bitmap as ohb
from oracle import sparse as osp
from tests.gpu_util import require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return require_cuda()


def directory_want(m, parts, seed, rng_keys):
    """The directory from its definition: row p, column r counts the
    indices x < min(r * range, M) with h0(x) = p."""
    p = osp.h0(np.arange(m, dtype=np.int64), parts, seed)
    R = -(-m // rng_keys)
    want = np.zeros((parts, R + 1), dtype=np.int64)
    for r in range(R):
        blk = p[r * rng_keys:(r + 1) * rng_keys]
        want[:, r + 1] = want[:, r] + np.bincount(blk, minlength=parts)
    return want


def dir_counts(hb, m, parts, rng_keys):
    """The directory's count rows (row stride R + 1 rounded up to 4)."""
    R = -(-m // rng_keys)
    stride = (R + 1 + 3) // 4 * 4
    return hb.directory[64: 64 + parts * stride].view(parts, stride)[:, : R + 1]


def slices_want(m, parts, seed, rng_keys):
    """The directory's slices from their definition: word (r, b, lane) has
    bit k set iff bit b of h0(r * range + 64 * lane + k) is (indices at or
    past M count as 0)."""
    nb = max(0, (parts - 1).bit_length())
    R = -(-m // rng_keys)
    p = np.zeros(R * rng_keys, dtype=np.uint64)
    p[:m] = osp.h0(np.arange(m, dtype=np.int64), parts, seed)
    p = p.reshape(R, 32, 64)
    out = np.zeros((R, nb, 32), dtype=np.uint64)
    for b in range(nb):
        bits = (p >> np.uint64(b)) & np.uint64(1)
        out[:, b, :] = (bits << np.arange(64, dtype=np.uint64)).sum(axis=2, dtype=np.uint64)
    return out


def check(torch, zr, m, parts, seed, keys):
    hb = zr.HashBitmap(m, parts, seed)
    rk = zr.ZR_HASH_RANGE
    got = dir_counts(hb, m, parts, rk).cpu().numpy()
    assert np.array_equal(got, directory_want(m, parts, seed, rk))
    R = -(-m // rk)
    counts_bytes = -(-(parts * ((R + 1 + 3) // 4 * 4) * 4) // 256) * 256
    sl = hb.directory.cpu().numpy().view(np.uint8)[256 + counts_bytes:].view(np.uint64)
    want_sl = slices_want(m, parts, seed, rk)
    # bits of indices past M are unspecified in the last lanes: compare below M
    valid = np.zeros(R * rk, dtype=bool)
    valid[:m] = True
    vmask = (valid.reshape(R, 32, 64).astype(np.uint64) << np.arange(64, dtype=np.uint64)).sum(
        axis=2, dtype=np.uint64)
    assert np.array_equal(sl.reshape(want_sl.shape) & vmask[:, None, :], want_sl & vmask[:, None, :])
    d_keys = torch.from_numpy(np.ascontiguousarray(keys, dtype=np.int32)).cuda()
    bits, woff = hb.encode(d_keys)
    torch.cuda.synchronize()
    assert hb.status() == zr.ZR_OK
    want_bits, want_woff = ohb.encode_all(m, parts, seed, keys)
    assert np.array_equal(woff.cpu().numpy(), want_woff)
    got = bits.cpu().numpy().view(np.uint32)[: want_woff[-1]]
    assert np.array_equal(got, want_bits)
    out = torch.full((max(1, len(keys)),), -1, dtype=torch.int32, device="cuda")
    koff = torch.empty(parts + 1, dtype=torch.int64, device="cuda")
    hb.decode(bits, out, koff)
    torch.cuda.synchronize()
    assert hb.status() == zr.ZR_OK
    want_keys, want_koff = ohb.decode_all(m, parts, seed, want_bits, want_woff)
    assert np.array_equal(koff.cpu().numpy(), want_koff)
    assert np.array_equal(out.cpu().numpy()[: len(want_keys)], want_keys)
    return hb


@pytest.mark.parametrize("parts", [1, 2, 3, 8, 16, 17, 32, 64, 200, 256])
def test_small_and_ragged(env, parts):
    torch, zr = env
    rng = np.random.default_rng(parts)
    # sizes below one lane, one range, ragged ranges and several ranges
    for m in (1, 15, 33, 64, 1000, 2048, 2049, 100_003):
        for density in (0.0, 0.3, 1.0):
            keys = np.nonzero(rng.random(m) < density)[0].astype(np.int32)
            check(torch, zr, m, parts, int(rng.integers(0, 1 << 62)), rng.permutation(keys))


def test_index_sets(env):
    torch, zr = env
    for m, parts, seed in ((1, 1, 0), (1000, 3, 5), (100_003, 8, 7), (50_000, 256, 9)):
        sets, off = zr.hash_index_sets(m, parts, seed)
        want_sets, want_off = ohb.index_sets(m, parts, seed)
        assert np.array_equal(sets.cpu().numpy(), want_sets)
        assert np.array_equal(off.cpu().numpy(), want_off)


def test_union_keys_round_trip_c4(env):
    torch, zr = env
    c = workloads.SPARSE_C4
    idx, val = workloads.sparse_c4()
    u_idx, _u_val, u_off = osp.aggregate(idx, val, c["n_parts"], c["part_seed"])
    hb = check(torch, zr, c["m"], c["n_parts"], c["part_seed"], u_idx)
    # the decoded keys are the partitioned union's keys, in its order
    bits, _woff = hb.encode(torch.from_numpy(u_idx).cuda())
    out = torch.empty(len(u_idx), dtype=torch.int32, device="cuda")
    koff = torch.empty(c["n_parts"] + 1, dtype=torch.int64, device="cuda")
    hb.decode(bits, out, koff)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), u_idx)
    assert np.array_equal(koff.cpu().numpy(), u_off)


def test_status_errors(env):
    torch, zr = env
    hb = zr.HashBitmap(1000, 4, 1)
    hb.encode(torch.tensor([3, 1000], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert hb.status() == zr.ZR_ERR_INPUT_UNSORTED
    keys = torch.arange(0, 1000, 2, dtype=torch.int32, device="cuda")
    bits, _ = hb.encode(keys)
    big = torch.full((600,), -1, dtype=torch.int32, device="cuda")
    koff = torch.empty(5, dtype=torch.int64, device="cuda")
    hb.decode(bits, big[:10], koff)
    torch.cuda.synchronize()
    assert hb.status() == zr.ZR_ERR_CAPACITY
    # nothing is written past the capacity
    assert bool((big[10:] == -1).all())


def test_padding_bit_and_foreign_directory(env):
    torch, zr = env
    m, parts = 5000, 3
    # a seed whose partition 0 ends inside a word
    seed = next(sd for sd in range(100) if ohb.index_sets(m, parts, sd)[1][1] % 32)
    hb = zr.HashBitmap(m, parts, seed)
    keys = torch.arange(0, m, 3, dtype=torch.int32, device="cuda")
    bits, woff = hb.encode(keys)
    torch.cuda.synchronize()
    out = torch.empty(m, dtype=torch.int32, device="cuda")
    koff = torch.empty(parts + 1, dtype=torch.int64, device="cuda")
    # a set padding bit past the end of partition 0's set
    w = woff.cpu().numpy()
    n0 = int(dir_counts(hb, m, parts, zr.ZR_HASH_RANGE)[0, -1])
    assert n0 % 32, "partition 0 must end inside a word for this case"
    bad = bits.clone()
    bad[int(w[1]) - 1] |= -(1 << 31)  # bit 31
    hb.decode(bad, out, koff)
    torch.cuda.synchronize()
    assert hb.status() == zr.ZR_ERR_INVALID_ARG
    # a directory built for another seed: every call reports it, and writes
    # stay inside the given buffers
    other = zr.HashBitmap(m, parts, seed + 1)
    hb.directory, saved = other.directory, hb.directory
    hb.encode(keys)
    torch.cuda.synchronize()
    assert hb.status() == zr.ZR_ERR_INVALID_ARG
    hb.decode(bits, out, koff)
    torch.cuda.synchronize()
    assert hb.status() == zr.ZR_ERR_INVALID_ARG
    # lengths that do not add up to M
    broken = saved.clone()
    hb.directory = broken
    dir_counts(hb, m, parts, zr.ZR_HASH_RANGE)[0, -1] += 1
    hb.encode(keys)
    torch.cuda.synchronize()
    assert hb.status() == zr.ZR_ERR_INVALID_ARG
    hb.directory = saved
    hb.encode(keys)
    torch.cuda.synchronize()
    assert hb.status() == zr.ZR_OK


def test_maximum_size_round_trip(env):
    """M = 2^31 - 1 and 256 partitions (the largest request: a 3 GB
    directory, 2^20 ranges, the last one ragged).  Properties that hold at
    any size: the directory's lengths are the partition sizes of h0 (their
    sum is M), and decode(encode(keys)) is the keys grouped by h0 and
    ascending inside each partition."""
    torch, zr = env
    m, parts, seed = (1 << 31) - 1, zr.ZR_MAX_PARTS, 77
    rng = np.random.default_rng(5)
    keys = np.unique(np.concatenate([
        rng.integers(0, m, size=200_000, dtype=np.int64),
        np.array([0, 1, 2047, 2048, m - 2048, m - 2, m - 1], dtype=np.int64)])).astype(np.int32)
    hb = zr.HashBitmap(m, parts, seed)
    lengths = dir_counts(hb, m, parts, zr.ZR_HASH_RANGE)[:, -1].cpu().numpy()
    assert int(lengths.sum()) == m and lengths.min() > 0
    bits, woff = hb.encode(torch.from_numpy(rng.permutation(keys)).cuda())
    torch.cuda.synchronize()
    assert hb.status() == zr.ZR_OK
    w = woff.cpu().numpy()
    assert np.array_equal(np.diff(w), (lengths + 31) // 32)
    out = torch.full((keys.size,), -1, dtype=torch.int32, device="cuda")
    koff = torch.empty(parts + 1, dtype=torch.int64, device="cuda")
    hb.decode(bits, out, koff)
    torch.cuda.synchronize()
    assert hb.status() == zr.ZR_OK
    p = osp.h0(keys.astype(np.int64), parts, seed)
    order = np.lexsort((keys, p))
    assert np.array_equal(out.cpu().numpy(), keys[order])
    want_koff = np.zeros(parts + 1, dtype=np.int64)
    want_koff[1:] = np.cumsum(np.bincount(p, minlength=parts))
    assert np.array_equal(koff.cpu().numpy(), want_koff)
    # the set bits total the keys
    ones = np.array([bin(i).count("1") for i in range(256)], dtype=np.int64)
    words = bits[: int(w[-1])].cpu().numpy().view(np.uint8)
    assert int(ones[words].sum()) == keys.size
