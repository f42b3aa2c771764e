"""GPU parity: Zen's index sets and hash bitmap encode / decode (through the
C ABI) against the CPU oracle, bit for bit; the C4 union at full size."""

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


def check(torch, zr, m, parts, seed, keys):
    hb = zr.HashBitmap(m, parts, seed)
    sets, off = ohb.index_sets(m, parts, seed)
    assert np.array_equal(hb.sets.cpu().numpy(), sets)
    assert np.array_equal(hb.offsets.cpu().numpy(), off)
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


@pytest.mark.parametrize("parts", [1, 3, 8, 16, 64, 256])
def test_small_and_ragged(env, parts):
    torch, zr = env
    rng = np.random.default_rng(parts)
    for m in (1, 15, 33, 1000, 100_003):
        for density in (0.0, 0.3, 1.0):
            keys = np.nonzero(rng.random(m) < density)[0].astype(np.int32)
            check(torch, zr, m, parts, int(rng.integers(0, 1 << 62)), rng.permutation(keys))


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
    small = torch.full((10,), -1, dtype=torch.int32, device="cuda")
    koff = torch.empty(5, dtype=torch.int64, device="cuda")
    hb.decode(bits, small, koff)
    torch.cuda.synchronize()
    assert hb.status() == zr.ZR_ERR_CAPACITY
