"""Pins for the oracle's bf16 rounding and its SplitMix64 generator (CPU only).

* bf16: the oracle's bit-level round-to-nearest-even is compared with torch's
  CPU float32 -> bfloat16 cast (an independent implementation) on random bit
  patterns, every exact halfway case of random mantissas, and the special
  values.
* SplitMix64: the oracle's generator reproduces published known-answer
  vectors (tests/golden/splitmix64_kat.txt).
"""

import os

import numpy as np
import torch

from oracle import bf16, splitmix

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def torch_round(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def compare(bits):
    x = bits.view(np.float32)
    ours = bf16.round_rne(x)
    ref = torch_round(x)
    nan = np.isnan(x)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    # NaN payloads are not pinned; both sides must give a NaN.
    assert np.isnan(bf16.widen(ours[nan])).all()


def test_random_patterns():
    rng = np.random.default_rng(1)
    compare(rng.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32))


def test_halfway_cases():
    rng = np.random.default_rng(2)
    hi = rng.integers(0, 1 << 16, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    compare((hi << np.uint32(16)) | np.uint32(0x8000))
    compare((hi << np.uint32(16)) | np.uint32(0x7FFF))
    compare((hi << np.uint32(16)) | np.uint32(0x8001))


def test_specials():
    vals = np.array([0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000,
                     0x7F800001, 0xFFC12345, 0x7F7FFFFF, 0x7F7F8000, 0x7F7F7FFF,
                     0x00000001, 0x00008000, 0x00018000, 0x807FFFFF, 0x3F808000,
                     0x3F818000], dtype=np.uint32)
    compare(vals)
    assert bf16.round_rne(np.array([np.float32(3.4028235e38)]))[0] == 0x7F80  # rounds to inf


def test_widen_exact():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    ours = bf16.widen(bits)
    ok = ~np.isnan(t)
    np.testing.assert_array_equal(ours[ok].view(np.uint32), t[ok].view(np.uint32))
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(t))


def test_splitmix_known_answers():
    with open(os.path.join(GOLDEN, "splitmix64_kat.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 2
    for row in rows:
        seed = int(row[0], 0)
        want = [int(v, 0) for v in row[1:]]
        assert splitmix.sequence(seed, len(want)) == want
        assert [splitmix.output(seed, i) for i in range(len(want))] == want


def test_range_reduce_bounds():
    for n in (1, 2, 3, 8, 16, 64):
        assert splitmix.range_reduce(0, n) == 0
        assert splitmix.range_reduce((1 << 32) - 1, n) == n - 1


def test_vectorised_outputs_equal_scalar_definition():
    import numpy as np

    from oracle import splitmix as sm

    rng = np.random.default_rng(5)
    for seed in (0, 1, 0x9E3779B97F4A7C15, (1 << 64) - 1, 123456789):
        idx = np.concatenate([np.arange(40), rng.integers(0, 1 << 40, size=200)])
        got = sm.outputs(seed, idx)
        want = [sm.output(seed, int(i)) for i in idx]
        assert [int(v) for v in got] == want
