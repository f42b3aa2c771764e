"""Pins for the hash-bitmap oracle (CPU only): Zen's Figure 10 worked
example, the size property of section 3.3.2 (all servers' bitmaps total |G|
bits), brute force against Python sets, and the round trip."""

import os

import numpy as np
import pytest

from oracle import hash_bitmap as hb
from oracle import sparse

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "zen_fig10_hash_bitmap.txt")


def read_golden():
    d = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        k, *v = line.split()
        d[k] = [int(x) for x in v]
    return d


def test_figure10_worked_example():
    g = read_golden()
    i0 = np.array(g["I_0"]) - 1  # to 0-based indices
    nz = np.array(g["nonzero"]) - 1
    bm = hb.encode(i0, nz)
    bits = [(int(bm[j // 32]) >> (j % 32)) & 1 for j in range(i0.size)]
    assert bits == g["bits"]
    assert (hb.decode(i0, bm) + 1).tolist() == g["nonzero"]


@pytest.mark.parametrize("m,n,seed", [(15, 3, 0), (1000, 4, 1), (4097, 16, 7), (100_000, 64, 3)])
def test_index_sets_partition_the_range(m, n, seed):
    sets, off = hb.index_sets(m, n, seed)
    assert off[0] == 0 and off[-1] == m
    assert sorted(sets.tolist()) == list(range(m))
    for i in range(n):
        part = sets[off[i]:off[i + 1]]
        assert np.all(np.diff(part) > 0)
        if part.size:
            assert set(sparse.h0(part, n, seed).tolist()) == {i}
    # every server's bitmap together: |G| bits, at most one padded word each
    total_words = sum(hb.words(int(off[i + 1] - off[i])) for i in range(n))
    assert m / 32 <= total_words <= m / 32 + n


def test_brute_force_and_round_trip():
    rng = np.random.default_rng(4)
    for trial in range(30):
        m = int(rng.integers(1, 300))
        n = int(rng.integers(1, 9))
        seed = int(rng.integers(0, 1 << 63))
        nz = np.unique(rng.integers(0, m, size=int(rng.integers(0, m + 1))))
        bm, woff = hb.encode_all(m, n, seed, nz)
        sets, off = hb.index_sets(m, n, seed)
        for i in range(n):
            part = [int(v) for v in sets[off[i]:off[i + 1]]]
            words = bm[woff[i]:woff[i + 1]]
            for j, x in enumerate(part):
                assert ((int(words[j // 32]) >> (j % 32)) & 1) == (x in set(nz.tolist()))
            for j in range(len(part), 32 * len(words)):  # padding bits are zero
                assert ((int(words[j // 32]) >> (j % 32)) & 1) == 0
        keys, koff = hb.decode_all(m, n, seed, bm, woff)
        assert sorted(keys.tolist()) == nz.tolist()
        for i in range(n):
            seg = keys[koff[i]:koff[i + 1]]
            assert np.all(np.diff(seg) > 0)
            if seg.size:
                assert set(sparse.h0(seg, n, seed).tolist()) == {i}


def test_decoded_union_equals_partitioned_aggregate_keys():
    # The servers' decoded indices are exactly the partitioned union's keys.
    rng = np.random.default_rng(6)
    m, n, seed = 5000, 8, 2
    lists = [np.unique(rng.integers(0, m, size=400)).astype(np.int32) for _ in range(4)]
    vals = [np.ones(a.size, np.float32) for a in lists]
    u_idx, _u_val, u_off = sparse.aggregate(lists, vals, n, seed)
    bm, woff = hb.encode_all(m, n, seed, u_idx)
    keys, koff = hb.decode_all(m, n, seed, bm, woff)
    assert np.array_equal(keys, u_idx) and np.array_equal(koff, u_off)
