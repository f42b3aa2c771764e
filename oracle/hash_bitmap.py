"""Zen's hash bitmap -- oracle side (test infrastructure only).

Zen, section 3.3.2 "Hash bitmap", Figure 10 and Algorithm 2: with the
first-level hash h0 of Algorithm 1, the indices a worker pushes to server i
are I_i = {idx in [0, |G|) : h0(idx) = i}, fixed for the whole training run
(computed once, offline, and sorted).  Server i describes the nonzeros of
its aggregated partition by one bit per element of I_i instead of one bit
per element of the whole range: hash_bitmap_encode sets bit j when I_i[j]
is a nonzero index, and hash_bitmap_decode maps the set bits j back to the
indices I_i[j].  Because the I_i are disjoint and cover [0, |G|), the bitmaps
of all servers total |G| bits (|G|/32 words) however many servers there are.

Readings: indices are 0-based (the pages count from 1); bit j of a bitmap is
bit (j mod 32) of 32-bit word floor(j / 32), least significant bit first;
the last word of a bitmap is zero-padded.
"""

import numpy as np

from . import sparse


def index_sets(m, n_parts, seed):
    """All I_i, concatenated in partition order (each ascending), and
    offsets[n_parts + 1] (I_i = sets[offsets[i]:offsets[i+1]])."""
    idx = np.arange(m, dtype=np.int64)
    p = sparse.h0(idx, n_parts, seed)
    order = np.argsort(p, kind="stable")
    counts = np.bincount(p, minlength=n_parts)
    offsets = np.zeros(n_parts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    return idx[order].astype(np.int32), offsets


def words(nbits):
    return (nbits + 31) // 32


def encode(index_set, nonzero):
    """Hash bitmap of one server: bit j set iff index_set[j] is in
    ``nonzero``.  Returns uint32 words."""
    index_set = np.asarray(index_set, dtype=np.int64)
    present = np.isin(index_set, np.asarray(nonzero, dtype=np.int64))
    j = np.nonzero(present)[0]
    out = np.zeros(words(index_set.size), dtype=np.uint64)
    np.bitwise_or.at(out, j // 32, np.uint64(1) << (j % 32).astype(np.uint64))
    return out.astype(np.uint32)


def decode(index_set, bitmap):
    """Indices index_set[j] for every set bit j, ascending in j."""
    index_set = np.asarray(index_set, dtype=np.int32)
    bitmap = np.asarray(bitmap, dtype=np.uint32)
    j = np.arange(index_set.size, dtype=np.int64)
    bit = (bitmap[j // 32] >> (j % 32).astype(np.uint32)) & np.uint32(1)
    return index_set[bit == 1]


def encode_all(m, n_parts, seed, nonzero):
    """Every server's hash bitmap for one set of nonzero indices (e.g. the
    union of the workers' lists), concatenated in partition order, with
    word offsets[n_parts + 1]."""
    sets, off = index_sets(m, n_parts, seed)
    parts = [encode(sets[off[i]:off[i + 1]], nonzero) for i in range(n_parts)]
    woff = np.zeros(n_parts + 1, dtype=np.int64)
    woff[1:] = np.cumsum([p.size for p in parts])
    return (np.concatenate(parts) if parts else np.zeros(0, np.uint32)), woff


def decode_all(m, n_parts, seed, bitmaps, woff):
    """Inverse of ``encode_all``: the nonzero indices, partition-major (each
    partition ascending), with key offsets[n_parts + 1]."""
    sets, off = index_sets(m, n_parts, seed)
    keys = [decode(sets[off[i]:off[i + 1]], bitmaps[woff[i]:woff[i + 1]]) for i in range(n_parts)]
    koff = np.zeros(n_parts + 1, dtype=np.int64)
    koff[1:] = np.cumsum([k.size for k in keys])
    return (np.concatenate(keys) if keys else np.zeros(0, np.int32)), koff
