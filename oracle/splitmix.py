"""SplitMix64 counter generator -- oracle side (test infrastructure).

The pages draw the Random SkipReduce slice offset from a generator seeded by
the iteration count, shared by every GPU (SkipReduce, section 4.3 "Random
SkipReduce" and Figure 6), and Zen's first-level hash h0 from seeded universal
hash functions broadcast at start (Zen, section 4 "Implementation").  They do
not name a generator we can reproduce (cuRAND's sequence and MurmurHash's
constants are not on the pages), so both sides implement one published
counter-based generator from its definition:

    SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast Splittable Pseudorandom
    Number Generators", OOPSLA 2014): the state advances by the odd constant
    gamma = 0x9E3779B97F4A7C15, and each output is the 64-bit finaliser
    z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB;
    z ^= z >> 31 applied to the new state.

Output number i (0-based) of the generator seeded with s is therefore
mix(s + (i + 1) * gamma mod 2**64).  This file computes it with Python
integers; the CUDA side has its own independent implementation.
"""

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15


def mix64(z):
    """The SplitMix64 output finaliser on one 64-bit integer."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def output(seed, i):
    """Output number ``i`` (0-based) of SplitMix64 seeded with ``seed``."""
    return mix64((seed + (i + 1) * GAMMA) & MASK64)


def outputs(seed, indices):
    """``output(seed, i)`` for every i of an integer array, in numpy uint64
    arithmetic (which wraps mod 2**64, as the definition does)."""
    import numpy as np

    i = np.asarray(indices, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & MASK64) + (i + np.uint64(1)) * np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def sequence(seed, count):
    """The first ``count`` outputs, by stepping the state (not by ``output``)."""
    state = seed & MASK64
    out = []
    for _ in range(count):
        state = (state + GAMMA) & MASK64
        out.append(mix64(state))
    return out


def range_reduce(h32, n):
    """Map a 32-bit value uniformly onto [0, n) by the multiply-high rule
    floor(h32 * n / 2**32)."""
    return (h32 * n) >> 32


def random_offset(seed, step, n):
    """Random SkipReduce slice offset o in [0, n) for iteration ``step``.

    SkipReduce, section 4.3: every GPU shifts its slice indices by the same
    per-iteration offset, derived from a seed and the iteration count.  Here o
    is the top 32 bits of output number ``step`` of SplitMix64(seed), range
    reduced onto [0, n).
    """
    return range_reduce(output(seed, step) >> 32, n)


def h0_params(part_seed):
    """Parameters (a, b) of the first-level hash h0: a odd, both 64-bit.

    a = output 0 of SplitMix64(part_seed) with its low bit set; b = output 1.
    """
    return output(part_seed, 0) | 1, output(part_seed, 1)
