"""CPU oracle for the gradient-aggregation hot path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the pages define, written in numpy and pure Python:

* ``oracle.ring``     -- the literal ring all-reduce (Reduce-Scatter in ring
  order, then AllGather), SkipReduce slice skipping (Static and Random), the
  1/N (or DropReduce 1/(N-k)) average, per-worker traffic counters, and the
  naive all-reduce used as a cross-check.
* ``oracle.bf16``     -- bf16 widening and round-to-nearest-even narrowing on
  raw bit patterns.
* ``oracle.splitmix`` -- the SplitMix64 counter generator (Steele, Lea and
  Flood, OOPSLA 2014) that draws the Random SkipReduce offset and the
  partition-hash parameters.
* ``oracle.sparse``   -- the COO union with rank-ordered sums and the h0
  partition (Zen, Problem 1 and Algorithm 1's first-level hash).
* ``oracle.stats``    -- overlap, densification, skew and imbalance ratios
  (Zen, Definitions 3, 4, 5 and 8).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import it.  The product path (the CUDA library under
``gradient_synchronisation_gb300/`` and its binding) never imports, links or
calls anything here, and nothing here imports the product path.  The two share
only the seeded input generators in ``workloads/``, which hold none of the
method's arithmetic.

Every function cites the passage it follows as "page title, section /
algorithm / equation".  The pages are:

* "Zen: Empowering Distributed Training with Sparsity-driven Data
  Synchronization" (OSDI'25 digest) -- "Zen" below.
* "SkipReduce: (Interconnection) Network Sparsity to Accelerate Distributed
  Machine Learning" (MICRO'25 digest) -- "SkipReduce" below.
* "15642 Machine Learning Systems: Distributed Training and Parallelization"
  (CMU course notes) -- "15-642 notes" below.

Parity status: every function here is pinned by a ``-m "not gpu"`` test against
something other than itself (closed forms, brute force, symbolic fold order,
a library routine for a special case); none is "parity unpinned".
"""

from . import bf16, ring, sparse, splitmix, stats  # noqa: F401
