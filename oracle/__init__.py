"""CPU oracle for the ring-ordered collectives -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may import anything from this package.  The library
(``a2a_ring_ordered_gb300``) never imports it, and it imports nothing from the
library: the two share no code.  The only shared module is the seeded input
generator ``a2a_ring_ordered_gb300.workloads``, which holds no arithmetic of
the method.

What it is: a plain, slow, obviously correct restatement of the pages'
collectives in numpy.

* ``ring``        -- the literal ring all-reduce: a reduce-scatter phase of
                     p-1 steps followed by an all-gather phase of p-1 steps,
                     simulated rank by rank and step by step with explicit
                     messages and per-rank byte counters.  Sources:
                     "Networks and Collective Communication" section 5.1
                     (ring: bandwidth optimal) and Exercise 2; "dist_train",
                     section "Ring Algorithm"; "LLM Distributed Training
                     Collectives", section "Ring AllReduce".
* ``pointwise``   -- the same fold written per output element (used to check
                     sampled outputs of huge buffers).
* ``collectives`` -- the primitives' definitions ("Networks and Collective
                     Communication" section 4.1; "dist_train", section
                     "Collective Communication Primitives"): broadcast,
                     reduce, scatter, gather, all-gather, all-to-all(v).
* ``bf16``        -- fp32 -> bf16 round-to-nearest-even by the published bit
                     method, and the exact bf16 -> fp32 widening.

Arithmetic is fp32 for floating point, because the method fixes it: the
partial sums travel and accumulate in fp32 in a fixed ring order, and bf16
results are rounded once at the end.  int32 sums wrap around (two's
complement).

Data conventions: a rank buffer is a 1-D numpy array; fp32 is ``float32``,
int32 is ``int32``, bf16 is ``uint16`` holding the raw bit pattern.

Every function is pinned by ``tests/test_oracle_*.py`` against things other
than itself: the worked example of section 4.1 (outputs derived by hand),
exact integer sums by brute force, a fold-order discriminator, the identities
of section 4.2, the byte lower bounds of section 4.3, numpy's ``array_split``
and torch's bf16 cast.  No function here is "parity unpinned".
"""
