"""CPU oracle of the ZeRO gradient-bucket reduction -- TEST INFRASTRUCTURE.

A plain, slow, obviously correct restatement of what the reduction computes,
written from the pages that define it, in numpy and plain C on the host.  It exists to
check the CUDA library, never to stand in for it: only the test suite, the
package smoke check and the bench's CPU-baseline leg may import it.  It shares
no code with the CUDA path (the only common module is the seeded input
generator, which holds none of the reduction's arithmetic).

Modules
  bf16     -- bf16 <-> fp32 bit conversions (round to nearest, ties to even)
  ring     -- explicit simulation of the ring reduce-scatter / all-gather /
              all-reduce rounds with per-link messages, a round trace and
              traffic counters
  flatten  -- gradient-bucket formation and the flat-bucket gather
  ring_c   -- loader of ring_sim.c, the same ring rounds and flat-bucket
              gather restated in plain C (compiled by the package build step
              with the host compiler), which the bench's CPU legs time

Every function is pinned by tests against values the pages print, closed
forms, invariants or exact (rational) brute force; none is "parity unpinned".
"""
from . import bf16, flatten, ring  # noqa: F401
