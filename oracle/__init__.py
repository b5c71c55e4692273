"""CPU oracle for the DFlash/DSpark block-draft selector and verifier.

TEST INFRASTRUCTURE ONLY. Plain, slow numpy code that states what the hot path computes,
step by step, in the pages' order. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it; the library never does, and shares no code,
header, table or constant generator with it. Inputs come from ``dspark_inputs`` (random
numbers only).

Modules and what pins them (the tests under ``tests/test_oracle_*.py``):
  fp32      correctly rounded float32 FMA emulation (pinned against exact rational
            arithmetic) and the softmax weight function (pinned against the exponential's
            error bound and w(0) = 1);
  philox    Philox4x32-10 (pinned by the generator's published known-answer vectors) and
            the 53-bit double uniform (closed-form extremes, moments);
  sampling  temperature softmax, top-p nucleus, multinomial draw (pinned by chi-square fits,
            by an independent thresholded-nucleus construction, by the pages' worked
            example of float versus double sums, and by T -> 0 equal to argmax);
  draft     row transform, Top-K, d2t, gate, lattice, max-sum / greedy / sampled chains
            (pinned by full sorts, exhaustive enumeration of all K^B chains, zero-table and
            K = V reductions, d2t round trips, and hand-computed rank-1 lattices);
  walk      dense Markov walk (pinned by the zero-table and K = V reductions);
  verify    rejection-sampling verification (pinned by chi-square fits of the emitted token
            to p, the closed-form acceptance rate sum min(p, q), the pages' worked example,
            and greedy acceptance equal to argmax matching);
  conv      DFlash-2 grouped dynamic convolution over packed block rows (pinned by one tap
            equal to a per-group scaling, one block with fixed taps equal to numpy's causal
            convolution of every channel, block isolation under perturbation, linearity).
No function here is "parity unpinned".
"""
from . import conv, draft, fp32, philox, sampling, verify, walk  # noqa: F401
