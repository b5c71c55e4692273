"""Philox4x32-10 counter-based generator and the 53-bit double uniform (oracle; test infrastructure only).

The pages leave the random engine unnamed; what they fix is that a multinomial draw and
the acceptance test of rejection sampling each take a double uniform built from two
outputs of the engine (openvino.genai PR #4847, commit on drawing with a double
uniform), and that the draft and the verifier draw from independently seeded streams
(same PR, commit on exact sampled speculative decoding). The engine used here is
Philox4x32 with 10 rounds, written from its published definition in Salmon, Moraes,
Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11): each round
multiplies words 0 and 2 by the two Philox multipliers, swaps and xors the high halves
with the other words and the key, and the key is bumped by the two Weyl constants
between rounds.

Stream layout (one Philox block per decision):
    key     = (seed mod 2^32, seed >> 32)
    counter = (step mod 2^32, position, purpose * 2^20 + draw, step >> 32)
    purpose 0 = draft draw, 1 = acceptance test, 2 = residual or bonus draw.
The double uniform from outputs (x0, x1) is ((x0 >> 5) * 2^26 + (x1 >> 6)) * 2^-53,
the 53-bit construction of Matsumoto and Nishimura's genrand_res53; it lies in [0, 1).
"""
from __future__ import annotations

import numpy as np

MASK32 = np.uint64(0xFFFFFFFF)
PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint64(0x9E3779B9)
PHILOX_W1 = np.uint64(0xBB67AE85)

PURPOSE_DRAFT = 0
PURPOSE_ACCEPT = 1
PURPOSE_RESIDUAL = 2


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Ten Philox rounds on 32-bit words held in uint64 arrays; returns (x0, x1, x2, x3)."""
    c0, c1, c2, c3, k0, k1 = (np.asarray(v, dtype=np.uint64) & MASK32 for v in (c0, c1, c2, c3, k0, k1))
    for rnd in range(10):
        p0 = PHILOX_M0 * c0            # < 2^64: exact in uint64
        p1 = PHILOX_M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0) & MASK32, lo1, (hi0 ^ c3 ^ k1) & MASK32, lo0
        k0 = (k0 + PHILOX_W0) & MASK32
        k1 = (k1 + PHILOX_W1) & MASK32
    return c0, c1, c2, c3


def uniform53_from(x0, x1) -> np.ndarray:
    a = (np.asarray(x0, dtype=np.uint64) >> np.uint64(5)).astype(np.float64)
    b = (np.asarray(x1, dtype=np.uint64) >> np.uint64(6)).astype(np.float64)
    return (a * 67108864.0 + b) * (1.0 / 9007199254740992.0)


def uniform(seed, step, position, purpose, draw=0) -> np.ndarray:
    """Double uniform in [0, 1) for (seed, step, position, purpose, draw); broadcasts."""
    seed = np.asarray(seed, dtype=np.uint64)
    step = np.asarray(step, dtype=np.uint64)
    position = np.asarray(position, dtype=np.uint64)
    word2 = (np.asarray(purpose, dtype=np.uint64) << np.uint64(20)) + np.asarray(draw, dtype=np.uint64)
    x0, x1, _, _ = philox4x32_10(step & MASK32, position, word2, step >> np.uint64(32),
                                 seed & MASK32, seed >> np.uint64(32))
    return uniform53_from(x0, x1)
