"""Pins for the oracle's Philox4x32-10 stream and its double uniform."""
import numpy as np

from oracle.philox import philox4x32_10, uniform, uniform53_from

# Known-answer vectors published with the Random123 library (Salmon et al., SC'11) for
# philox4x32 with 10 rounds: (counter words, key words) -> output words.
KAT = [
    ((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2, (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


def test_philox_known_answers():
    for ctr, key, want in KAT:
        got = philox4x32_10(*ctr, *key)
        assert tuple(int(x) for x in got) == want


def test_uniform53_extremes():
    assert uniform53_from(0, 0) == 0.0
    top = uniform53_from(0xFFFFFFFF, 0xFFFFFFFF)
    assert top == 1.0 - 2.0 ** -53 and top < 1.0
    # the two words contribute disjoint bit ranges: 27 high bits, 26 low bits
    assert uniform53_from(1 << 5, 0) == 2.0 ** -27
    assert uniform53_from(0, 1 << 6) == 2.0 ** -53


def test_uniform_moments_and_streams():
    n = 1_000_000
    u = uniform(12345, np.arange(n, dtype=np.uint64), 3, 0)
    assert u.min() >= 0.0 and u.max() < 1.0
    se = np.sqrt(1.0 / 12.0 / n)
    assert abs(u.mean() - 0.5) < 5 * se
    assert abs(u.var() - 1.0 / 12.0) < 5 * np.sqrt(1.0 / 180.0 / n)
    # purposes and positions give unrelated streams
    v = uniform(12345, np.arange(n, dtype=np.uint64), 3, 1)
    w = uniform(12345, np.arange(n, dtype=np.uint64), 4, 0)
    for other in (v, w):
        assert abs(np.corrcoef(u, other)[0, 1]) < 5 / np.sqrt(n)
    # a 64-bit seed and step use both halves
    a = uniform(np.uint64(1), np.uint64(7), 0, 0)
    b = uniform(np.uint64(1 + (1 << 32)), np.uint64(7), 0, 0)
    c = uniform(np.uint64(1), np.uint64(7 + (1 << 32)), 0, 0)
    assert len({float(a), float(b), float(c)}) == 3
