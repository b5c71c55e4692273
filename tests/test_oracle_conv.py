"""Pins of the oracle's DFlash-2 grouped dynamic convolution against what the mathematics fixes
(CPU only)."""
import numpy as np

from oracle import conv


def _case(seed, N=23, C=12, G=3, L=4, nblocks=4):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, C))
    k = rng.standard_normal((N, G, L))
    cuts = np.sort(rng.choice(np.arange(1, N), nblocks - 1, replace=False))
    block = np.zeros(N, dtype=np.int32)
    for c in cuts:
        block[c:] += 1
    return x, block, k


def test_one_tap_is_a_scaling_per_group():
    x, block, k = _case(1, L=1)
    y = conv.grouped_dynamic_conv(x, block, k)
    G, gs = k.shape[1], x.shape[1] // k.shape[1]
    want = x * np.repeat(k[:, :, 0], gs, axis=1)
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-14)


def test_one_block_with_fixed_taps_is_numpy_causal_convolution():
    rng = np.random.default_rng(2)
    N, C, G, L = 19, 8, 2, 5
    x = rng.standard_normal((N, C))
    taps = rng.standard_normal((G, L))
    k = np.broadcast_to(taps, (N, G, L)).copy()
    y = conv.grouped_dynamic_conv(x, np.zeros(N, dtype=np.int32), k)
    gs = C // G
    for c in range(C):
        want = np.convolve(x[:, c], taps[c // gs])[:N]     # y[i] = sum_t taps[t] x[i - t]
        np.testing.assert_allclose(y[:, c], want, rtol=1e-12, atol=1e-12)


def test_taps_never_cross_a_block_boundary():
    x, block, k = _case(3)
    y = conv.grouped_dynamic_conv(x, block, k)
    for b in np.unique(block):
        x2 = x.copy()
        x2[block == b] += 100.0                            # perturb one block only
        y2 = conv.grouped_dynamic_conv(x2, block, k)
        other = block != b
        np.testing.assert_array_equal(y2[other], y[other])
        assert not np.allclose(y2[block == b], y[block == b])
    # the first row of every block sees its own row only (tap 0)
    first = np.r_[True, block[1:] != block[:-1]]
    G, gs = k.shape[1], x.shape[1] // k.shape[1]
    np.testing.assert_allclose(y[first], (x * np.repeat(k[:, :, 0], gs, axis=1))[first], atol=1e-14)


def test_linear_in_rows_and_in_taps():
    x, block, k = _case(4)
    x2, _, k2 = _case(5)
    f = conv.grouped_dynamic_conv
    np.testing.assert_allclose(f(2.0 * x + x2, block, k), 2.0 * f(x, block, k) + f(x2, block, k), atol=1e-12)
    np.testing.assert_allclose(f(x, block, k - 3.0 * k2), f(x, block, k) - 3.0 * f(x, block, k2), atol=1e-12)
