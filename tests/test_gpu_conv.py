"""GPU parity of dspark_grouped_conv (DFlash-2 grouped dynamic convolution over packed block rows)
against the oracle. Float32 FMAs in tap order against float64 sums: each output is within
4 L 2^-24 of the sum of its terms' magnitudes."""
import numpy as np
import pytest
import torch

import dspark_inputs as di
from oracle import conv
from tests.gpu_util import as_f32, dev, host

pytestmark = pytest.mark.gpu


def _check(x, block, k, y):
    xf = as_f32(x).astype(np.float64)
    want = conv.grouped_dynamic_conv(xf, block, k)
    mag = conv.grouped_dynamic_conv(np.abs(xf), block, np.abs(k))       # sum of |terms|
    L = k.shape[2]
    bad = np.abs(y - want) > 4 * L * 2.0 ** -24 * mag + 1e-30
    assert not bad.any(), (np.argwhere(bad)[:5], y[bad][:5], want[bad][:5])


def _random_case(seed, N, C, G, L, dtype, blocks):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, C)).astype(np.float32)
    if dtype == "bf16":
        x = di.f32_to_bf16_bits(x)
    k = rng.standard_normal((N, G, L)).astype(np.float32)
    cuts = np.sort(rng.choice(np.arange(1, N), blocks - 1, replace=False)) if blocks > 1 else []
    block = np.zeros(N, dtype=np.int32)
    for c in cuts:
        block[c:] += 1
    return x, block, k


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N,C,G,L,blocks", [(37, 64, 8, 4, 6),      # vector path, ragged blocks
                                            (50, 24, 3, 16, 9),     # vector path, 16 taps
                                            (29, 30, 5, 3, 4),      # groups of 6 channels: element path
                                            (13, 7, 1, 2, 13)])     # every row its own block
def test_small_cases_match_the_oracle(dtype, N, C, G, L, blocks):
    import dspark_draft_selection_gb300 as ds
    x, block, k = _random_case(N * 131 + C, N, C, G, L, dtype, blocks)
    y = host(ds.dspark_grouped_conv(dev(x), dev(k), dev(block)))
    _check(x, block, k, y)


def test_row_stride_and_empty_batch():
    import dspark_draft_selection_gb300 as ds
    x, block, k = _random_case(7, 21, 40, 4, 4, "f32", 3)
    wide = torch.zeros((21, 56), dtype=torch.float32, device="cuda")
    wide[:, :40] = dev(x)
    yw = torch.full((21, 48), 9.5, dtype=torch.float32, device="cuda")
    ds.dspark_grouped_conv(wide[:, :40], dev(k), dev(block), out=yw[:, :40])
    y = host(yw)
    _check(x, block, k, y[:, :40])
    assert np.all(y[:, 40:] == 9.5)                                  # the padding is untouched
    e = ds.dspark_grouped_conv(torch.zeros((0, 40), device="cuda"), torch.zeros((0, 4, 4), device="cuda"),
                               torch.zeros((0,), dtype=torch.int32, device="cuda"))
    assert e.shape == (0, 40)


def test_full_size_packed_blocks():
    """128 requests x (1 context row + 7 block rows) x 5,120 channels, 32 groups, 4 taps; the
    oracle checks the first 16 requests' rows and the last request's rows."""
    import dspark_draft_selection_gb300 as ds
    w = di.conv_workload()
    y = host(ds.dspark_grouped_conv(dev(w["x"]), dev(w["k"]), dev(w["block"])))
    per = 1 + w["B"]
    for lo, hi in ((0, 16 * per), (w["N"] - per, w["N"])):
        _check(w["x"][lo:hi], w["block"][lo:hi], w["k"][lo:hi], y[lo:hi])
