"""GPU parity of dspark_d2t_check against the oracle's verdict (exact status codes).

DFlash commit on the d2t checks: one entry per draft logit, every mapped id inside the target
vocabulary, and a one-to-one map where drafting samples.
"""
import numpy as np
import pytest

import dspark_draft_selection_gb300 as ds
import dspark_inputs as di
from gpu_util import dev
from oracle import draft as od

pytestmark = pytest.mark.gpu


def gpu_verdict(d2t, V_t, injective, ws=None):
    st = ds.dspark_d2t_check(dev(np.asarray(d2t, dtype=np.int64)), V_t, injective, ws=ws)
    return ds.read_status(st)


def pruned_map(cid, V_d, V_t):
    S = di.generator(cid, 99).permutation(V_t)[:V_d].astype(np.int64)
    return S - np.arange(V_d, dtype=np.int64)


@pytest.mark.parametrize("V_d,V_t", [(1, 1), (7, 9), (1000, 1000), (114688, 248100), (151936, 151936)])
def test_valid_maps(V_d, V_t):
    d2t = pruned_map(V_d, V_d, V_t)
    for inj in (True, False):
        assert od.d2t_check(d2t, V_t, inj) == od.OK
        assert gpu_verdict(d2t, V_t, inj) == od.OK


@pytest.mark.parametrize("where", [0, 1, 4095, 4096, 114687])
@pytest.mark.parametrize("kind", ["low", "high", "dup"])
def test_single_fault_anywhere(where, kind):
    V_d, V_t = 114688, 248100
    d2t = pruned_map(3, V_d, V_t)
    bad = d2t.copy()
    if kind == "low":
        bad[where] = -where - 1                        # maps to -1
    elif kind == "high":
        bad[where] = V_t - where                       # maps to V_t
    else:
        other = (where + 77) % V_d
        bad[where] = other + d2t[other] - where        # same target id as `other`
    for inj in (True, False):
        want = od.d2t_check(bad, V_t, inj)
        assert want == (od.OK if (kind == "dup" and not inj) else od.EDUP if kind == "dup" else od.ERANGE)
        assert gpu_verdict(bad, V_t, inj) == want


def test_range_wins_over_duplicates_and_workspace_is_reused():
    V_d, V_t = 50000, 60000
    d2t = pruned_map(4, V_d, V_t)
    ws = ds.workspace(ds.OP_D2T_CHECK, 1, 1, V_t, 0, "cuda")
    both = d2t.copy()
    both[10] = both[11] + 1                              # duplicate of 11
    both[20000] = V_t                                    # out of range
    assert od.d2t_check(both, V_t, True) == od.ERANGE
    # the same workspace, dirty from earlier calls, gives the same verdicts every time
    for _ in range(3):
        assert gpu_verdict(both, V_t, True, ws=ws) == od.ERANGE
        assert gpu_verdict(d2t, V_t, True, ws=ws) == od.OK
        dup = d2t.copy()
        dup[V_d - 1] = d2t[0] - (V_d - 1)
        assert gpu_verdict(dup, V_t, True, ws=ws) == od.EDUP


def test_identity_map_and_huge_offsets():
    V = 151936
    assert gpu_verdict(np.zeros(V, np.int64), V, True) == od.OK
    far = np.zeros(V, np.int64)
    far[5] = 2**40                                     # far outside, no int32 wrap-around
    assert od.d2t_check(far, V, False) == od.ERANGE
    assert gpu_verdict(far, V, False) == od.ERANGE
    neg = np.zeros(V, np.int64)
    neg[V - 1] = -(2**40)
    assert gpu_verdict(neg, V, True) == od.ERANGE
