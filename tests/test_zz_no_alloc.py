"""GPU test of dspark_d2t_check_noalloc, called through the C ABI.

Its verdicts must equal those of dspark_d2t_check (the workspace entry point) on the same maps,
on two calls in a row (the second finds the static bitmap dirty from the first). Collected last
so that it also runs after every other GPU test in the same process; it needs no earlier call.
"""
import ctypes

import numpy as np
import pytest
import torch

import dspark_inputs as di

pytestmark = pytest.mark.gpu

MAX_VT = 1 << 20


def _maps():
    g = di.generator(90, 0)
    V_d, V_t = 114688, 248100
    S = g.permutation(V_t)[:V_d].astype(np.int64)
    ok = S - np.arange(V_d, dtype=np.int64)
    dup = ok.copy()
    dup[V_d - 1] = ok[7] + 7 - (V_d - 1)                 # same target id as draft index 7
    low = ok.copy()
    low[100] = -101                                      # maps to -1
    high = ok.copy()
    high[5000] = V_t - 5000                              # maps to V_t
    edge = np.zeros(1000, dtype=np.int64)
    edge[999] = MAX_VT - 1 - 999                         # the largest id the static bitmap holds
    return [(ok, V_t), (dup, V_t), (low, V_t), (high, V_t), (edge, MAX_VT)]


def _noalloc(lib, d2t, V_t, inj):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    code = lib.dspark_d2t_check_noalloc(ctypes.c_void_p(d2t.data_ptr()), d2t.numel(), V_t, int(inj),
                                        ctypes.c_void_p(st.data_ptr()),
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0
    return st


def test_noalloc_verdicts_equal_workspace_entry_two_calls_in_a_row():
    import dspark_draft_selection_gb300 as ds
    lib = ds.lib()
    for d2t_h, V_t in _maps():
        d2t = torch.from_numpy(d2t_h).cuda()
        for inj in (True, False):
            for _ in range(2):
                want = ds.dspark_d2t_check(d2t, V_t, inj)
                got = _noalloc(lib, d2t, V_t, inj)
                torch.cuda.synchronize()
                assert int(got.item()) == int(want.item()), (V_t, inj)


def test_noalloc_refuses_vocabularies_beyond_its_bitmap():
    import dspark_draft_selection_gb300 as ds
    lib = ds.lib()
    d2t = torch.zeros(16, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    code = lib.dspark_d2t_check_noalloc(ctypes.c_void_p(d2t.data_ptr()), 16, MAX_VT + 1, 1,
                                        ctypes.c_void_p(st.data_ptr()), None)
    assert code == 1                                     # DSPARK_EINVAL, nothing launched
    torch.cuda.synchronize()
    assert int(st.item()) == 0
