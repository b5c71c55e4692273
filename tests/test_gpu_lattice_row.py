"""The block sampler's lattice-row branch (dspark_lattice_row_sample), GPU against the oracle:
full-row samples of the walk row after the token before, ending at a token outside the candidates."""
import numpy as np
import pytest
import torch

import dspark_inputs as di
from oracle import draft as od
from oracle.sampling import draw_margin
from tests.gpu_util import as_f32, dev, host

pytestmark = pytest.mark.gpu


def _run(w, K, T, top_p, min_p, record):
    import dspark_draft_selection_gb300 as ds
    R, B = w["R"], w["B"]
    kw = dict(d2t=dev(w["d2t"]), V_t=w["V_t"]) if w["d2t"] is not None else {}
    cd, ct, cv, st = ds.dspark_topk(dev(w["logits"]), B, K, **kw)
    trans, gate, st2 = ds.dspark_lattice_score(ct, dev(w["prev"]), dev(w["E"]), dev(w["W"]))
    V = w["V_d"]
    if record == "dense":
        q = ds.dense_record(R * B, V)
    else:
        q = (torch.full((R * B, 4096), -1, dtype=torch.int32, device="cuda"),
             torch.zeros((R * B, 4096), dtype=torch.float32, device="cuda"),
             torch.zeros((R * B,), dtype=torch.int32, device="cuda"))
    tgt, idx, nd, st3 = ds.dspark_lattice_row_sample(dev(w["logits"]), B, cd, cv, trans, temperature=T, top_p=top_p,
                                                     min_p=min_p, seed=dev(w["seed"]), step=dev(w["step"]), q=q, **kw)
    torch.cuda.synchronize()
    for s in (st, st2, st3):
        assert ds.read_status(s) == 0
    return host(cd), host(cv), host(trans), host(tgt), host(idx), host(nd), tuple(host(t) for t in q)


def _check(w, K, T, top_p, min_p, record, got, requests):
    cd, cv, trans, tgt, idx, nd, rec = got
    B = w["B"]
    rows = as_f32(w["logits"])
    amb = 0
    for r in requests:
        toks, recs = od.lattice_row_sample(rows[r * B:(r + 1) * B], cd[r], cv[r], trans[r], T, top_p,
                                           int(w["seed"][r]), int(w["step"][r]), min_p)
        n = len(toks)
        if nd[r] != n or not np.array_equal(idx[r, :n], toks):
            # admissible only at a rounding-level draw boundary of the first differing position
            j = next(j for j in range(min(n, nd[r])) if idx[r, j] != toks[j])
            from oracle.philox import uniform
            m = draw_margin(recs[j]["w"], recs[j]["kept"], float(uniform(int(w["seed"][r]), int(w["step"][r]), j, 0)))
            assert m < 1e-12, (r, j, idx[r, :nd[r]], toks)
            amb += 1
            continue
        assert np.all(idx[r, n:] == -1) and np.all(tgt[r, n:] == -1)
        assert np.array_equal(tgt[r, :n], od.d2t_map(toks, w["d2t"]))
        for j in range(n):
            i = r * B + j
            if record == "sparse":
                ids, qp, qn = rec
                k = len(recs[j]["kept"])
                assert qn[i] == k and np.array_equal(ids[i, :k], od.d2t_map(recs[j]["kept"], w["d2t"]))
                np.testing.assert_allclose(qp[i, :k], recs[j]["q"], rtol=2e-7, atol=0)
            else:
                z, zmax, wsum, wcut, icut = rec
                assert np.array_equal(z[i], recs[j]["z"]) and zmax[i] == recs[j]["zmax"]
                assert abs(wsum[i] - recs[j]["wsum"]) <= 1e-12 * recs[j]["wsum"]
                assert wcut[i] == recs[j]["w_cut"] and icut[i] == recs[j]["i_cut"]
        if record == "sparse":
            assert np.all(rec[2][r * B + n:(r + 1) * B] == 0)
    return amb


@pytest.mark.parametrize("T,top_p,min_p,record", [(1.0, 1.0, 0.0, "dense"), (0.8, 0.95, 0.0, "sparse"),
                                                  (0.7, 1.0, 0.01, "sparse"), (1.2, 0.9, 0.001, "dense")])
def test_lattice_row_branch_matches_the_oracle(T, top_p, min_p, record):
    w = di.lattice_workload(111, R=8, B=15, V_d=3000, V_t=7000, K=64, rank=64, pruned=True, with_seeds=True,
                            head_sigma=0.4)
    got = _run(w, 64, T, top_p, min_p, record)
    assert _check(w, 64, T, top_p, min_p, record, got, range(w["R"])) <= 1
    nd = got[5]
    assert nd.min() >= 1 and nd.max() <= w["B"]


def test_lattice_row_branch_pruned_config_full_size():
    """The pruned DSpark draft's shape (16 requests x block 15, 114,688 draft ids over 248,100):
    every request's block against the oracle, with a dense record."""
    w = di.config3()
    got = _run(w, w["K"], w["temperature"], w["top_p"], 0.0, "dense")   # nuclei of tens of thousands of ids
    assert _check(w, w["K"], w["temperature"], w["top_p"], 0.0, "dense", got, range(w["R"])) <= 1
