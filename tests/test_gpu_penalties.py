"""Repetition / presence penalties in the lattice walks (greedy and sampled), over each request's
history and the tokens drafted before, GPU against the oracle."""
import numpy as np
import pytest
import torch

import dspark_inputs as di
from oracle import draft as od
from tests.gpu_util import dev, host

pytestmark = pytest.mark.gpu


def _setup(seed, R=6, B=15):
    import dspark_draft_selection_gb300 as ds
    w = di.lattice_workload(seed, R=R, B=B, V_d=3000, V_t=7000, K=64, rank=64, pruned=True, with_seeds=True,
                            head_sigma=0.3)
    cd, ct, cv, st = ds.dspark_topk(dev(w["logits"]), B, 64, d2t=dev(w["d2t"]), V_t=7000)
    trans, gate, st2 = ds.dspark_lattice_score(ct, dev(w["prev"]), dev(w["E"]), dev(w["W"]))
    torch.cuda.synchronize()
    # histories: the tokens of each request's unpenalized greedy walk (so that the penalties bite),
    # some of its other candidates and random ids; one request has an empty history
    rng = np.random.default_rng(seed)
    cth, cvh, th = host(ct), host(cv), host(trans)
    cap = 40
    ids = np.full((R, cap), -1, dtype=np.int32)
    n = np.zeros(R, dtype=np.int32)
    for r in range(1, R):
        walk = cth[r][np.arange(B), od.chain_walk(cvh[r], th[r])[0]]
        pool = np.unique(np.concatenate([walk[:rng.integers(1, B + 1)], cth[r].ravel()[rng.integers(0, B * 64, size=8)],
                                         rng.integers(0, 7000, size=8)]))[:cap]
        n[r] = len(pool)
        ids[r, :n[r]] = rng.permutation(pool)
    return w, ct, cv, trans, ids, n


@pytest.mark.parametrize("rep,pres", [(1.3, 0.0), (1.0, 0.5), (2.0, 1.5), (0.8, -0.2)])
def test_greedy_walk_with_penalties(rep, pres):
    import dspark_draft_selection_gb300 as ds
    w, ct, cv, trans, ids, n = _setup(101)
    out = ds.dspark_chain_select(cv, trans, ct, "walk", history=(dev(ids), dev(n)), repetition=rep, presence=pres)
    torch.cuda.synchronize()
    assert ds.read_status(out[-1]) == 0
    chain, score = host(out[0]), host(out[2])
    cvh, th, cth = host(cv), host(trans), host(ct)
    changed = 0
    for r in range(w["R"]):
        och, osc = od.chain_walk(cvh[r], th[r], cth[r], history=set(ids[r, :n[r]].tolist()), repetition=rep,
                                 presence=pres)
        assert np.array_equal(och, chain[r]), r
        assert abs(osc - float(score[r])) <= 1e-5 * max(1.0, abs(osc))
        changed += not np.array_equal(och, od.chain_walk(cvh[r], th[r])[0])
    if rep >= 2.0:
        assert changed > 0                               # strong penalties change some walks


@pytest.mark.parametrize("T,top_p,min_p", [(0.8, 0.95, 0.0), (1.0, 1.0, 0.02)])
def test_sampled_walk_with_penalties_and_records(T, top_p, min_p):
    import dspark_draft_selection_gb300 as ds
    w, ct, cv, trans, ids, n = _setup(102)
    out = ds.dspark_chain_select(cv, trans, ct, "sample", temperature=T, top_p=top_p, min_p=min_p,
                                 seed=dev(w["seed"]), step=dev(w["step"]), history=(dev(ids), dev(n)),
                                 repetition=1.4, presence=0.3)
    torch.cuda.synchronize()
    assert ds.read_status(out[-1]) == 0
    chain, (qi, qp, qn) = host(out[0]), tuple(host(t) for t in out[3:6])
    cvh, th, cth = host(cv), host(trans), host(ct)
    for r in range(w["R"]):
        och, _, recs = od.chain_sample(cvh[r], th[r], cth[r], T, top_p, int(w["seed"][r]), int(w["step"][r]),
                                       min_p=min_p, history=set(ids[r, :n[r]].tolist()), repetition=1.4,
                                       presence=0.3)
        assert np.array_equal(och, chain[r]), r
        for j, rec in enumerate(recs):
            k = len(rec["kept"])
            assert qn[r, j] == k and np.array_equal(qi[r, j, :k], rec["ids"]) and np.array_equal(qp[r, j, :k], rec["q"])


def test_max_sum_refuses_penalties():
    import dspark_draft_selection_gb300 as ds
    w, ct, cv, trans, ids, n = _setup(103, R=2, B=3)
    with pytest.raises(ds.DsparkError):
        ds.dspark_chain_select(cv, trans, ct, "maxsum", history=(dev(ids), dev(n)), repetition=1.2)
