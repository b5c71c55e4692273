"""min-p in sampled drafting and in verification (after top-p: tokens whose probability is at
least min_p times the top token's), GPU against the oracle."""
import numpy as np
import pytest
import torch

import dspark_inputs as di
from oracle import draft as od
from tests.gpu_util import as_f32, dev, host
from tests.test_gpu_sample import check_rows, seeds
from tests.test_gpu_verify import oracle_check

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("V,T,top_p,min_p", [(20011, 1.0, 1.0, 0.05), (30011, 0.8, 0.95, 0.01), (5000, 1.3, 0.9, 0.3),
                                             (248320, 0.8, 1.0, 0.002), (37, 1.0, 1.0, 1.0)])
@pytest.mark.parametrize("record", ["dense", "sparse"])
def test_sample_min_p_matches_the_oracle(V, T, top_p, min_p, record):
    import dspark_draft_selection_gb300 as ds
    R, B = 3, 4
    w = di.lattice_workload(71 + V % 89, R=R, B=B, V_d=V, K=1, rank=8)
    seed, step = seeds(R, 71)
    rows = R * B
    if record == "dense":
        q = ds.dense_record(rows, V)
    else:
        q = (torch.full((rows, min(V, 8192)), -1, dtype=torch.int32, device="cuda"),
             torch.zeros((rows, min(V, 8192)), dtype=torch.float32, device="cuda"),
             torch.zeros((rows,), dtype=torch.int32, device="cuda"))
    tgt, idx, st = ds.dspark_sample(dev(w["logits"]), B, temperature=T, top_p=top_p, min_p=min_p, seed=dev(seed),
                                    step=dev(step), q=q)
    torch.cuda.synchronize()
    assert ds.read_status(st) == 0
    rec = tuple(host(t) for t in q)
    assert check_rows(as_f32(w["logits"]), B, T, top_p, seed, step, host(idx), rec=rec, record=record,
                      min_p=min_p) <= 1


def test_chain_sample_min_p_and_per_request_values():
    import dspark_draft_selection_gb300 as ds
    w = di.lattice_workload(94, R=5, B=15, V_d=3000, V_t=7000, K=64, rank=64, pruned=True, with_seeds=True,
                            head_sigma=0.3)
    cd, ct, cv, st = ds.dspark_topk(dev(w["logits"]), w["B"], 64, d2t=dev(w["d2t"]), V_t=7000)
    trans, gate, st2 = ds.dspark_lattice_score(ct, dev(w["prev"]), dev(w["E"]), dev(w["W"]))
    mp_r = np.array([0.0, 0.05, 0.3, 1.0, 0.01], dtype=np.float32)
    T_r = np.array([0.8, 1.0, 0.7, 0.9, 1.2], dtype=np.float32)
    P_r = np.array([0.95, 1.0, 0.9, 1.0, 0.8], dtype=np.float32)
    out = ds.dspark_chain_select(cv, trans, ct, "sample", seed=dev(w["seed"]), step=dev(w["step"]),
                                 temperature_r=dev(T_r), top_p_r=dev(P_r), min_p_r=dev(mp_r))
    torch.cuda.synchronize()
    assert ds.read_status(out[-1]) == 0
    chain, (ids, qp, qn) = host(out[0]), tuple(host(t) for t in out[3:6])
    cvh, th, cth = host(cv), host(trans), host(ct)
    for r in range(5):
        och, _, recs = od.chain_sample(cvh[r], th[r], cth[r], float(T_r[r]), float(P_r[r]), int(w["seed"][r]),
                                       int(w["step"][r]), min_p=float(mp_r[r]))
        assert np.array_equal(och, chain[r]), r
        for j, rec in enumerate(recs):
            n = len(rec["kept"])
            assert qn[r, j] == n and np.array_equal(ids[r, j, :n], rec["ids"]) and np.array_equal(qp[r, j, :n], rec["q"])


@pytest.mark.parametrize("top_p", [1.0, 0.9])
def test_verify_min_p_matches_the_oracle(top_p):
    """Drafted with min-p, verified with the same min-p (statistics path with top_p = 1, nucleus
    path with top_p < 1)."""
    import dspark_draft_selection_gb300 as ds
    w = di.lattice_workload(95, R=6, B=7, V_d=3000, V_t=7000, K=64, rank=64, pruned=True, with_seeds=True,
                            head_sigma=0.3)
    R, B, T, mp = w["R"], w["B"], 0.9, 0.02
    cd, ct, cv, st = ds.dspark_topk(dev(w["logits"]), B, 64, d2t=dev(w["d2t"]), V_t=7000)
    trans, gate, st2 = ds.dspark_lattice_score(ct, dev(w["prev"]), dev(w["E"]), dev(w["W"]))
    out = ds.dspark_chain_select(cv, trans, ct, "sample", temperature=T, top_p=top_p, min_p=mp, seed=dev(w["seed"]),
                                 step=dev(w["step"]))
    torch.cuda.synchronize()
    drafted = host(out[1])
    ids_h, qp_h, qn_h = (host(t) for t in out[3:6])
    tf = as_f32(di.normal(di.generator(95, 20), (R * (B + 1), 7000), 2.0, "bf16")).copy()
    for r in range(1, R, 2):
        for j in range(B):
            k = qn_h[r, j]
            tf[r * (B + 1) + j] = -40.0
            tf[r * (B + 1) + j, ids_h[r, j, :k]] = T * np.log(qp_h[r, j, :k].astype(np.float64))
    target = di.f32_to_bf16_bits(tf)
    vseed = np.arange(R, dtype=np.uint64) * 7907 + 5
    n = np.full(R, B, dtype=np.int32)
    toks, nacc, lp, st3 = ds.dspark_verify(dev(target), B, out[1], dev(n), out[3:6], temperature=T, top_p=top_p,
                                           min_p=mp, vseed=dev(vseed), step=dev(w["step"]))
    torch.cuda.synchronize()
    assert ds.read_status(st3) == 0

    def qfun(r, j):
        full = np.zeros(7000)
        k = qn_h[r, j]
        full[ids_h[r, j, :k]] = qp_h[r, j, :k].astype(np.float64)
        return full

    assert oracle_check(target, B, drafted, n, qfun, T, top_p, vseed, w["step"], host(toks), host(nacc), host(lp),
                        min_p=mp) == 0
