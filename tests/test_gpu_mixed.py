"""Mixed greedy/sampled batches: per-request temperature and top-p in one call of
dspark_chain_select, dspark_sample and dspark_verify, each request checked against the oracle run
with that request's own values (the same per-request definition; the batch only groups them).
Also sparse-q verification at the pruned draft's full size."""
import numpy as np
import pytest
import torch

import dspark_inputs as di
from oracle import draft as od
from tests.gpu_util import as_f32, dev, host
from tests.test_gpu_sample import check_rows, seeds
from tests.test_gpu_verify import oracle_check

pytestmark = pytest.mark.gpu

T_R = np.array([0.0, 0.8, 0.3, 1.0, 0.0, 1.2], dtype=np.float32)
P_R = np.array([1.0, 0.95, 0.5, 1.0, 0.7, 0.9], dtype=np.float32)


def _draft_mixed(w, T_r, P_r):
    import dspark_draft_selection_gb300 as ds
    cd, ct, cv, st = ds.dspark_topk(dev(w["logits"]), w["B"], 64, d2t=dev(w["d2t"]), V_t=w["V_t"])
    trans, gate, st2 = ds.dspark_lattice_score(ct, dev(w["prev"]), dev(w["E"]), dev(w["W"]))
    out = ds.dspark_chain_select(cv, trans, ct, "sample", seed=dev(w["seed"]), step=dev(w["step"]),
                                 temperature_r=dev(T_r), top_p_r=dev(P_r))
    torch.cuda.synchronize()
    for s in (st, st2, out[-1]):
        assert ds.read_status(s) == 0
    return host(cv), host(trans), host(ct), host(out[0]), host(out[1]), tuple(host(t) for t in out[3:6]), out


def test_chain_select_mixed_batch():
    w = di.lattice_workload(91, R=6, B=15, V_d=3000, V_t=7000, K=64, rank=64, pruned=True, with_seeds=True,
                            head_sigma=0.3)
    cv, trans, ct, chain, chain_tgt, (ids, qp, qn), _ = _draft_mixed(w, T_R, P_R)
    for r in range(w["R"]):
        och, score, recs = od.chain_sample(cv[r], trans[r], ct[r], float(T_R[r]), float(P_R[r]), int(w["seed"][r]),
                                           int(w["step"][r]))
        assert np.array_equal(och, chain[r]), r
        for j, rec in enumerate(recs):
            n = len(rec["kept"])
            assert qn[r, j] == n and np.array_equal(ids[r, j, :n], rec["ids"]) and np.array_equal(qp[r, j, :n], rec["q"])
        if T_R[r] <= 0:
            assert np.all(qn[r] == 1) and np.all(qp[r, :, 0] == 1.0)
            assert np.array_equal(chain[r], od.chain_walk(cv[r], trans[r])[0])


def test_sample_mixed_batch_per_request_values():
    import dspark_draft_selection_gb300 as ds
    R, B, V = 6, 4, 20011
    w = di.lattice_workload(92, R=R, B=B, V_d=V, K=1, rank=8)
    seed, step = seeds(R, 92)
    q = ds.dense_record(R * B, V)
    tgt, idx, st = ds.dspark_sample(dev(w["logits"]), B, seed=dev(seed), step=dev(step), q=q,
                                    temperature_r=dev(T_R), top_p_r=dev(P_R))
    torch.cuda.synchronize()
    assert ds.read_status(st) == 0
    rec = tuple(host(t) for t in q)
    s = as_f32(w["logits"])
    got = host(idx)
    for r in range(R):
        sl = slice(r * B, (r + 1) * B)
        sub = tuple(x[sl] for x in rec)
        check_rows(s[sl], B, float(T_R[r]), float(P_R[r]), seed[r:r + 1], step[r:r + 1], got[r:r + 1],
                   rec=sub, record="dense")


@pytest.mark.parametrize("with_top_p", [False, True])
def test_verify_mixed_batch(with_top_p):
    """Greedy and sampled requests verified in one call: the statistics kernel path (per-request
    temperature) and the nucleus path (per-request top-p)."""
    import dspark_draft_selection_gb300 as ds
    w = di.lattice_workload(93, R=6, B=7, V_d=3000, V_t=7000, K=64, rank=64, pruned=True, with_seeds=True,
                            head_sigma=0.3)
    R, B = w["R"], w["B"]
    P_r = P_R if with_top_p else np.ones(R, dtype=np.float32)
    cv, trans, ct, chain, drafted, (ids_h, qp_h, qn_h), out = _draft_mixed(w, T_R, P_r)
    target = di.normal(di.generator(93, 20), (R * (B + 1), 7000), 2.0, "bf16")
    tf = as_f32(target).copy()
    for r in (1, 3, 5):                                  # sampled requests: targets near their proposals
        for j in range(B):
            k = qn_h[r, j]
            tf[r * (B + 1) + j] = -40.0
            tf[r * (B + 1) + j, ids_h[r, j, :k]] = T_R[r] * np.log(qp_h[r, j, :k].astype(np.float64))
    for j in range(B):                                   # greedy request 4: its tokens are the argmax
        tf[4 * (B + 1) + j, drafted[4, j]] = 30.0
    target = di.f32_to_bf16_bits(tf)
    vseed = np.arange(R, dtype=np.uint64) * 104729 + 11
    n = np.array([B, B, 5, B, B, 3], dtype=np.int32)
    toks, nacc, lp, st = ds.dspark_verify(dev(target), B, dev(drafted.astype(np.int32)), dev(n), out[3:6],
                                          vseed=dev(vseed), step=dev(w["step"]), temperature_r=dev(T_R),
                                          top_p_r=dev(P_r) if with_top_p else None)
    torch.cuda.synchronize()
    assert ds.read_status(st) == 0
    toks, nacc, lp = host(toks), host(nacc), host(lp)
    for r in range(R):
        def qfun(rr, j):
            full = np.zeros(7000)
            k = qn_h[r, j]
            full[ids_h[r, j, :k]] = qp_h[r, j, :k].astype(np.float64)
            return full
        sl = slice(r * (B + 1), (r + 1) * (B + 1))
        assert oracle_check(target[sl], B, drafted[r:r + 1], n[r:r + 1], qfun, float(T_R[r]), float(P_r[r]),
                            vseed[r:r + 1], w["step"][r:r + 1], toks[r:r + 1], nacc[r:r + 1], lp[r:r + 1]) == 0, r
    assert nacc[4] == B                                  # the greedy request's tokens are all accepted


def test_sparse_q_verify_pruned_config_full_size():
    """The pruned DSpark draft at full size (16 requests x block 15, 248,100 target ids): sampled
    chains with their sparse records, verified against target rows planted near the proposals for
    half of the requests."""
    import dspark_draft_selection_gb300 as ds
    w = di.config3()
    R, B, V_t = w["R"], w["B"], w["V_t"]
    cd, ct, cv, st = ds.dspark_topk(dev(w["logits"]), B, w["K"], d2t=dev(w["d2t"]), V_t=V_t)
    trans, gate, st2 = ds.dspark_lattice_score(ct, dev(w["prev"]), dev(w["E"]), dev(w["W"]))
    out = ds.dspark_chain_select(cv, trans, ct, "sample", temperature=w["temperature"], top_p=w["top_p"],
                                 seed=dev(w["seed"]), step=dev(w["step"]))
    drafted = host(out[1])
    ids_h, qp_h, qn_h = (host(t) for t in out[3:6])
    tf = as_f32(di.normal(di.generator(3, 40), (R * (B + 1), V_t), 2.0, "bf16")).copy()
    T = w["temperature"]
    for r in range(0, R, 2):
        for j in range(B):
            k = qn_h[r, j]
            tf[r * (B + 1) + j] = -40.0
            tf[r * (B + 1) + j, ids_h[r, j, :k]] = T * np.log(qp_h[r, j, :k].astype(np.float64))
    target = di.f32_to_bf16_bits(tf)
    vseed = np.arange(R, dtype=np.uint64) * 15485863 + 7
    n = np.full(R, B, dtype=np.int32)
    toks, nacc, lp, st3 = ds.dspark_verify(dev(target), B, out[1], dev(n), out[3:6], temperature=T,
                                           top_p=w["top_p"], vseed=dev(vseed), step=dev(w["step"]))
    torch.cuda.synchronize()
    assert ds.read_status(st3) == 0
    toks, nacc, lp = host(toks), host(nacc), host(lp)

    def qfun(r, j):
        full = np.zeros(V_t)
        k = qn_h[r, j]
        full[ids_h[r, j, :k]] = qp_h[r, j, :k].astype(np.float64)
        return full

    assert oracle_check(target, B, drafted, n, qfun, T, w["top_p"], vseed, w["step"], toks, nacc, lp) == 0
    assert nacc[0::2].mean() > 2
