"""GPU parity of dspark_verify against the oracle's rejection-sampling verification.

Both sides verify the same drafted tokens against the same proposal record (the record the GPU
drafting kernels wrote). The target weights are the same float32 function on both sides, so
acceptance decisions and residual draws must agree; a difference is admissible only where the
oracle's margin (|u - p/q|, or the distance of the draw target to a running-sum boundary) is at
double rounding level.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import dspark_inputs as di
from oracle import verify as ov
from oracle.philox import uniform
from oracle.sampling import dense_q
from tests.gpu_util import as_f32, dev, host

pytestmark = pytest.mark.gpu


def gpu_verify(target, B, drafted, n, q, T, top_p, vseed, step, V_q=None):
    import dspark_draft_selection_gb300 as ds
    toks, nacc, lp, st = ds.dspark_verify(dev(target), B, dev(drafted.astype(np.int32)), dev(n.astype(np.int32)), q,
                                          V_q=V_q, temperature=T, top_p=top_p, vseed=dev(vseed), step=dev(step))
    torch.cuda.synchronize()
    return host(toks), host(nacc), host(lp), ds.read_status(st)


def oracle_check(target, B, drafted, n, qfun, T, top_p, vseed, step, toks, nacc, lp, min_p=0.0):
    t = as_f32(target)
    R = drafted.shape[0]
    amb = 0
    for r in range(R):
        rows = t[r * (B + 1):(r + 1) * (B + 1)]
        res = ov.verify_request(rows, drafted[r], int(n[r]), lambda j: qfun(r, j), T, top_p, int(vseed[r]),
                                int(step[r]), min_p=min_p)
        if res["n_accepted"] != nacc[r] or list(res["tokens"]) != list(toks[r, :len(res["tokens"])]):
            m = min(res["margins"]) if res["margins"] else 1.0
            assert m < 1e-12, (r, res["n_accepted"], nacc[r], res["tokens"], toks[r])
            amb += 1
            continue
        k = len(res["tokens"])
        assert np.all(toks[r, k:] == -1)
        np.testing.assert_allclose(lp[r, :k], res["logprobs"], rtol=1e-4, atol=1e-4)
    return amb


def test_verify_after_gpu_dense_walk_dense_record():
    import dspark_draft_selection_gb300 as ds
    w = di.config5(R=6, V=30000)
    R, B, V = w["R"], w["B"], w["V_d"]
    q = ds.dense_record(R * B, V)
    tgt, idx, st = ds.dspark_dense_walk(dev(w["logits"]), B, dev(w["prev"]), dev(w["E"]), dev(w["W"]),
                                        temperature=1.0, top_p=1.0, seed=dev(w["seed"]), step=dev(w["step"]), q=q)
    torch.cuda.synchronize()
    drafted = host(tgt)
    rec = tuple(host(x) for x in q)
    n = np.array([B, B, 3, 0, 7, B], dtype=np.int32)
    toks, nacc, lp, st = gpu_verify(w["target"], B, drafted, n, q, 1.0, 1.0, w["vseed"], w["step"])
    assert st == 0
    z, zmax, wsum, wcut, icut = rec

    def qfun(r, j):
        i = r * B + j
        return dense_q(z[i], zmax[i], wsum[i], wcut[i], icut[i], np.arange(V))

    assert oracle_check(w["target"], B, drafted, n, qfun, 1.0, 1.0, w["vseed"], w["step"], toks, nacc, lp) == 0
    assert np.all(nacc <= n) and np.all(nacc >= 0)


@pytest.mark.parametrize("T,top_p", [(0.8, 0.95), (1.0, 1.0)])
def test_verify_sparse_record_pruned_draft(T, top_p):
    import dspark_draft_selection_gb300 as ds
    w = di.lattice_workload(80, R=6, B=7, V_d=3000, V_t=7000, K=64, rank=64, pruned=True, with_seeds=True,
                            head_sigma=0.3)
    R, B = w["R"], w["B"]
    cd, ct, cv, st = ds.dspark_topk(dev(w["logits"]), B, 64, d2t=dev(w["d2t"]), V_t=7000)
    trans, gate, st2 = ds.dspark_lattice_score(ct, dev(w["prev"]), dev(w["E"]), dev(w["W"]))
    rank_, chain_tgt, score, ids, qp, qn, st3 = ds.dspark_chain_select(cv, trans, ct, "sample", temperature=T,
                                                                      top_p=top_p, seed=dev(w["seed"]),
                                                                      step=dev(w["step"]))
    torch.cuda.synchronize()
    drafted = host(chain_tgt)
    ids_h, qp_h, qn_h = host(ids), host(qp), host(qn)
    target = di.normal(di.generator(80, 20), (R * (B + 1), 7000), 2.0, "bf16")
    # requests 1.. get targets close to their proposals (p ~ q: mostly accepted); request 0 keeps a
    # random target (mostly rejected)
    tf = as_f32(target).copy()
    for r in range(1, R):
        for j in range(B):
            k = qn_h[r, j]
            tf[r * (B + 1) + j] = -40.0
            tf[r * (B + 1) + j, ids_h[r, j, :k]] = T * np.log(qp_h[r, j, :k].astype(np.float64))
    target = di.f32_to_bf16_bits(tf)
    vseed = np.arange(R, dtype=np.uint64) * 7919 + 3
    n = np.full(R, B, dtype=np.int32)
    toks, nacc, lp, st = gpu_verify(target, B, drafted, n, (ids, qp, qn), T, top_p, vseed, w["step"])
    assert st == 0

    def qfun(r, j):
        full = np.zeros(7000)
        k = qn_h[r, j]
        full[ids_h[r, j, :k]] = qp_h[r, j, :k].astype(np.float64)
        return full

    assert oracle_check(target, B, drafted, n, qfun, T, top_p, vseed, w["step"], toks, nacc, lp) == 0
    assert nacc[1:].mean() > 2


def test_verify_greedy_is_argmax_matching():
    R, B, V = 5, 6, 5000
    target = di.normal(di.generator(81, 1), (R * (B + 1), V), 2.0, "bf16")
    t = as_f32(target)
    am = t.argmax(axis=1).reshape(R, B + 1)
    drafted = am[:, :B].copy()
    drafted[1, 2] = (drafted[1, 2] + 1) % V
    drafted[3, 0] = (drafted[3, 0] + 5) % V
    n = np.full(R, B, dtype=np.int32)
    seed = np.zeros(R, dtype=np.uint64)
    toks, nacc, lp, st = gpu_verify(target, B, drafted, n, None, 0.0, 1.0, seed, seed)
    assert st == 0
    assert list(nacc) == [B, 2, B, 0, B]
    for r in range(R):
        k = nacc[r]
        assert list(toks[r, :k + 1]) == list(am[r, :k + 1])
    assert oracle_check(target, B, drafted, n, None, 0.0, 1.0, seed, seed, toks, nacc, lp) == 0


def test_verify_emitted_token_follows_p_chi_square():
    import dspark_draft_selection_gb300 as ds
    V, R, B = 12, 20000, 1
    rng = np.random.default_rng(12)
    prow = (rng.standard_normal(V) * 1.2).astype(np.float32)
    qrow = (rng.standard_normal(V) * 1.2).astype(np.float32)
    target = np.tile(np.stack([prow, prow]), (R, 1))              # row 0 verifies, row 1 is the bonus row
    drafts = np.tile(qrow, (R, 1))
    seed = np.full(R, 5, dtype=np.uint64)
    step = np.arange(R, dtype=np.uint64)
    q = ds.dense_record(R, V)
    tgt, idx, st = ds.dspark_sample(dev(drafts), 1, temperature=1.0, seed=dev(seed), step=dev(step), q=q)
    vseed = np.full(R, 11, dtype=np.uint64)
    toks, nacc, lp, st = gpu_verify(target, B, host(tgt), np.ones(R, dtype=np.int32), q, 1.0, 1.0, vseed, step)
    assert st == 0
    # the first emitted token (accepted draft or residual correction) follows p
    first = toks[:, 0]
    p = np.exp(prow.astype(np.float64) - prow.max())
    p /= p.sum()
    counts = np.bincount(first, minlength=V)
    exp = p * R
    stat = np.sum((counts - exp) ** 2 / exp)
    assert stat < stats.chi2.ppf(0.999, V - 1)
    qq = np.exp(qrow.astype(np.float64) - qrow.max())
    qq /= qq.sum()
    rate = np.minimum(p, qq).sum()
    assert abs(nacc.mean() - rate) < 5 * np.sqrt(rate * (1 - rate) / R)


def test_verify_zero_proposal_reports_status():
    import dspark_draft_selection_gb300 as ds
    R, B, V = 2, 2, 100
    target = np.zeros((R * (B + 1), V), dtype=np.float32)
    target[0, 5] = 30.0                                           # position 0 of request 0 is accepted
    ids = torch.tensor([[[5, 6], [7, 8]], [[1, 2], [3, 4]]], dtype=torch.int32, device="cuda")
    qp = torch.full((R, B, 2), 0.5, dtype=torch.float32, device="cuda")
    qn = torch.full((R, B), 2, dtype=torch.int32, device="cuda")
    drafted = np.array([[5, 9], [1, 3]], dtype=np.int32)        # 9 is not in its position's record
    seed = np.arange(R, dtype=np.uint64)
    toks, nacc, lp, st = gpu_verify(target, B, drafted, np.full(R, B, dtype=np.int32), (ids, qp, qn), 1.0, 1.0,
                                    seed, seed)
    assert st == 4
    assert nacc[0] == -1 and np.all(toks[0] == -1)


def _walk_and_record(w, T=1.0, top_p=1.0, d2t=None):
    import dspark_draft_selection_gb300 as ds
    R, B, V = w["R"], w["B"], w["V_d"]
    q = ds.dense_record(R * B, V)
    kw = {"d2t": dev(d2t)} if d2t is not None else {}
    tgt, idx, st = ds.dspark_dense_walk(dev(w["logits"]), B, dev(w["prev"]), dev(w["E"]), dev(w["W"]),
                                        temperature=T, top_p=top_p, seed=dev(w["seed"]), step=dev(w["step"]), q=q,
                                        **kw)
    torch.cuda.synchronize()
    assert ds.read_status(st) == 0
    return host(tgt), q, tuple(host(x) for x in q)


def _dense_qfun(rec, B, V, m=None, V_t=None):
    z, zmax, wsum, wcut, icut = rec

    def qfun(r, j):
        i = r * B + j
        qd = dense_q(z[i], zmax[i], wsum[i], wcut[i], icut[i], np.arange(V))
        if m is None:
            return qd
        full = np.zeros(V_t)
        full[m] = qd
        return full
    return qfun


def test_verify_full_size_dense_walk_config():
    # the benchmarked shape: 64 requests x 15 drafted tokens, 1,024 target rows of 151,936 logits,
    # a dense record of the same width (149 cells of 1,024 ids per draw row); split windows
    w = di.config5()
    R, B, V = w["R"], w["B"], w["V_d"]
    drafted, q, rec = _walk_and_record(w, w["temperature"], w["top_p"])
    rng = np.random.default_rng(55)
    n = rng.integers(0, B + 1, size=R).astype(np.int32)
    n[:4] = B
    toks, nacc, lp, st = gpu_verify(w["target"], B, drafted, n, q, 1.0, 1.0, w["vseed"], w["step"])
    assert st == 0
    assert np.all((nacc >= 0) & (nacc <= n))
    for r in range(R):
        k = nacc[r]
        assert np.all(toks[r, :k] == drafted[r, :k]) and 0 <= toks[r, k] < V and np.all(toks[r, k + 1:] == -1)
    reqs = [0, 1, 2, 3, 17, 40, 63] + [int(r) for r in np.nonzero(n < B)[0][:3]]
    sub = np.array(sorted(set(reqs)))
    qfun = _dense_qfun(rec, B, V)
    t = w["target"].reshape(R, B + 1, V)
    assert oracle_check(t[sub].reshape(-1, V), B, drafted[sub], n[sub],
                        lambda rr, j: qfun(int(sub[rr]), j), 1.0, 1.0, w["vseed"][sub], w["step"][sub],
                        toks[sub], nacc[sub], lp[sub]) == 0
    assert (nacc[n == B] < B).any() and (nacc == n).any()     # both residual and bonus draws ran


def test_verify_full_size_greedy():
    w = di.config5()
    R, B, V = w["R"], w["B"], w["V_d"]
    t = as_f32(w["target"])
    am = t.argmax(axis=1).reshape(R, B + 1)
    rng = np.random.default_rng(56)
    drafted = am[:, :B].copy()
    bad = rng.random((R, B)) < 0.15
    drafted[bad] = (drafted[bad] + 1 + rng.integers(0, V - 1, size=bad.sum())) % V
    n = np.full(R, B, dtype=np.int32)
    seed = np.zeros(R, dtype=np.uint64)
    toks, nacc, lp, st = gpu_verify(w["target"], B, drafted, n, None, 0.0, 1.0, seed, seed)
    assert st == 0
    for r in range(R):
        k = int(np.argmax(bad[r])) if bad[r].any() else B
        assert nacc[r] == k
        assert list(toks[r, :k + 1]) == list(am[r, :k + 1])
    sub = np.arange(0, R, 9)
    assert oracle_check(w["target"].reshape(R, B + 1, V)[sub].reshape(-1, V), B, drafted[sub], n[sub], None, 0.0,
                        1.0, seed[sub], seed[sub], toks[sub], nacc[sub], lp[sub]) == 0


def test_verify_sparse_record_larger_than_a_thousand_entries():
    # a full-row sampled draft at high temperature keeps thousands of tokens in its nucleus: the
    # residual draw must use every entry of the sparse record
    import dspark_draft_selection_gb300 as ds
    R, B, V = 6, 3, 6000
    drafts = di.normal(di.generator(83, 1), (R * B, V), 0.5, "bf16")
    seed = np.arange(R, dtype=np.uint64) + 11
    step = np.arange(R, dtype=np.uint64) * 3
    cap = V
    ids = torch.full((R, B, cap), -1, dtype=torch.int32, device="cuda")
    qp = torch.zeros((R, B, cap), dtype=torch.float32, device="cuda")
    qn = torch.zeros((R, B), dtype=torch.int32, device="cuda")
    tgt, idx, st = ds.dspark_sample(dev(drafts), B, temperature=1.5, top_p=0.99, seed=dev(seed), step=dev(step),
                                    q=(ids, qp, qn))
    torch.cuda.synchronize()
    assert ds.read_status(st) == 0
    qn_h, ids_h, qp_h = host(qn), host(ids), host(qp)
    assert qn_h.min() > 1024
    target = di.normal(di.generator(83, 2), (R * (B + 1), V), 0.5, "bf16")
    vseed = np.arange(R, dtype=np.uint64) * 101 + 7
    n = np.full(R, B, dtype=np.int32)
    toks, nacc, lp, st = gpu_verify(target, B, host(tgt), n, (ids, qp, qn), 1.0, 1.0, vseed, step)
    assert st == 0

    def qfun(r, j):
        full = np.zeros(V)
        k = qn_h[r, j]
        full[ids_h[r, j, :k]] = qp_h[r, j, :k].astype(np.float64)
        return full

    assert oracle_check(target, B, host(tgt), n, qfun, 1.0, 1.0, vseed, step, toks, nacc, lp) == 0
    assert (nacc < n).any()


@pytest.mark.parametrize("T,top_p", [(1.0, 1.0), (0.8, 0.9)])
def test_verify_dense_record_over_a_pruned_draft(T, top_p):
    # [P]: the dense walk on a pruned draft records q over draft indices; verification reads it in
    # target ids through d2t
    import dspark_draft_selection_gb300 as ds
    w = di.lattice_workload(84, R=5, B=4, V_d=6000, V_t=15000, K=0, rank=64, pruned=True, with_seeds=True,
                            head_sigma=0.3)
    R, B, V_d, V_t = w["R"], w["B"], w["V_d"], w["V_t"]
    drafted, q, rec = _walk_and_record(w, T, top_p, d2t=w["d2t"])
    m = w["subset"]
    assert np.all(np.isin(drafted, m))
    # targets close to the draft rows on the subset (mostly accepted), noise elsewhere
    tf = as_f32(di.normal(di.generator(84, 30), (R * (B + 1), V_t), 2.0, "bf16")).copy()
    s = as_f32(w["logits"])
    for r in range(R):
        for j in range(B):
            tf[r * (B + 1) + j, m] = 0.9 * s[r * B + j] + 0.1 * tf[r * (B + 1) + j, m]
    target = di.f32_to_bf16_bits(tf)
    vseed = np.arange(R, dtype=np.uint64) * 13 + 1
    n = np.array([B, B, 2, 0, B], dtype=np.int32)
    toks, nacc, lp, st = ds.dspark_verify(dev(target), B, dev(drafted.astype(np.int32)), dev(n), q, q_d2t=dev(w["d2t"]),
                                          temperature=T, top_p=top_p, vseed=dev(vseed), step=dev(w["step"]))
    torch.cuda.synchronize()
    assert ds.read_status(st) == 0
    toks, nacc, lp = host(toks), host(nacc), host(lp)
    qfun = _dense_qfun(rec, B, V_d, m=m, V_t=V_t)
    assert oracle_check(target, B, drafted, n, qfun, T, top_p, vseed, w["step"], toks, nacc, lp) == 0
    assert nacc[:2].sum() > 0


def test_verify_n_draft_out_of_range_is_an_error_not_a_fault():
    import dspark_draft_selection_gb300 as ds
    R, B, V = 3, 4, 3000
    target = di.normal(di.generator(85, 1), (R * (B + 1), V), 2.0, "bf16")
    drafted = np.tile(np.arange(B, dtype=np.int32), (R, 1))
    n = np.array([B + 1, -1, 2], dtype=np.int32)
    seed = np.arange(R, dtype=np.uint64)
    for T in (0.0, 1.0):
        q = None
        if T > 0:
            ids = torch.tensor(np.tile(np.arange(B, dtype=np.int32)[None, :, None], (R, 1, 1)), device="cuda")
            q = (ids, torch.ones((R, B, 1), dtype=torch.float32, device="cuda"),
                 torch.ones((R, B), dtype=torch.int32, device="cuda"))
        toks, nacc, lp, st = gpu_verify(target, B, drafted, n, q, T, 1.0, seed, seed)
        assert st == 1                                             # DSPARK_EINVAL
        assert nacc[0] == -1 and nacc[1] == -1 and np.all(toks[:2] == -1)
        assert 0 <= nacc[2] <= 2 and toks[2, nacc[2]] >= 0
