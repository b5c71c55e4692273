"""Pins for the oracle's rejection-sampling verification."""
import json
import os

import numpy as np
import pytest
from scipy import stats

from oracle import verify as ov
from oracle.fp32 import F32, F64
from oracle.philox import uniform
from oracle.sampling import draw_from_weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def chi2_ok(counts, probs, alpha=1e-3):
    exp = np.asarray(probs, dtype=np.float64) * counts.sum()
    keep = exp > 5
    stat = np.sum((counts[keep] - exp[keep]) ** 2 / exp[keep])
    return stat < stats.chi2.ppf(1 - alpha, keep.sum() - 1), stat


@pytest.mark.parametrize("V", [4, 8, 16])
def test_emitted_token_follows_p(V):
    rng = np.random.default_rng(100 + V)
    p = rng.dirichlet(np.ones(V) * 0.7)
    wq = rng.dirichlet(np.ones(V) * 0.7).astype(F32)
    n = 1_000_000
    steps = np.arange(n, dtype=np.uint64)
    x, wsum = draw_from_weights(wq, np.arange(V), uniform(1, steps, 0, 0))
    q = wq.astype(F64) / wsum
    acc, emitted = ov.verify_step(p, q, x, uniform(2, steps, 0, 1), uniform(2, steps, 0, 2))
    ok, stat = chi2_ok(np.bincount(emitted, minlength=V), p)
    assert ok, stat
    rate = np.minimum(p, q).sum()
    assert abs(acc.mean() - rate) < 5 * np.sqrt(rate * (1 - rate) / n)


def test_worked_example_exact_verification():
    g = json.load(open(os.path.join(GOLDEN, "worked_example_float_sums.json")))
    wq = np.concatenate([np.array(g["head_weights"], dtype=F32),
                         np.full(g["tail_count"], g["tail_weight"], dtype=F32)])
    V = wq.shape[0]
    p = np.zeros(V)
    p[:2] = g["target_p"]
    n = 1_000_000
    steps = np.arange(n, dtype=np.uint64)
    u = uniform(3, steps, 0, 0)
    x, wsum = draw_from_weights(wq, np.arange(V), u)
    q = wq.astype(F64) / wsum
    _, emitted = ov.verify_step(p, q, x, uniform(4, steps, 0, 1), uniform(4, steps, 0, 2))
    p1 = np.mean(emitted == 1)
    se = np.sqrt(0.25 / n)
    assert abs(p1 - g["p_token1_exact"]) < 5 * se
    # the float-sum proposal of the pages' example drifts to 0.505 and would fail this bound
    assert abs(g["p_token1_float_sums"] - g["p_token1_exact"]) > 9 * se
    c32 = np.cumsum(wq, dtype=F32)
    x32 = np.minimum(np.searchsorted(c32, (u * c32[-1]).astype(F32), side="right"), V - 1)
    _, em32 = ov.verify_step(p, q, x32, uniform(4, steps, 0, 1), uniform(4, steps, 0, 2))
    assert abs(np.mean(em32 == 1) - g["p_token1_float_sums"]) < 5 * se


def test_greedy_verification_is_argmax_matching():
    rng = np.random.default_rng(8)
    B, V = 6, 50
    for trial in range(50):
        rows = (rng.standard_normal((B + 1, V)) * 2).astype(F32)
        am = rows.argmax(axis=1)
        drafted = am[:B].copy()
        k = int(rng.integers(0, B + 1))
        if k < B:
            drafted[k] = (drafted[k] + 1) % V
        res = ov.verify_request(rows, drafted, B, None, 0.0, 1.0, 0, 0)
        assert res["n_accepted"] == k
        assert list(res["tokens"]) == list(am[:k]) + [int(am[k])]


def test_identical_q_and_p_accept_all_and_draw_a_bonus():
    rng = np.random.default_rng(9)
    B, V = 4, 30
    rows = (rng.standard_normal((B + 1, V)) * 2).astype(F32)
    dists = [ov.TargetDist(rows[j], 0.8, 1.0) for j in range(B + 1)]
    drafted = [int(np.argmax(d.p())) for d in dists[:B]]
    res = ov.verify_request(rows, drafted, B, lambda j: dists[j].p(), 0.8, 1.0, 77, 5)
    assert res["n_accepted"] == B and len(res["tokens"]) == B + 1
    u = float(uniform(77, 5, B, 2))
    assert res["tokens"][B] == int(draw_from_weights(dists[B].w, dists[B].kept, u)[0])


def test_zero_proposal_and_out_of_width_ids():
    rows = np.zeros((3, 10), dtype=F32)
    q = np.full(10, 0.1)
    q0 = q.copy()
    q0[4] = 0.0
    assert ov.verify_request(rows, [4, 1], 2, lambda j: q0, 1.0, 1.0, 0, 0)["status"] == ov.EPROPOSAL
    # a drafted id beyond the target's row has zero target probability: always rejected
    qw = np.full(12, 1.0 / 12)
    for s in range(20):
        res = ov.verify_request(rows, [11, 1], 2, lambda j: qw, 1.0, 1.0, s, 0)
        assert res["n_accepted"] == 0 and res["tokens"][0] < 10


def test_min_p_one_makes_verification_argmax_matching():
    """With min_p = 1 the target's post-filter p is a point mass on its argmax: a drafted token
    (with q > 0) is accepted exactly when it is the argmax, and a rejection emits the argmax."""
    from oracle import verify as ov
    rng = np.random.default_rng(5)
    V, B = 50, 6
    rows = rng.standard_normal((B + 1, V)).astype(np.float32) * 2
    amax = rows.argmax(axis=1)
    drafted = np.where(rng.random(B) < 0.5, amax[:B], (amax[:B] + 1) % V)
    q = np.full(V, 1.0 / V)
    res = ov.verify_request(rows, drafted, B, lambda j: q, 0.9, 1.0, 77, 3, min_p=1.0)
    first_bad = next((j for j in range(B) if drafted[j] != amax[j]), B)
    assert res["n_accepted"] == first_bad
    assert list(res["tokens"]) == list(amax[:first_bad + 1]) if first_bad < B else list(res["tokens"][:B]) == list(amax[:B])
