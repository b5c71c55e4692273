"""Pins for the oracle's Top-K, d2t, head, lattice and chain selection."""
import json
import math
import os

import numpy as np

import dspark_inputs as di
from oracle import draft as od
from oracle import walk as ow
from oracle.fp32 import F32, F64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_topk_is_full_sort_with_ties_and_signed_zero():
    rng = np.random.default_rng(11)
    for trial in range(300):
        V = int(rng.integers(1, 400))
        s = np.round(rng.standard_normal(V) * 3).astype(F32)     # heavy ties
        s[rng.random(V) < 0.1] = F32(-0.0)
        s[rng.random(V) < 0.1] = F32(0.0)
        K = int(rng.integers(1, 70))
        idx, val = od.topk_row(s, K)
        want = sorted(range(V), key=lambda i: (-float(s[i]), i))[:min(K, V)]
        assert list(idx) == want
        assert np.array_equal(val, s[want])


def test_dominant_planted_peak_is_rank_zero():
    w = di.lattice_workload(90, R=2, B=3, V_d=5000, K=64, rank=8)
    s = di.bf16_bits_to_f32(w["logits"]).copy()
    rng = np.random.default_rng(4)
    for r in range(6):
        i = int(rng.integers(0, 5000))
        s[r, i] = s[r].max() + F32(8.0)
        idx, val = od.topk_row(s[r], 64)
        assert idx[0] == i and val[0] == s[r, i]
        assert val[1] <= val[0] - 8


def test_k_rule_from_the_pages():
    g = json.load(open(os.path.join(GOLDEN, "pruned_vocabulary.json")))
    for case in g["cases"]:
        assert od.top_k_count(64, case["draft_vocab"]) == case["k"]
        s = np.arange(min(case["draft_vocab"], 1000), dtype=F32)
        if case["draft_vocab"] <= 1000:
            assert od.topk_row(s, 64)[0].shape[0] == case["k"]


def test_d2t_round_trip_and_checks():
    g = json.load(open(os.path.join(GOLDEN, "pruned_vocabulary.json")))
    V_d, V_t = g["tiny_draft_vocab"], 1000
    w = di.lattice_workload(91, R=1, B=2, V_d=V_d, V_t=V_t, K=64, rank=8, pruned=True)
    S, d2t = w["subset"], w["d2t"]
    assert not np.all(np.diff(S) > 0)                       # unsorted subset
    m = od.d2t_map(np.arange(V_d), d2t)
    assert np.array_equal(m, S)
    t2d = {int(t): i for i, t in enumerate(m)}
    assert all(t2d[int(m[i])] == i for i in range(V_d))
    assert od.d2t_check(d2t, V_t, True) == od.OK
    bad = d2t.copy()
    bad[5] = V_t - 5                                         # maps to V_t: out of range
    assert od.d2t_check(bad, V_t, False) == od.ERANGE
    bad[5] = -6                                              # maps to -1
    assert od.d2t_check(bad, V_t, False) == od.ERANGE
    dup = d2t.copy()
    dup[7] = S[3] - 7                                        # two draft tokens on one target id
    assert od.d2t_check(dup, V_t, True) == od.EDUP
    assert od.d2t_check(dup, V_t, False) == od.OK          # greedy drafting accepts any mapping
    # the next-token table is zero outside the draft vocabulary, so are its transitions
    outside = np.setdiff1d(np.arange(V_t), S)
    E = di.bf16_bits_to_f32(w["E"])
    W = di.bf16_bits_to_f32(w["W"])
    t = od.tau(E, W, np.arange(20), outside[:50])
    assert np.all(t == 0.0)
    assert np.any(od.tau(E, W, np.arange(20), S[:50]) != 0.0)


def test_gate_and_head_hand_cases():
    assert od.gate(np.ones(16), np.zeros(16)) == 0.5
    assert od.gate([1.0, 2.0], [0.5, -0.25]) == 0.5
    assert abs(od.gate([2.0], [1.0]) - 1.0 / (1.0 + math.exp(-2.0))) < 1e-16
    E = np.array([[1.0], [2.0], [3.0]])
    W = np.array([[4.0], [5.0], [6.0]])
    cand = np.array([[0, 1], [2, 0]])
    A = od.lattice_request(cand, 2, E, W, [0.5, 2.0])
    np.testing.assert_array_equal(A[0], [[6.0, 7.5], [0.0, 0.0]])     # 0.5 * [3*4, 3*5]
    np.testing.assert_array_equal(A[1], [[12.0, 8.0], [24.0, 16.0]])  # 2 * [[1*6, 1*4], [2*6, 2*4]]
    assert np.all(od.lattice_request(cand, 2, np.zeros_like(E), W, [1.0, 1.0]) == 0)


def all_chain_scores(u, A):
    """Score of every one of the K^B chains, materialised (exhaustive enumeration)."""
    B, K = u.shape
    scores = u[0] + A[0, 0]
    for j in range(1, B):
        scores = scores[..., :, None] + A[j] + u[j]
    return scores


def check_against_enumeration(u, A):
    chain, score = od.chain_maxsum(u, A)
    scores = all_chain_scores(np.asarray(u, F64), A)
    best = scores.max()
    assert abs(score - best) <= 1e-12 * max(1.0, abs(best))
    flat = np.sort(scores.ravel())
    gap = flat[-1] - flat[-2]
    brute = np.unravel_index(np.argmax(scores), scores.shape)
    if gap > 1e-9:
        assert tuple(chain) == tuple(int(b) for b in brute)
    assert abs(od.chain_score(u, A, chain) - best) <= 1e-12 * max(1.0, abs(best))
    return chain


def test_maxsum_equals_exhaustive_enumeration_tiny_config():
    w = di.config1()
    rows = w["logits"]
    res = od.select_request(rows, w["K"], w["E"], w["W"], int(w["prev"][0]), "maxsum")
    assert res["cand_val"].shape == (7, 8)
    check_against_enumeration(res["cand_val"], res["A"])


def test_maxsum_equals_enumeration_strong_head():
    # rank-16 tables ~N(0,1): transitions of a few units, so the lattice changes chains
    rng = np.random.default_rng(5)
    changed = 0
    for trial in range(6):
        w = di.config1()
        E = rng.standard_normal((1024, 16))
        W = rng.standard_normal((1024, 16))
        res = od.select_request(w["logits"], 8, E, W, int(w["prev"][0]), "maxsum")
        chain = check_against_enumeration(res["cand_val"], res["A"])
        changed += int(np.any(chain != 0))
    assert changed >= 4


def test_zero_table_reduces_to_per_position_argmax():
    w = di.config1()
    E = np.zeros((1024, 16))
    for mode in ("maxsum", "walk"):
        res = od.select_request(w["logits"], 8, E, w["W"], 3, mode)
        assert np.all(res["chain"] == 0)
        for j in range(7):
            assert res["chain_tgt"][j] == int(np.argmax(w["logits"][j]))


def test_maxsum_and_walk_differ_on_a_hand_lattice():
    u = np.array([[1.0, 0.0], [0.0, 0.0]], dtype=F32)
    A = np.zeros((2, 2, 2))
    A[1, 1, 0] = 5.0
    assert list(od.chain_walk(u, A)[0]) == [0, 0]
    chain, score = od.chain_maxsum(u, A)
    assert list(chain) == [1, 0] and score == 5.0


def test_lattice_with_k_equal_v_is_the_dense_walk():
    rng = np.random.default_rng(17)
    V, B = 64, 7
    for trial in range(20):
        logits = (rng.standard_normal((B, V)) * 2).astype(F32)
        E = rng.standard_normal((V, 8)) * 0.7
        W = rng.standard_normal((V, 8)) * 0.7
        prev = int(rng.integers(0, V))
        res = od.select_request(logits, V, E, W, prev, "walk")
        dw = ow.dense_walk_request(logits, prev, E, W, T=0.0)
        assert list(res["chain_tgt"]) == list(dw["tokens"])


def test_dense_walk_with_zero_table_samples_the_raw_rows():
    from oracle.sampling import sample_row
    w = di.lattice_workload(92, R=1, B=5, V_d=3000, K=0, rank=16, dtype="f32", with_seeds=True)
    E = np.zeros((3000, 16))
    seed, step = int(w["seed"][0]), int(w["step"][0])
    dw = ow.dense_walk_request(w["logits"], 7, E, w["W"], T=0.9, top_p=0.8, seed=seed, step=step)
    from oracle.philox import uniform
    for j in range(5):
        tok, _ = sample_row(w["logits"][j], 0.9, 0.8, float(uniform(seed, step, j, 0)))
        assert dw["tokens"][j] == tok
