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


# ---- row transform: output multiplier, then soft cap ([G] block-sampler commit) ---------------

def test_row_transform_multiplier_is_one_rounded_product():
    # hand values: products by powers of two are exact; 0.1f * 3 rounds once
    l = np.array([3.0, -2.5, F32(0.1), 0.0, -0.0], dtype=F32)
    np.testing.assert_array_equal(od.row_transform(l, mult=0.5), np.array([1.5, -1.25, F32(0.1) / 2, 0.0, 0.0], F32))
    assert od.row_transform(np.array([F32(0.1)]), mult=3.0)[0] == F32(0.30000001192092896)
    # a float32 product is exact in double: one rounding of the exact product is the answer
    rng = np.random.default_rng(21)
    for mult in (0.75, 1.3, 23.0, 1e-3):
        x = (rng.standard_normal(5000) * 4).astype(F32)
        exact = x.astype(F64) * F64(F32(mult))
        np.testing.assert_array_equal(od.row_transform(x, mult=mult), exact.astype(F32))
    # identity when neither is set, and the input is not modified
    x = np.array([1.0, 2.0], dtype=F32)
    assert od.row_transform(x) is not x or np.array_equal(od.row_transform(x), x)
    np.testing.assert_array_equal(od.row_transform(x), x)


def test_row_transform_soft_cap_hand_values():
    tanh1 = 0.7615941559557649                              # tanh(1)
    s = od.row_transform(np.array([2.0, -2.0, 0.0, 1e6, -1e6], dtype=F32), softcap=2.0)
    np.testing.assert_allclose(s[:2], [2 * tanh1, -2 * tanh1], rtol=2 ** -23)
    assert s[2] == 0.0 and s[3] == F32(2.0) and s[4] == F32(-2.0)
    # multiplier first, then the cap: 4 * 0.5 = 2 -> 2 tanh(1)
    np.testing.assert_allclose(od.row_transform(np.array([4.0], F32), mult=0.5, softcap=2.0), [2 * tanh1],
                               rtol=2 ** -23)
    # the cap is 30 tanh(s / 30): s = 30 atanh(1/2) gives 15
    x = F32(30.0 * math.atanh(0.5))
    np.testing.assert_allclose(od.row_transform(np.array([x]), softcap=30.0), [15.0], rtol=2 ** -22)
    # near zero the cap is the identity to first order
    np.testing.assert_allclose(od.row_transform(np.array([1e-3], F32), softcap=30.0), [1e-3], rtol=1e-6)


def test_soft_cap_is_monotone_and_keeps_the_top_k():
    rng = np.random.default_rng(22)
    for trial in range(200):
        x = np.sort((rng.standard_normal(2000) * 6).astype(F32))
        y = od.row_transform(x, mult=float(rng.choice([1.0, 0.8, 2.5])), softcap=float(rng.choice([5.0, 15.0, 30.0])))
        assert np.all(np.diff(y.astype(F64)) >= 0)            # order preserving (ties possible when saturated)
        perm = rng.permutation(2000)
        xs, ys = x[perm], y[perm]
        idx_x, _ = od.topk_row(xs, 64)
        idx_y, vy = od.topk_row(ys, 64)
        if np.unique(vy).shape[0] == 64 and ys[ys >= vy[-1]].shape[0] == 64:
            assert list(idx_x) == list(idx_y)


# ---- sampled walk ([G] block-sampler commit: a sampled request walks the lattice with its draft RNG) ----

def test_chain_sample_low_temperature_is_the_greedy_walk():
    rng = np.random.default_rng(23)
    checked = 0
    for trial in range(60):
        B, K = 5, 16
        u = (rng.standard_normal((B, K)) * 2).astype(F32)
        A = rng.standard_normal((B, K, K)) * 2
        rows_ok = True
        walk, _ = od.chain_walk(u, A)
        prev = None
        for j in range(B):                                    # every row on the walk has a clear maximum
            v = np.sort(od.walk_rows(u, A, prev, j).astype(F64))
            rows_ok &= (v[-1] - v[-2]) > 0.05
            prev = walk[j]
        if not rows_ok:
            continue
        chain, _, recs = od.chain_sample(u, A, np.arange(B * K).reshape(B, K), 1e-4, 1.0, 77 + trial, 5)
        assert list(chain) == list(walk)
        assert all(r["kept"].shape[0] == 1 for r in recs)     # every other weight is flushed
        checked += 1
    assert checked >= 20


def test_chain_sample_draws_follow_the_hand_row():
    # one position, no transitions: the row is T log q for a hand q, so the draws follow q, and
    # top-p 0.7 keeps {0, 1} (0.5 + 0.25 is the first prefix above 0.7), renormalised to {2/3, 1/3}
    T = 0.8
    q = np.array([0.5, 0.25, 0.125, 0.125])
    u = (T * np.log(q)).astype(F32)[None, :]
    A = np.zeros((1, 4, 4))
    ids = np.array([[40, 41, 42, 43]])
    from scipy import stats
    for top_p, want in ((1.0, q), (0.7, np.array([2 / 3, 1 / 3, 0.0, 0.0]))):
        n = 20000
        counts = np.zeros(4)
        for s in range(n):
            chain, _, recs = od.chain_sample(u, A, ids, T, top_p, 1234, s)
            counts[chain[0]] += 1
        kept = want > 0
        assert counts[~kept].sum() == 0
        exp = want[kept] * n
        stat = np.sum((counts[kept] - exp) ** 2 / exp)
        assert stat < stats.chi2.ppf(0.999, kept.sum() - 1), stat
        np.testing.assert_allclose(recs[0]["q"], want[kept], rtol=1e-6)
        assert list(recs[0]["ids"]) == list(ids[0][kept])


def test_chain_sample_uses_the_position_word_of_the_draft_stream():
    # p = (1/2, 1/2) at every position: the index-order draw takes rank 1 exactly when u_j >= 1/2,
    # u_j = U(seed, step, j, purpose 0)
    from oracle.philox import uniform
    B = 12
    u = np.zeros((B, 2), dtype=F32)
    A = np.zeros((B, 2, 2))
    ids = np.tile(np.array([7, 9]), (B, 1))
    varied = 0
    for seed, step in ((1, 0), (2**40 + 3, 17), (99, 2**33 + 5)):
        chain, score, _ = od.chain_sample(u, A, ids, 1.0, 1.0, seed, step)
        want = [int(uniform(seed, step, j, 0) >= 0.5) for j in range(B)]
        assert list(chain) == want
        # the pin has teeth: the acceptance stream or the next position's word give other chains
        assert want != [int(uniform(seed, step, j, 1) >= 0.5) for j in range(B)]
        assert want != [int(uniform(seed, step, j + 1, 0) >= 0.5) for j in range(B)]
        varied += len(set(want)) > 1
    assert varied == 3


def test_chain_sample_reads_the_row_after_the_token_before():
    # A_j[a, b] = 50 exactly when b = a + 3 (mod K): the walk must step by +3 from the first draw
    # (a transposed lattice would step by -3); with top-p 0.5 the record keeps only the drawn rank
    rng = np.random.default_rng(24)
    B, K = 6, 8
    A = np.zeros((B, K, K))
    for j in range(1, B):
        for a in range(K):
            A[j, a, (a + 3) % K] = 50.0
    ids = rng.permutation(1000)[:B * K].reshape(B, K)
    for trial in range(10):
        u = (rng.standard_normal((B, K)) * 0.5).astype(F32)
        chain, score, recs = od.chain_sample(u, A, ids, 1.0, 0.5, 5 + trial, 3)
        for j in range(1, B):
            assert chain[j] == (chain[j - 1] + 3) % K
            assert list(recs[j]["ids"]) == [ids[j, chain[j]]]
        assert abs(score - od.chain_score(u, A, chain)) < 1e-4


def test_chain_sample_min_p_one_is_the_greedy_walk():
    """min_p = 1 keeps only the top candidate of every lattice row, so the sampled walk is the
    greedy walk, with q a point mass on its token."""
    rng = np.random.default_rng(31)
    B, K = 7, 16
    u = rng.standard_normal((B, K)).astype(np.float32)
    A = (rng.standard_normal((B, K, K)) * 0.5).astype(np.float32)
    tgt = rng.integers(0, 1000, size=(B, K))
    chain, _, recs = od.chain_sample(u, A, tgt, 0.8, 1.0, 12345, 9, min_p=1.0)
    walk, _ = od.chain_walk(u, A)
    assert np.array_equal(chain, walk)
    assert all(len(r["kept"]) == 1 and r["q"][0] == 1.0 for r in recs)


# ---- repetition / presence penalties over the history and the tokens drafted before -------------

def _rows2(v0, v1):
    """u rows for a 2-position walk with zero transitions (each row is its own lattice row)."""
    u = np.array([v0, v1], dtype=np.float32)
    A = np.zeros((2, len(v0), len(v0)), dtype=np.float32)
    return u, A


def test_penalties_neutral_values_leave_the_walk_unchanged():
    rng = np.random.default_rng(3)
    u = rng.standard_normal((6, 16)).astype(np.float32)
    A = (rng.standard_normal((6, 16, 16)) * 0.5).astype(np.float32)
    tgt = rng.integers(0, 40, size=(6, 16))
    plain, _ = od.chain_walk(u, A)
    pen, _ = od.chain_walk(u, A, tgt, history=set(range(40)), repetition=1.0, presence=0.0)
    assert np.array_equal(plain, pen)


def test_repetition_divides_positive_and_multiplies_negative_logits():
    tgt = np.array([[10, 11, 12], [10, 11, 12]])
    u, A = _rows2([2.0, 1.5, -1.0], [-1.0, -1.5, -3.0])
    # position 0: 2.0 / 2 = 1.0 < 1.5 -> candidate 1 (id 11); position 1: id 10 is in the history
    # (-1.0 * 2 = -2.0) and id 11 was drafted (-1.5 * 2 = -3.0), id 12 stays -3.0 -> candidate 0
    chain, score = od.chain_walk(u, A, tgt, history={10}, repetition=2.0)
    v1 = od.penalize(np.array([-1.0, -1.5, -3.0], np.float32), tgt[1], {10, 11}, 2.0, 0.0)
    assert list(v1) == [-2.0, -3.0, -3.0]
    assert list(chain) == [1, 0]


def test_presence_subtracts_and_drafted_tokens_join_the_history():
    tgt = np.array([[7, 8, 9], [9, 7, 5]])
    u, A = _rows2([2.0, 1.5, 0.0], [3.0, 2.9, 1.0])
    # position 0: id 7 (2.0) is not in the history: chosen; position 1: id 7 (2.9) was drafted and
    # id 9 (3.0) is in the history: 3.0 - 0.4 = 2.6, 2.9 - 0.4 = 2.5, 1.0 -> id 9
    chain, _ = od.chain_walk(u, A, tgt, history={9}, presence=0.4)
    assert list(chain) == [0, 0]
    # a large presence penalty pushes both penalized ids below id 5
    chain, _ = od.chain_walk(u, A, tgt, history={9}, presence=5.0)
    assert list(chain) == [0, 2]
    # position 0 is penalized too when its best id is in the history
    chain, _ = od.chain_walk(u, A, tgt, history={7}, presence=0.6)
    assert chain[0] == 1


def test_penalized_sampled_row_follows_the_penalized_softmax():
    from scipy import stats
    tgt = np.array([[1, 2, 3, 4]])
    u = np.array([[0.0, np.log(2.0), -1.0, 0.5]], dtype=np.float32)
    A = np.zeros((1, 4, 4), dtype=np.float32)
    hist = {2, 4}
    v = od.penalize(u[0], tgt[0], hist, 1.5, 0.3)        # ln2/1.5 - 0.3, 0.5/1.5 - 0.3
    p = np.exp(v.astype(np.float64) - v.max())
    p /= p.sum()
    n = 3000
    counts = np.zeros(4)
    for s in range(n):
        chain, _, recs = od.chain_sample(u, A, tgt, 1.0, 1.0, 1000 + s, 5, history=hist, repetition=1.5,
                                         presence=0.3)
        counts[chain[0]] += 1
    assert stats.chisquare(counts, p * n).pvalue > 1e-3
    np.testing.assert_allclose(np.asarray(recs[0]["q"], np.float64), p, rtol=2e-6)


# ---- the lattice-row branch: full-row samples of the walk row, ending outside the candidates ----

def test_lattice_row_sample_with_zero_transitions_samples_each_row():
    """A zero table leaves every candidate at its own logit, so each position is a plain full-row
    sample of its row (and a drawn non-candidate ends the block)."""
    from oracle.sampling import sample_row
    from oracle.philox import uniform
    rng = np.random.default_rng(8)
    B, V, K = 6, 200, 16
    rows = (rng.standard_normal((B, V)) * 2).astype(np.float32)
    cand = np.array([od.topk_row(r, K)[0] for r in rows])
    u = np.array([od.topk_row(r, K)[1] for r in rows], dtype=np.float32)
    A = np.zeros((B, K, K), dtype=np.float32)
    toks, recs = od.lattice_row_sample(rows, cand, u, A, 0.9, 1.0, 4242, 17)
    for j, t in enumerate(toks):
        want, _ = sample_row(rows[j], 0.9, 1.0, float(uniform(4242, 17, j, 0)))
        assert t == want
    ends = [j for j, t in enumerate(toks) if t not in cand[j]]
    assert ends == ([len(toks) - 1] if len(toks) < B else [])


def test_lattice_row_sample_with_every_token_a_candidate_is_the_sampled_walk():
    """K = V with the candidates in index order: the row is the walk row itself, ranks are indices,
    so the branch equals the sampled walk (tokens and q) and never ends early."""
    rng = np.random.default_rng(9)
    B, V = 5, 24
    rows = (rng.standard_normal((B, V)) * 1.5).astype(np.float32)
    cand = np.tile(np.arange(V), (B, 1))
    u = rows.copy()
    A = (rng.standard_normal((B, V, V)) * 0.7).astype(np.float32)
    toks, recs = od.lattice_row_sample(rows, cand, u, A, 0.8, 0.9, 777, 3)
    chain, _, crecs = od.chain_sample(u, A, cand, 0.8, 0.9, 777, 3)
    assert len(toks) == B and np.array_equal(toks, chain)
    for a, b in zip(recs, crecs):
        assert np.array_equal(a["kept"], b["kept"]) and np.array_equal(a["q"], b["q"])


def test_lattice_row_sample_ends_at_a_token_outside_the_candidates():
    """Candidates pushed far below the rest: the first draw is a non-candidate and ends the block."""
    rng = np.random.default_rng(10)
    B, V, K = 4, 50, 8
    rows = rng.standard_normal((B, V)).astype(np.float32)
    cand = np.tile(np.arange(K), (B, 1))
    u = rows[:, :K].copy()
    A = np.full((B, K, K), -200.0, dtype=np.float32)        # every walk value far below the rest
    toks, recs = od.lattice_row_sample(rows, cand, u, A, 1.0, 1.0, 5, 6)
    assert len(toks) == 1 and toks[0] >= K
