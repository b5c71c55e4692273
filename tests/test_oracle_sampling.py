"""Pins for the oracle's softmax, nucleus and multinomial draw."""
import json
import os

import numpy as np
import pytest
from scipy import stats

from oracle.fp32 import F32, F64
from oracle.philox import uniform
from oracle.sampling import draw_from_weights, nucleus_kept, sample_row, softmax_weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def chi2_ok(counts, probs, alpha=1e-3):
    counts = np.asarray(counts, dtype=np.float64)
    exp = np.asarray(probs, dtype=np.float64) * counts.sum()
    keep = exp > 5
    stat = np.sum((counts[keep] - exp[keep]) ** 2 / exp[keep])
    return stat < stats.chi2.ppf(1 - alpha, keep.sum() - 1), stat


@pytest.mark.parametrize("V,T,top_p", [(8, 0.7, 1.0), (64, 1.0, 0.9), (64, 0.5, 0.95)])
def test_draws_follow_q(V, T, top_p):
    rng = np.random.default_rng(V)
    s = (rng.standard_normal(V) * 2).astype(F32)
    z, zmax, w = softmax_weights(s, T)
    kept, _, _ = nucleus_kept(w, top_p)
    n = 1_000_000
    u = uniform(99, np.arange(n, dtype=np.uint64), 0, 0)
    tok, wsum = draw_from_weights(w, kept, u)
    counts = np.bincount(tok, minlength=V)
    q = np.zeros(V)
    q[kept] = w[kept].astype(F64) / wsum
    assert counts[q == 0].sum() == 0
    ok, stat = chi2_ok(counts, q)
    assert ok, stat
    # the reference distribution is the plain softmax at T, restricted to the nucleus
    ref = np.exp((s.astype(F64) - s.max()) / T)
    ref /= ref.sum()
    if top_p >= 1:
        np.testing.assert_allclose(q, ref, rtol=1e-5)


def thresholded_nucleus(w, top_p):
    """Independent construction of the nucleus by threshold rounds (openvino.genai PR #4847,
    commit on the thresholded TopPFilter): keep tokens with p >= p_max * e^-10, then e^-20,
    e^-40, then all; sort the survivors by probability with ties by index; walk them until
    the mass exceeds top_p."""
    total = np.cumsum(w.astype(F64))[-1]
    p = w.astype(F64) / total
    pmax = p.max()
    for thr in (pmax * np.exp(-10.0), pmax * np.exp(-20.0), pmax * np.exp(-40.0), 0.0):
        cand = [i for i in range(len(p)) if p[i] >= thr and p[i] > 0]
        cand.sort(key=lambda i: (-p[i], i))
        mass = 0.0
        for k, i in enumerate(cand):
            mass += p[i]
            if mass > float(F32(top_p)):
                return sorted(cand[:k + 1])
    return sorted(i for i in range(len(p)) if p[i] > 0)


def test_nucleus_is_full_sort_prefix():
    rng = np.random.default_rng(7)
    for trial in range(10000):
        V = int(rng.integers(2, 64))
        scale = float(rng.choice([0.1, 1.0, 4.0, 20.0]))
        s = (rng.standard_normal(V) * scale).astype(F32)
        if trial % 3 == 0:
            s = np.round(s)            # many exact ties
        top_p = float(rng.choice([0.1, 0.5, 0.9, 0.95, 0.999]))
        _, _, w = softmax_weights(s, 1.0)
        kept, w_cut, i_cut = nucleus_kept(w, top_p)
        assert list(kept) == thresholded_nucleus(w, top_p)
        idx = np.arange(V)
        by_cut = np.nonzero((w > 0) & ((w > w_cut) | ((w == w_cut) & (idx <= i_cut))))[0]
        assert list(by_cut) == list(kept)


def test_worked_example_tail_is_drawn():
    g = json.load(open(os.path.join(GOLDEN, "worked_example_float_sums.json")))
    w = np.concatenate([np.array(g["head_weights"], dtype=F32),
                        np.full(g["tail_count"], g["tail_weight"], dtype=F32)])
    kept = np.arange(w.shape[0])
    n = 1_000_000
    u = uniform(2024, np.arange(n, dtype=np.uint64), 0, 0)
    tok, wsum = draw_from_weights(w, kept, u)
    tail = np.mean(tok >= 2)
    se = np.sqrt(g["tail_mass"] * (1 - g["tail_mass"]) / n)
    assert abs(tail - g["tail_mass"]) < 5 * se
    # the pin has teeth: running sums in float32 never reach the tail
    c32 = np.cumsum(w, dtype=F32)
    tok32 = np.minimum(np.searchsorted(c32, (u * c32[-1]).astype(F32), side="right"), w.shape[0] - 1)
    assert np.mean(tok32 >= 2) < 1e-4


def test_low_temperature_is_argmax_and_greedy_ties():
    rng = np.random.default_rng(3)
    for _ in range(200):
        s = (rng.standard_normal(1000) * 2).astype(F32)
        tok, _ = sample_row(s, 1e-3, 1.0, float(rng.random()))
        assert tok == int(np.argmax(s))
    s = np.array([1.0, 3.0, 3.0, -0.0, 0.0], dtype=F32)
    assert sample_row(s, 0.0, 1.0, 0.5)[0] == 1
    assert sample_row(s, -1.0, 1.0, 0.5)[0] == 1


def test_flush_below_minus_64():
    s = np.array([0.0, -63.5, -64.5, -200.0], dtype=F32)
    _, _, w = softmax_weights(s, 1.0)
    assert w[0] == 1 and w[1] > 0 and w[2] == 0 and w[3] == 0


def test_dense_q_is_the_distribution_drawn_from():
    # [G] exact sampled speculative decoding: the record is the post-filter q each token was drawn
    # from. Rebuilt from a dense record (z, zmax, W_kept, cut), q must equal sample_row's q on the
    # kept set and vanish elsewhere, ties at the cut included.
    from oracle.sampling import dense_q
    rng = np.random.default_rng(31)
    for trial in range(10000):
        V = int(rng.integers(2, 64))
        s = (rng.standard_normal(V) * float(rng.choice([0.5, 2.0, 8.0]))).astype(F32)
        if trial % 2 == 0:
            s = np.round(s)                                   # exact ties, also at the cut
        T = float(rng.choice([0.5, 0.8, 1.0, 1.7]))
        top_p = float(rng.choice([0.3, 0.5, 0.9, 0.95, 1.0]))
        tok, rec = sample_row(s, T, top_p, float(rng.random()))
        dq = dense_q(rec["z"], rec["zmax"], rec["wsum"], rec["w_cut"], rec["i_cut"], np.arange(V))
        mask = np.zeros(V, dtype=bool)
        mask[rec["kept"]] = True
        assert np.all(dq[~mask] == 0.0)
        assert np.array_equal(dq[mask].astype(F32), rec["q"])
        assert dq[tok] > 0.0
        assert abs(dq.sum() - 1.0) < 1e-12


def test_dense_q_matches_draw_frequencies():
    from oracle.sampling import dense_q
    rng = np.random.default_rng(32)
    s = np.round(rng.standard_normal(40) * 2).astype(F32)
    n = 400000
    _, rec = sample_row(s, 0.9, 0.8, 0.5)
    u = uniform(3, np.arange(n, dtype=np.uint64), 0, 0)
    tok, _ = draw_from_weights(rec["w"], rec["kept"], u)      # the draw sample_row makes, vectorised
    counts = np.bincount(tok, minlength=40).astype(np.float64)
    dq = dense_q(rec["z"], rec["zmax"], rec["wsum"], rec["w_cut"], rec["i_cut"], np.arange(40))
    assert counts[dq == 0].sum() == 0
    ok, stat = chi2_ok(counts, dq)
    assert ok, stat


# ---- min-p (pinned by hand-computed kept sets, the intersection with top-p, the record's cut and
# the draws' frequencies) ------------------------------------------------------------------------

def _halving_row():
    # weights 1, 1/2, 1/4, 1/8 (to the polynomial's accuracy) and one flushed token
    return np.array([0.0, -np.log(2.0), -2 * np.log(2.0), -3 * np.log(2.0), -80.0], dtype=np.float32)


@pytest.mark.parametrize("min_p,want", [(0.0, [0, 1, 2, 3]), (0.3, [0, 1]), (0.2, [0, 1, 2]), (0.5001, [0]),
                                        (1.0, [0]), (0.124, [0, 1, 2, 3])])
def test_min_p_keeps_tokens_at_least_min_p_times_the_top(min_p, want):
    from oracle.sampling import filtered_kept, softmax_weights
    _, _, w = softmax_weights(_halving_row(), 1.0)
    kept, w_cut, i_cut = filtered_kept(w, 1.0, min_p)
    assert list(kept) == want


def test_min_p_after_top_p_is_the_intersection():
    from oracle.sampling import filtered_kept, softmax_weights
    _, _, w = softmax_weights(_halving_row(), 1.0)
    # p = (8, 4, 2, 1) / 15: the running mass 8/15, 12/15, 14/15 first exceeds 0.85 at the third token
    assert list(filtered_kept(w, 0.85, 0.0)[0]) == [0, 1, 2]
    assert list(filtered_kept(w, 0.85, 0.3)[0]) == [0, 1]          # min-p cuts inside the nucleus
    assert list(filtered_kept(w, 0.85, 0.1)[0]) == [0, 1, 2]       # the nucleus cuts first
    assert list(filtered_kept(w, 0.5, 0.3)[0]) == [0]              # 8/15 > 0.5 already


def test_min_p_record_cut_describes_the_kept_set():
    from oracle.sampling import dense_q, sample_row
    rng = np.random.default_rng(17)
    for trial in range(40):
        s = np.round(rng.standard_normal(300) * 2, 1).astype(np.float32)   # many equal weights
        T, top_p, min_p = [(1.0, 1.0, 0.05), (0.7, 0.9, 0.2), (1.3, 0.95, 0.01)][trial % 3]
        tok, rec = sample_row(s, T, top_p, 0.37, min_p)
        q = dense_q(rec["z"], rec["zmax"], rec["wsum"], rec["w_cut"], rec["i_cut"], np.arange(300))
        kept = np.nonzero(q > 0)[0]
        assert np.array_equal(kept, rec["kept"])
        assert np.all(rec["w"][kept].astype(np.float64) >= np.float64(np.float32(min_p)))
        np.testing.assert_allclose(q[kept], rec["q"].astype(np.float64), rtol=1e-6)


def test_min_p_draws_follow_the_renormalised_kept_mass():
    from scipy import stats
    from oracle.sampling import sample_row
    s = _halving_row()
    n = 4000
    u = (np.arange(n) + 0.5) / n                                  # an exact quadrature of the uniform
    toks = np.array([sample_row(s, 1.0, 1.0, float(x), 0.2)[0] for x in u])
    counts = np.bincount(toks, minlength=5)
    assert counts[3] == 0 and counts[4] == 0
    exp = np.array([4, 2, 1]) / 7 * n
    assert stats.chisquare(counts[:3], exp).pvalue > 0.99


def test_nucleus_membership_is_the_mass_above_at_most_top_p():
    """The sampled walk decides membership without sorting: candidate i is kept when the mass of
    the candidates above it in the (weight desc, index asc) order is at most top_p. Against the
    oracle's sorted prefix, with that mass summed exactly (math.fsum): equal except where a running
    sum lies within rounding of top_p."""
    import math
    rng = np.random.default_rng(17)
    for trial in range(5000):
        V = int(rng.integers(2, 65))
        s = (rng.standard_normal(V) * float(rng.choice([0.3, 2.0, 8.0]))).astype(F32)
        if trial % 2 == 0:
            s = np.round(s)            # ties in weight: the index decides the order
        top_p = float(rng.choice([0.2, 0.5, 0.9, 0.95]))
        _, _, w = softmax_weights(s, 1.0)
        kept, _, _ = nucleus_kept(w, top_p)
        total = math.fsum(float(x) for x in w)
        tp = float(F32(top_p))
        above = [math.fsum(float(w[k]) for k in range(V) if (w[k], -k) > (w[i], -i)) / total for i in range(V)]
        by_mass = [i for i in range(V) if w[i] > 0 and above[i] <= tp]
        if by_mass != list(kept):
            near = min(abs(a - tp) for a in above) < 1e-12 or \
                min(abs(a + float(w[i]) / total - tp) for i, a in enumerate(above)) < 1e-12
            assert near, (trial, by_mass, list(kept))
