"""Temperature softmax, top-p nucleus and the multinomial draw (oracle; test infrastructure only).

Follows openvino.genai PR #4847 ("Add DSpark and DFlash v2 drafts and sampled drafting
to DFlash speculative decoding"):
  * Description > Change > Sampled drafting: a multinomial request draws with the
    draft's RNG and records the distribution q of every candidate;
  * commit on the thresholded TopPFilter: the nucleus is the shortest prefix of the
    tokens ordered by probability (ties by index) whose mass exceeds top_p; exponents
    below -64 are flushed to zero;
  * commit on exact sampled speculative decoding: q is the post-filter distribution,
    sparse over the kept tokens or dense;
  * commit on double-precision multinomial sums: weights are summed in double;
  * commit on the double uniform: a draw takes one double uniform.

Readings where the pages are silent (each listed in the design notes):
  * the exponent that is flushed is z - zmax, z = s / T;
  * the draw walks the kept tokens in ascending index order and takes the first whose
    running double sum exceeds u * W_kept (W_kept is that same running sum's total);
    if rounding leaves none, the last kept token;
  * tokens of zero weight are never kept; with top_p >= 1, or when the mass never
    exceeds top_p, every token of positive weight is kept;
  * T <= 0 means greedy: the argmax, lowest index on ties, with q a point mass.
  * min-p (commit on the thresholded filters: MinPFilter collects the tokens whose probability
    is at least min_p times the top token's): applied after top-p, so the kept set is the
    nucleus intersected with {p_i >= min_p * p_max}; the common normaliser cancels, so the test
    is w_i >= min_p * w_max on the float32 weights (w_max = 1). The kept set stays a prefix of the
    (weight desc, index asc) order; when min-p cuts inside the nucleus, the record's cut is
    (min_p, the largest int32) (the pages leave the record's form open).
"""
from __future__ import annotations

import numpy as np

from .fp32 import F32, F64, weight


def softmax_weights(s, T):
    """z = s / T (float32 division), zmax, and the float32 weights of z - zmax."""
    s = np.asarray(s, dtype=F32)
    z = (s / F32(T)).astype(F32) if F32(T) != F32(1.0) else s.copy()
    zmax = z.max()
    d = (z - zmax).astype(F32)
    return z, zmax, weight(d)


def running_sum(w_in_order) -> np.ndarray:
    """Double running sum, one addition after another (numpy's accumulate is sequential)."""
    return np.cumsum(np.asarray(w_in_order, dtype=F64))


def nucleus_kept(w, top_p):
    """Indices kept by top-p, and the cut (w_cut, i_cut) that describes them:
    token i is kept iff w_i > w_cut, or w_i == w_cut and i <= i_cut."""
    w = np.asarray(w, dtype=F32)
    n = w.shape[0]
    positive = np.nonzero(w > 0)[0]
    if top_p >= 1.0:
        return positive, F32(0.0), -1
    total = running_sum(w)[-1]                       # W over the whole row, ascending index
    p = w.astype(F64) / total
    order = np.lexsort((np.arange(n), -w.astype(F64)))   # probability descending, index ascending
    order = order[w[order] > 0]
    cum = running_sum(p[order])
    over = np.nonzero(cum > F64(F32(top_p)))[0]
    if over.size == 0:
        return positive, F32(0.0), -1
    k = int(over[0])
    kept = np.sort(order[:k + 1])
    return kept, w[order[k]], int(order[k])


def min_p_kept(w, kept, min_p):
    """The kept tokens whose probability is at least min_p times the top token's:
    p_i >= min_p * p_max, i.e. w_i >= min_p * w_max (the normaliser cancels)."""
    w = np.asarray(w, dtype=F32)
    kept = np.asarray(kept)
    thr = F64(F32(min_p)) * F64(w.max())
    return kept[w[kept].astype(F64) >= thr]


MAX_INDEX = 2**31 - 1


def filtered_kept(w, top_p, min_p=0.0):
    """Top-p, then min-p: the kept indices (ascending) and their cut. When min-p cuts inside the
    nucleus (or there is none), the cut is (min_p, the largest int32), which the cut's rule reads
    as w_i >= min_p."""
    kept, w_cut, i_cut = nucleus_kept(w, top_p)
    if min_p > 0:
        kept = min_p_kept(w, kept, min_p)
        if not (F32(w_cut) >= F32(min_p)):
            w_cut, i_cut = F32(min_p), MAX_INDEX
    return kept, w_cut, i_cut


def draw_from_weights(w, kept, u):
    """First kept index (ascending) whose running double sum exceeds u * W_kept."""
    kept = np.asarray(kept)
    c = running_sum(np.asarray(w, dtype=F32)[kept])
    target = np.asarray(u, dtype=F64) * c[-1]
    pos = np.searchsorted(c, target, side="right")   # first c > target
    pos = np.minimum(pos, kept.size - 1)
    return kept[pos], c[-1]


def sample_row(s, T, top_p, u, min_p=0.0):
    """One draw from row s at temperature T, top-p and min-p, with the record of q.

    Returns (token, record) where record holds: z (float32 row), zmax, kept ids
    (ascending), q of each kept id (float32), W_kept (double), and the nucleus cut."""
    s = np.asarray(s, dtype=F32)
    if T <= 0:
        tok = int(np.argmax(s))
        rec = dict(kind="greedy", z=s, zmax=s[tok], kept=np.array([tok]), q=np.array([1.0], F32),
                   wsum=1.0, w_cut=F32(0.0), i_cut=-1)
        return tok, rec
    z, zmax, w = softmax_weights(s, T)
    kept, w_cut, i_cut = filtered_kept(w, top_p, min_p)
    tok, wsum = draw_from_weights(w, kept, u)
    q = (w[kept].astype(F64) / wsum).astype(F32)
    rec = dict(kind="sampled", z=z, zmax=zmax, w=w, kept=kept, q=q, wsum=wsum, w_cut=w_cut, i_cut=i_cut)
    return int(tok), rec


def dense_q(z, zmax, wsum, w_cut, i_cut, idx):
    """q(idx) from a dense record: the weight of z[idx] - zmax over W_kept, zero outside the cut."""
    idx = np.asarray(idx)
    d = (np.asarray(z, dtype=F32)[idx] - F32(zmax)).astype(F32)
    w = weight(d)
    kept = (w > F32(w_cut)) | ((w == F32(w_cut)) & (idx <= i_cut))
    kept &= w > 0
    return np.where(kept, w.astype(F64) / F64(wsum), 0.0)


def draw_margin(w, kept, u):
    """Distance, relative to W_kept, from u * W_kept to the nearest running-sum boundary;
    a GPU draw may differ from the oracle's only when this is at rounding level."""
    c = running_sum(np.asarray(w, dtype=F32)[np.asarray(kept)])
    target = F64(u) * c[-1]
    edges = np.concatenate(([0.0], c))
    return float(np.min(np.abs(edges - target)) / c[-1])
