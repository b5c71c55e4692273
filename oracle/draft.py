"""Draft-side candidate selection (oracle; test infrastructure only).

Pages followed:
  [G] openvino.genai PR #4847, "Add DSpark and DFlash v2 drafts and sampled drafting to
      DFlash speculative decoding": Description > Change > Markov heads (Top-K
      candidate scorer over neighbouring positions; dense Markov walk); the commit on the
      block sampler and the DFlash candidate selector (rows scaled by the output
      multiplier and soft-capped; greedy walk taking the best candidate after the token
      before; sampled walk with the draft RNG; dense step biasing the scaled rows by the
      token drafted before); the commit on d2t checks (one entry per draft logit,
      injectivity required for sampled drafting only).
  [E] optimum-intel PR #2098, "[OpenVINO] Export DFlash v2 and DSpark drafts for
      PagedAttention and continuous batching": What does this PR do > DFlash v2 (packed
      Top-K lattice, transitions gated by the draft hidden states).
  [P] optimum-intel PR #2099, "[OpenVINO] Support MiniCPM-OCR-1.0-DSpark: DSpark drafts
      with a pruned vocabulary": What does this PR do > Pruned draft vocabulary (draft
      token i is target token i + d2t[i]) and > Markov head (table over the target
      vocabulary, zero outside the draft vocabulary; top_k = min(64, draft_vocab_size)).

Head form (the pages name it but give no formula; fixed by the specification of this
library): transition tau(a, b) = E[a] . W[b] with E, W in R^{V_t x rank}; gate
gamma = sigmoid(h . g) from the draft hidden state h of the position's own block row.

Precision: the pages fix none for the head or the chain, so tau, gamma, the lattice and
the max-sum recurrence run in float64 here. The greedy and sampled walks act on the
float rows the pages sample from, so their rows are float32: v = fl32(u + A).
"""
from __future__ import annotations

import math

import numpy as np

from .fp32 import F32, F64
from .philox import PURPOSE_DRAFT, uniform
from .sampling import sample_row

OK, EINVAL, ERANGE, EDUP = 0, 1, 2, 3


def row_transform(l, mult=1.0, softcap=0.0) -> np.ndarray:
    """s = l * mult, then softcap * tanh(s / softcap) when softcap > 0 (float32 rows)."""
    s = np.asarray(l, dtype=F32)
    if F32(mult) != F32(1.0):
        s = (s * F32(mult)).astype(F32)
    if softcap > 0:
        y = (s / F32(softcap)).astype(F32)
        s = (F32(softcap) * np.tanh(y.astype(F64)).astype(F32)).astype(F32)
    return s


def top_k_count(K: int, V_d: int) -> int:
    """K' = min(K, V_d): the scorer keeps at most one candidate per draft token [P]."""
    return min(int(K), int(V_d))


def topk_row(s, K):
    """The K' best entries of s ordered by (s descending, index ascending).
    -0.0 and +0.0 compare equal (then the lower index wins). Returns (idx, values)."""
    s = np.asarray(s, dtype=F32)
    Kp = top_k_count(K, s.shape[0])
    order = np.lexsort((np.arange(s.shape[0]), -s.astype(F64)))
    idx = order[:Kp]
    return idx, s[idx]


def d2t_map(idx, d2t):
    """Target id of draft index i: i + d2t[i] [P]; identity without a pruned vocabulary."""
    idx = np.asarray(idx, dtype=np.int64)
    return idx if d2t is None else idx + np.asarray(d2t, dtype=np.int64)[idx]


def d2t_check(d2t, V_t, require_injective) -> int:
    """Every draft index must map into [0, V_t); sampled drafting also needs a one-to-one map [G]."""
    d2t = np.asarray(d2t, dtype=np.int64)
    m = np.arange(d2t.shape[0], dtype=np.int64) + d2t
    if np.any(m < 0) or np.any(m >= V_t):
        return ERANGE
    if require_injective and np.unique(m).shape[0] != m.shape[0]:
        return EDUP
    return OK


def gate(h, g) -> float:
    """gamma = sigmoid(h . g), dot product in double [E]."""
    x = float(np.dot(np.asarray(h, dtype=F64), np.asarray(g, dtype=F64)))
    return 1.0 / (1.0 + math.exp(-x))


def tau(E, W, a_ids, b_ids) -> np.ndarray:
    """tau[a, b] = E[a_ids[a]] . W[b_ids[b]] in double."""
    Ea = np.asarray(E, dtype=F64)[np.asarray(a_ids)]
    Wb = np.asarray(W, dtype=F64)[np.asarray(b_ids)]
    return Ea @ Wb.T


def lattice_request(cand_tgt, prev, E, W, gammas) -> np.ndarray:
    """A[j, a, b] for one request (float64, shape [B, K', K']).
    Position 0: only row 0 is used, A[0, 0, b] = gamma_0 tau(prev, c_{0,b});
    position j >= 1: A[j, a, b] = gamma_j tau(c_{j-1,a}, c_{j,b})."""
    cand_tgt = np.asarray(cand_tgt)
    B, Kp = cand_tgt.shape
    A = np.zeros((B, Kp, Kp), dtype=F64)
    A[0, 0, :] = gammas[0] * tau(E, W, [prev], cand_tgt[0])[0]
    for j in range(1, B):
        A[j] = gammas[j] * tau(E, W, cand_tgt[j - 1], cand_tgt[j])
    return A


def chain_score(u, A, chain) -> float:
    """Sum of unary and transition scores along a chain of candidate ranks (double)."""
    u = np.asarray(u, dtype=F64)
    A = np.asarray(A, dtype=F64)
    total = u[0, chain[0]] + A[0, 0, chain[0]]
    for j in range(1, len(chain)):
        total += u[j, chain[j]] + A[j, chain[j - 1], chain[j]]
    return float(total)


def chain_maxsum(u, A):
    """Max-sum (Viterbi) chain over the lattice, in double. Ties: lowest predecessor
    rank in the recurrence, lowest final rank. Returns (ranks, score)."""
    u = np.asarray(u, dtype=F64)
    A = np.asarray(A, dtype=F64)
    B, Kp = u.shape
    delta = u[0] + A[0, 0]
    back = np.zeros((B, Kp), dtype=np.int64)
    for j in range(1, B):
        cand = delta[:, None] + A[j]            # [a, b]
        a_best = np.argmax(cand, axis=0)         # first maximum: lowest a
        delta = u[j] + cand[a_best, np.arange(Kp)]
        back[j] = a_best
    b = int(np.argmax(delta))
    score = float(delta[b])
    chain = [b]
    for j in range(B - 1, 0, -1):
        b = int(back[j, b])
        chain.append(b)
    return np.array(chain[::-1], dtype=np.int64), score


def walk_rows(u, A, chain_prefix_rank, j):
    """The float32 lattice row after the token before: v_b = fl32(u_j[b] + A_j[prev, b])."""
    row = A[0, 0] if j == 0 else A[j, chain_prefix_rank]
    return (np.asarray(u[j], dtype=F32) + np.asarray(row, dtype=F32)).astype(F32)


def penalize(v, ids, history, repetition=1.0, presence=0.0):
    """Repetition, then presence penalty on the row entries whose target id is in the history
    ([G] commit on the penalty history: the penalties apply to every token in the history whatever
    its count): s -> s / repetition if s > 0 else s * repetition, then s -> s - presence, in
    float32. repetition = 1 and presence = 0 leave the row unchanged."""
    v = np.asarray(v, dtype=F32).copy()
    hit = np.isin(np.asarray(ids), np.asarray(sorted(history), dtype=np.int64))
    if repetition != 1.0:
        r = F32(repetition)
        v[hit] = np.where(v[hit] > 0, (v[hit] / r).astype(F32), (v[hit] * r).astype(F32))
    if presence != 0.0:
        v[hit] = (v[hit] - F32(presence)).astype(F32)
    return v


def chain_walk(u, A, cand_tgt=None, history=None, repetition=1.0, presence=0.0):
    """Greedy walk [G]: b_0 = argmax(u_0 + A_0), b_j = argmax(u_j + A_j[b_{j-1}]) on float32
    rows, lowest rank on ties. Score: double sum of the chosen row entries. With a history (target
    ids), every row is penalized first over the history and the tokens drafted before it."""
    B = np.asarray(u).shape[0]
    chain, score, prev = [], 0.0, None
    seen = set(int(x) for x in history) if history is not None else None
    for j in range(B):
        v = walk_rows(u, A, prev, j)
        if seen is not None:
            v = penalize(v, cand_tgt[j], seen, repetition, presence)
        b = int(np.argmax(v))
        chain.append(b)
        score += float(v[b])
        prev = b
        if seen is not None:
            seen.add(int(cand_tgt[j][b]))
    return np.array(chain, dtype=np.int64), score


def chain_sample(u, A, cand_tgt, T, top_p, seed, step, min_p=0.0, history=None, repetition=1.0, presence=0.0):
    """Sampled walk [G]: at each position, sample the float32 lattice row after the token
    before over the K' candidates at temperature T, top-p and min-p, with the request's draft
    stream (purpose 0, position j). The candidate rank is the row index (ties in the
    nucleus order go to the lower rank). Returns (ranks, score, records) where each
    record holds the sparse q over kept ranks with their target ids."""
    B = np.asarray(u).shape[0]
    chain, score, recs, prev = [], 0.0, [], None
    seen = set(int(x) for x in history) if history is not None else None
    for j in range(B):
        v = walk_rows(u, A, prev, j)
        if seen is not None:
            v = penalize(v, cand_tgt[j], seen, repetition, presence)
        uu = float(uniform(seed, step, j, PURPOSE_DRAFT))
        b, rec = sample_row(v, T, top_p, uu, min_p)
        rec["ids"] = np.asarray(cand_tgt[j])[rec["kept"]]
        rec["u"] = uu
        rec["row"] = v
        chain.append(b)
        score += float(v[b])
        recs.append(rec)
        prev = b
        if seen is not None:
            seen.add(int(cand_tgt[j][b]))
    return np.array(chain, dtype=np.int64), score, recs


def lattice_row_sample(rows, cand_draft, u, A, T, top_p, seed, step, min_p=0.0, mult=1.0, softcap=0.0):
    """The block sampler's branch for any other request [G]: at position j, sample the lattice row
    after the token before over the whole draft vocabulary - the transformed row s_j with every
    candidate's entry replaced by its walk value fl32(u_j[b] + A_j[prev, b]) (position 0: A_0's
    row 0) - as a full-row multinomial request (temperature, top-p, min-p, U(seed, step, j, 0));
    a drawn token outside the candidates ends the block (no transition follows it).
    Returns (draft indices drawn, records); the number drawn is the block's length."""
    B = len(rows)
    toks, recs, prev = [], [], None
    for j in range(B):
        full = row_transform(rows[j], mult, softcap).copy()
        full[np.asarray(cand_draft[j])] = walk_rows(u, A, prev, j)
        uu = float(uniform(seed, step, j, PURPOSE_DRAFT)) if T > 0 else 0.0
        tok, rec = sample_row(full, T, top_p, uu, min_p)
        rec["row"] = full
        toks.append(int(tok))
        recs.append(rec)
        hit = np.nonzero(np.asarray(cand_draft[j]) == tok)[0]
        if hit.size == 0:
            break
        prev = int(hit[0])
    return np.array(toks, dtype=np.int64), recs


def select_request(logits_rows, K, E, W, prev, mode, d2t=None, hidden_rows=None, g=None,
                   mult=1.0, softcap=0.0, T=0.0, top_p=1.0, seed=0, step=0):
    """The whole Top-K scorer path for one request: rows -> candidates -> lattice -> chain."""
    B = len(logits_rows)
    cand, vals = [], []
    for j in range(B):
        s = row_transform(logits_rows[j], mult, softcap)
        i, v = topk_row(s, K)
        cand.append(i)
        vals.append(v)
    cand = np.array(cand)
    u = np.array(vals, dtype=F32)
    tgt = d2t_map(cand, d2t)
    gammas = [1.0] * B if hidden_rows is None else [gate(hidden_rows[j], g) for j in range(B)]
    A = lattice_request(tgt, prev, E, W, gammas)
    out = dict(cand_draft=cand, cand_tgt=tgt, cand_val=u, A=A, gammas=np.array(gammas))
    if mode == "maxsum":
        out["chain"], out["score"] = chain_maxsum(u, A)
    elif mode == "walk":
        out["chain"], out["score"] = chain_walk(u, A)
    else:
        out["chain"], out["score"], out["records"] = chain_sample(u, A, tgt, T, top_p, seed, step)
    out["chain_tgt"] = tgt[np.arange(B), out["chain"]]
    return out
