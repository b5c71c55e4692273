"""Dense Markov walk, markov_head_top_k = 0 (oracle; test infrastructure only).

openvino.genai PR #4847, "Add DSpark and DFlash v2 drafts and sampled drafting to DFlash
speculative decoding": Description > Change > Markov heads (the dense Markov walk corrects
every drafted position, one head inference per position) and the commit on the block
sampler (a dense step biases the scaled rows by the token drafted before; greedy takes the
best biased token). optimum-intel PR #2099 ("... DSpark drafts with a pruned vocabulary"),
What does this PR do > Markov head: the next-token table is over the target vocabulary, so
the bias of draft token i is read at target id i + d2t[i].

Per request, for j = 0..B-1:
    v_j[i] = fl32( s_j[i] + gamma_j * tau(prev_j, m(i)) ),  i < V_d   (tau, gamma in double)
    x_j    = argmax v_j (lowest i) when greedy, else a draw from v_j at T, top_p with the
             draft stream (purpose 0, position j);
    prev_{j+1} = m(x_j); the drafted target token is m(x_j).
``forced_prev`` replaces prev_{j+1} by a given sequence (teacher forcing), so that every
position of another implementation can be checked against this one on its own.
"""
from __future__ import annotations

import numpy as np

from .draft import d2t_map, row_transform
from .fp32 import F32, F64
from .philox import PURPOSE_DRAFT, uniform
from .sampling import sample_row


def biased_row(s, E, Wm64, prev, gamma):
    """v = fl32(s + gamma * E[prev] . W[m(i)]) for all i (double before the rounding)."""
    t = Wm64 @ np.asarray(E[prev], dtype=F64)
    return (np.asarray(s, dtype=F64) + gamma * t).astype(F32)


def dense_walk_request(logit_rows, prev, E, W, d2t=None, gammas=None, mult=1.0, softcap=0.0,
                       T=0.0, top_p=1.0, seed=0, step=0, forced_prev=None, Wm64=None):
    B = len(logit_rows)
    V_d = np.asarray(logit_rows[0]).shape[0]
    m = d2t_map(np.arange(V_d), d2t)
    if Wm64 is None:
        Wm64 = np.asarray(W, dtype=F64)[m]
    gammas = [1.0] * B if gammas is None else gammas
    toks, idx, recs, rows, us = [], [], [], [], []
    p = int(prev)
    for j in range(B):
        s = row_transform(logit_rows[j], mult, softcap)
        v = biased_row(s, E, Wm64, p, gammas[j])
        u = float(uniform(seed, step, j, PURPOSE_DRAFT)) if T > 0 else 0.0
        x, rec = sample_row(v, T, top_p, u)
        idx.append(x)
        toks.append(int(m[x]))
        recs.append(rec)
        rows.append(v)
        us.append(u)
        p = int(m[x]) if forced_prev is None else int(forced_prev[j])
    return dict(tokens=np.array(toks), draft_idx=np.array(idx), records=recs, rows=rows, u=us)
