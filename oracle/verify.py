"""Rejection-sampling verification of drafted tokens (oracle; test infrastructure only).

openvino.genai PR #4847, "Add DSpark and DFlash v2 drafts and sampled drafting to DFlash
speculative decoding":
  * commit on exact sampled speculative decoding: each window position is verified
    against the target's post-filter p with the standard test, accepting with probability
    min(1, p/q), otherwise emitting a sample of norm(max(0, p - q)) and dropping the later
    candidates; accepted tokens report the target's log-probability; ids beyond a model's
    row have zero probability under it; sums in double;
  * commit on the double uniform: the acceptance test takes a double uniform;
  * Description > Fixes > Split validation windows: every scheduled row validates the
    candidate after it, so row j checks drafted token j and row n is the bonus row.
This is the speculative sampling rule of Leviathan, Kalman and Matias (2023) and Chen et
al. (2023); its output follows p exactly.

Readings where the pages are silent (listed in the design notes):
  * u_accept = U(verify seed, step, j, purpose 1), u_residual = U(..., j, purpose 2);
    the bonus draw uses U(..., n, purpose 2);
  * if the residual has zero mass (possible only through rounding) the draw is from p;
  * every emitted token reports log p_j(token) of the post-filter target distribution;
    greedy requests (T <= 0) test x_j == argmax and report the T = 1 log-probability;
  * q(x_j) = 0 for a drafted token is a proposal error.
"""
from __future__ import annotations

import numpy as np

from .fp32 import F32, F64
from .philox import PURPOSE_ACCEPT, PURPOSE_RESIDUAL, uniform
from .sampling import draw_from_weights, filtered_kept, running_sum, softmax_weights

EPROPOSAL = 4


class TargetDist:
    """The target's post-filter distribution of one row at (T, top_p, min_p)."""

    def __init__(self, row, T, top_p, min_p=0.0):
        row = np.asarray(row, dtype=F32)
        self.V = row.shape[0]
        self.greedy = T <= 0
        Tw = 1.0 if self.greedy else T
        tp = 1.0 if self.greedy else top_p
        self.z, self.zmax, self.w = softmax_weights(row, Tw)
        self.argmax = int(np.argmax(row))
        self.kept, self.w_cut, self.i_cut = filtered_kept(self.w, tp, 0.0 if self.greedy else min_p)
        self.wsum = running_sum(self.w[self.kept])[-1]
        mask = np.zeros(self.V, dtype=bool)
        mask[self.kept] = True
        self.mask = mask

    def p(self, ids=None) -> np.ndarray:
        """Post-filter probabilities (double); ids outside the row have probability zero."""
        full = np.where(self.mask, self.w.astype(F64) / self.wsum, 0.0)
        if ids is None:
            return full
        ids = np.asarray(ids, dtype=np.int64)
        ok = (ids >= 0) & (ids < self.V)
        return np.where(ok, full[np.clip(ids, 0, self.V - 1)], 0.0)

    def logp(self, tok) -> float:
        return float(np.log(F64(self.w[tok])) - np.log(self.wsum))


def residual_draw(p_full, q_full, u):
    """Draw from norm(max(0, p - q)) over ascending ids; from p when that has no mass."""
    rho = np.maximum(0.0, np.asarray(p_full, dtype=F64) - np.asarray(q_full, dtype=F64))
    c = running_sum(rho)
    if c[-1] <= 0.0:
        c = running_sum(p_full)
    target = np.asarray(u, dtype=F64) * c[-1]
    pos = np.searchsorted(c, target, side="right")
    return np.minimum(pos, c.shape[0] - 1)


def verify_step(p_full, q_full, x, u_accept, u_residual):
    """One window position for arrays of trials (or scalars): accept x iff
    u_accept < p(x)/q(x); on rejection emit a residual draw. Returns (accepted, emitted)."""
    x = np.asarray(x, dtype=np.int64)
    px = np.asarray(p_full, dtype=F64)[x]
    qx = np.asarray(q_full, dtype=F64)[x]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = px / qx
    acc = np.asarray(u_accept, dtype=F64) < ratio
    res = residual_draw(p_full, q_full, u_residual)
    return acc, np.where(acc, x, res)


def verify_request(target_rows, drafted, n, q_rows, T, top_p, vseed, step, V_t=None, min_p=0.0):
    """Verify n drafted target tokens of one request.

    target_rows: [B+1, V_t] target logits; drafted: [B] target ids; q_rows(j) returns the
    dense q over target ids [V_t] recorded when token j was drafted.
    Returns dict(status, n_accepted, tokens (accepted + one correction or bonus),
    logprobs, margins)."""
    out_tokens, logps, margins = [], [], []
    for j in range(n):
        dist = TargetDist(target_rows[j], T, top_p, min_p)
        x = int(drafted[j])
        if dist.greedy:
            if x == dist.argmax:
                out_tokens.append(x)
                logps.append(dist.logp(x))
                continue
            out_tokens.append(dist.argmax)
            logps.append(dist.logp(dist.argmax))
            return dict(status=0, n_accepted=j, tokens=out_tokens, logprobs=logps, margins=margins)
        q_full = np.asarray(q_rows(j), dtype=F64)
        qx = q_full[x] if 0 <= x < q_full.shape[0] else 0.0
        if qx <= 0.0:
            return dict(status=EPROPOSAL, n_accepted=j, tokens=out_tokens, logprobs=logps, margins=margins)
        p_full = dist.p()
        ua = float(uniform(vseed, step, j, PURPOSE_ACCEPT))
        ur = float(uniform(vseed, step, j, PURPOSE_RESIDUAL))
        ratio = (p_full[x] if x < p_full.shape[0] else 0.0) / qx
        margins.append(abs(ua - ratio))
        if ua < ratio:
            out_tokens.append(x)
            logps.append(dist.logp(x))
            continue
        qq = np.zeros(dist.V, dtype=F64)
        lim = min(dist.V, q_full.shape[0])
        qq[:lim] = q_full[:lim]
        t = int(residual_draw(p_full, qq, ur))
        out_tokens.append(t)
        logps.append(dist.logp(t))
        return dict(status=0, n_accepted=j, tokens=out_tokens, logprobs=logps, margins=margins)
    dist = TargetDist(target_rows[n], T, top_p, min_p)
    if dist.greedy:
        t = dist.argmax
    else:
        ub = float(uniform(vseed, step, n, PURPOSE_RESIDUAL))
        t, _ = draw_from_weights(dist.w, dist.kept, ub)
        t = int(t)
    out_tokens.append(t)
    logps.append(dist.logp(t))
    return dict(status=0, n_accepted=n, tokens=out_tokens, logprobs=logps, margins=margins)
