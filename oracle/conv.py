"""DFlash-2 grouped dynamic convolution over packed block rows (oracle; test infrastructure only).

optimum-intel PR #2098 ("Export DFlash v2 and DSpark drafts for PagedAttention and continuous
batching"), What does this PR do > DFlash v2, and its commit on the per-row DFlash backbone: the
DFlash-2 draft's grouped dynamic convolution runs on the packed block rows of several requests,
shifts its taps along those rows, and masks every tap to the block of the row it produces, so no
tap reaches another request's block (openvino.genai PR #4847, Change > block sampler: every block
follows at least one context row, which keeps the blocks apart in the packed rows).

The pages give no formula; the plainest reading, stated here and used on both sides:
  x      [N, C] packed rows (one row per token of every request's block, blocks back to back);
  block  [N]    the block each row belongs to;
  k      [N, G, L] the dynamic taps: per produced row i, per channel group g, L taps;
  groups C channels in G contiguous groups of C / G channels (channel c is in group c // (C / G));
  y[i, c] = sum over t < L of k[i, g(c), t] * x[i - t, c], counting a tap only when row i - t
            exists and belongs to the same block as row i (the taps shift back along the rows).
Sums in float64 over the float32 (or bf16-exact) inputs.
"""
import numpy as np


def grouped_dynamic_conv(x, block, k) -> np.ndarray:
    """y[i, c] = sum_t k[i, g(c), t] * x[i - t, c] * [row i - t is in row i's block]."""
    x = np.asarray(x, dtype=np.float64)
    block = np.asarray(block)
    k = np.asarray(k, dtype=np.float64)
    N, C = x.shape
    G, L = k.shape[1], k.shape[2]
    assert k.shape[0] == N and C % G == 0
    gs = C // G
    y = np.zeros((N, C), dtype=np.float64)
    for i in range(N):
        for t in range(L):
            src = i - t
            if src < 0 or block[src] != block[i]:
                continue                          # the tap is masked to row i's block
            for g in range(G):
                y[i, g * gs:(g + 1) * gs] += k[i, g, t] * x[src, g * gs:(g + 1) * gs]
    return y
