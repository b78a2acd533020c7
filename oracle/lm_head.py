"""The target model's greedy token at every tree node, oracle side (test infrastructure
only).

[HB] section 实现: the verifier's forward returns lm_head(norm(x)) for every tree node
(forward_with_mask) and takes pred = logits[node].argmax() at each node it visits;
[EAGLE2] section 5 (evaluate_posterior) compares each candidate with
torch.argmax(logits) at its parent. Here the final norm has been applied: `hidden` is
its output.
"""
from __future__ import annotations

import numpy as np


def lm_head_argmax(hidden, weight, chunk: int = 8192):
    """argmax over the vocabulary of hidden @ weight.T, row by row, and the largest
    logit. hidden [rows, H], weight [V, H] (the lm_head weight, one row per vocabulary
    entry). The logits are formed in fp64 from the given (bf16-representable) values;
    ties go to the lower vocabulary index (the first maximum). Computed over vocabulary
    chunks so the fp64 copy of the weight never exists whole."""
    h = np.asarray(hidden, np.float64)
    rows, v = h.shape[0], weight.shape[0]
    best = np.full(rows, -np.inf)
    idx = np.zeros(rows, np.int64)
    for v0 in range(0, v, chunk):
        logits = h @ np.asarray(weight[v0:v0 + chunk], np.float64).T
        j = logits.argmax(axis=1)  # first maximum within the chunk
        m = logits[np.arange(rows), j]
        better = m > best          # strictly larger: an earlier chunk keeps a tie
        best[better] = m[better]
        idx[better] = v0 + j[better]
    return idx, best
