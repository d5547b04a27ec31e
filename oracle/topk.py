"""Per-query top-k selection (oracle; test infrastructure only).

[P1] §4.2 "Top-k token selection": S_t = TopK(I_{t,:}, k); the main attention then
reads only the entries in S_t.  [P2] 机制三: k = 512 for c4a.

Readings: ties are broken toward the lower entry index, so S_t is one definite set;
when fewer than k entries are visible, all of them are taken and the rest of the
row is -1.  The set is returned in increasing index order.
"""
import numpy as np


def topk(scores, n_valid, k):
    """Indices of the k largest of scores[:n_valid], ties to lower index; int64 [k]."""
    s = np.asarray(scores, dtype=np.float64)[:n_valid]
    idx = np.arange(len(s))
    order = np.lexsort((idx, -s))         # primary: larger score; secondary: lower index
    chosen = np.sort(order[:k])
    out = np.full(k, -1, dtype=np.int64)
    out[:len(chosen)] = chosen
    return out
