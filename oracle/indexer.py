"""Lightning-indexer scores (oracle; test infrastructure only).

[P1] §4.1 "Lightning Indexer": for query token t and history entry s the indexer
computes a cheap relevance score I_{t,s} with few heads, in FP8.  [P2] 机制三: the
indexer scores every compressed token and the top-K go on to the main attention.
The pages give no formula; the one used here is
    I(m, i) = sum_h w_h * ReLU(sq_h * sk_i * <q8_h, k8_i>)
with e4m3 query codes q8 and a per-(query, head) fp32 scale sq, e4m3 key codes k8
with a per-entry fp32 scale sk, and per-(query, head) weights w_h.

Causality ([P1] §5.3, [P2] 机制四): entry i is visible to the query at position m
only if the last raw token it covers is <= m, i.e. i < n_entries(m + 1).  Invisible
entries score -inf.
"""
import numpy as np

from .codecs import e4m3_decode, e2m1_decode
from .compress import n_entries


def visible_entries(m, kind):
    """Number of compressed entries a query at position m may see."""
    return n_entries(m + 1, kind)


def index_scores(q_codes, q_scale, w, k_codes, k_scale, n_visible, key_format="e4m3"):
    """Scores of one query against entries 0 .. len(k_codes) - 1.

    q_codes [H][d] uint8 (e4m3), q_scale [H], w [H], k_codes [n][d] uint8 (e4m3, or e2m1 codes 0..15 with
    key_format "e2m1": the fp4 indexer cache of [P2] 第三层), k_scale [n].
    Returns float64 [n]; entries at or beyond ``n_visible`` are -inf.
    """
    q = e4m3_decode(q_codes) * np.asarray(q_scale, dtype=np.float64)[:, None]   # [H][d]
    kdec = e2m1_decode if key_format == "e2m1" else e4m3_decode
    k = kdec(k_codes) * np.asarray(k_scale, dtype=np.float64)[:, None]          # [n][d]
    per_head = np.maximum(k @ q.T, 0.0)                                          # [n][H]
    scores = per_head @ np.asarray(w, dtype=np.float64)                          # [n]
    scores[n_visible:] = -np.inf
    return scores
