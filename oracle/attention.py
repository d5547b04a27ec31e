"""Sparse MQA attention with shared K = V, SWA merge and inverse RoPE (oracle; test infrastructure only).

[P1] §4.2-4.3: the main attention reads only the top-k entries, in an MQA-like mode
where every latent KV entry is shared by all query heads.  [P2] 机制一: K and V are
one stored tensor.  [P2] 机制四 / [P1] §5.3: a short sliding window of uncompressed
recent tokens is seen together with the compressed entries.  [P2] 深潜：为什么必须做
Inverse RoPE: since V = K carries R_n, the output is rotated back by R_m^-1, after
which it depends only on relative positions.  [P1] §2: softmax(QK^T / sqrt(d)) V.

Readings:
  * one softmax over the union of the selected compressed entries and the window
    rows (no deduplication: an entry and a window token are different vectors);
  * the window of the query at m is positions max(0, m - W + 1) .. m, W = 128,
    the current token included;
  * logit = <q_h, key> * sm_scale with sm_scale = 1/sqrt(512) by default;
  * out_h = R_m^-1 (sum_j p_j key_j), rotation acting on the last rope_dim dims.
"""
import numpy as np

from .codecs import e4m3_encode, fp8_row_scale
from .rope import rope, ROPE_THETA

SWA_WINDOW = 128
OUT_Q8_BLOCK = 128   # dims per fp8 output scale


def window_positions(m, window=SWA_WINDOW):
    """Raw positions in the sliding window of the query at m."""
    return np.arange(max(0, m - window + 1), m + 1)


def sparse_attention(q, keys, m, rope_dim, sm_scale, theta=ROPE_THETA, inverse_rope=True):
    """One query row: q [H][d] (already rotated at m), keys [n][d] (K = V).

    Returns (out [H][d], lse [H]) with lse the natural log of the softmax denominator
    of the scaled logits.  ``inverse_rope=False`` skips the final rotation (used only
    as a negative control in the tests).
    """
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    logits = (q @ keys.T) * sm_scale                      # [H][n]
    mx = np.max(logits, axis=1, keepdims=True)
    p = np.exp(logits - mx)
    l = np.sum(p, axis=1, keepdims=True)
    o = (p @ keys) / l                                    # [H][d]
    lse = (mx + np.log(l))[:, 0]
    if inverse_rope:
        o = rope(o, m, rope_dim, theta, inverse=True)
    return o, lse


def query_prep(q_raw, m, rope_dim, gamma=None, eps=1e-6, theta=ROPE_THETA):
    """The query of the attention from its raw projection ([P2] 融合点 3: Q-norm, done beside the key RoPE and
    insert): q_raw [..., H, d] at position m; every head's row is RMS-normalised,
    v_h = gamma * q_h / sqrt(mean(q_h^2) + eps), then rotated by R_m on the last rope_dim dims (the attention
    takes its queries rotated at their position, reading 4 of the attention above).

    Reading (the pages name the Q-norm only): the compressor's RMSNorm (gamma = 1, eps = 1e-6 unless given)
    and the rotation at the query's own position.
    """
    q = np.asarray(q_raw, dtype=np.float64)
    v = q / np.sqrt(np.mean(q * q, axis=-1, keepdims=True) + eps)
    if gamma is not None:
        v = v * np.asarray(gamma, dtype=np.float64)
    return rope(v, m, rope_dim, theta)


def quantize_output(o, block=OUT_Q8_BLOCK):
    """The fp8 form of an attention output ([P2] 融合点 2: the inverse-rotated output is quantised to fp8 for
    the o_lora projection that follows).  o [..., d] float64 (after R_m^-1); every `block` consecutive dims of a
    row share one fp32 scale = amax / 448 (1 for an all-zero block) and code = e4m3(value / scale).

    Reading (the pages name no granularity): one scale per (token, head, 128-dim block).
    Returns (codes uint8 [..., d], scales float64 [..., d / block]).
    """
    o = np.asarray(o, dtype=np.float64)
    d = o.shape[-1]
    assert d % block == 0
    blocks = o.reshape(o.shape[:-1] + (d // block, block))
    scale = fp8_row_scale(blocks)                             # [..., d/block], fp32 values
    codes = e4m3_encode(blocks / scale[..., None])
    return codes.reshape(o.shape), scale
