"""Rotary position embedding on the last ``rope_dim`` dims (oracle; test infrastructure only).

[P2] "DeepSeek V4 稀疏注意力完全解剖", 深潜：为什么必须做 Inverse RoPE: a query at
position m is rotated by R_m, a key at n by R_n, and R_m R_n^T = R_(m-n).  The
cache rows carry RoPE on their last 64 dims (the rest, 448 of 512, carry none).

Reading of what the pages leave open: pair j (j = 0 .. rope_dim/2 - 1) is the
interleaved pair of dims (d - rope_dim + 2j, d - rope_dim + 2j + 1), rotated by
angle pos * theta^(-2j / rope_dim) with theta = 10000.  The pages do not say
whether pairs are interleaved or split in halves; every invariance used as a pin
holds for either.
"""
import numpy as np

ROPE_THETA = 10000.0


def inv_freq(rope_dim, theta=ROPE_THETA):
    """theta^(-2j/rope_dim) for j = 0 .. rope_dim/2 - 1, float64."""
    j = np.arange(rope_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * j / rope_dim)


def rope(v, pos, rope_dim, theta=ROPE_THETA, inverse=False):
    """Apply R_pos (or R_pos^-1 when ``inverse``) to the last ``rope_dim`` dims of v.

    v: [..., d] float64.  pos: scalar or array broadcastable to v.shape[:-1].
    """
    v = np.array(v, dtype=np.float64, copy=True)
    d = v.shape[-1]
    pos = np.asarray(pos, dtype=np.float64)
    ang = pos[..., None] * inv_freq(rope_dim, theta)          # [..., rope_dim/2]
    if inverse:
        ang = -ang
    c, s = np.cos(ang), np.sin(ang)
    x0 = v[..., d - rope_dim + 0::2].copy()
    x1 = v[..., d - rope_dim + 1::2].copy()
    v[..., d - rope_dim + 0::2] = x0 * c - x1 * s
    v[..., d - rope_dim + 1::2] = x0 * s + x1 * c
    return v
