"""c4a / c128a compressor and SWA rows (oracle; test infrastructure only).

[P1] §5.2 "多token压缩：c4a和c128a" and [P2] 机制二: a c4a compressed token is a
weighted sum of 8 raw tokens taken at stride 4 (neighbours overlap by 4), so about
T/4 entries remain; a c128a token sums 128 raw tokens at stride 128, T/128 entries.
[P2] 融合点 1 fixes the chain that follows the sum: RMSNorm, then RoPE, then the
cache insert.  [P2] 设计 2: the compressor keeps a rolling residual of the last
coff * ratio raw tokens (8 for c4a, 128 for c128a) between steps.

Readings where the pages are open (each also listed in the design notes):
  * gate: g_j = softmax_j(z) over the window, one scalar logit z per raw token, the
    same logit in both windows that contain a token;
  * per-channel gate (a variant; the pages say only "weighted sum"): one logit per raw token and
    channel, z [T][d], and a separate softmax over the window for every channel c,
    u_c = sum_j softmax_j(z_{., c})_j x_{j, c};
  * RMSNorm: v = gamma * u / sqrt(mean(u^2) + eps), gamma = 1, eps = 1e-6 unless given;
  * entry i covers raw positions s*i .. s*i + w - 1 and is rotated at the last one,
    pos_i = s*i + w - 1;
  * an SWA row is the raw token rotated at its own position, s_p = R_p x_p
    ([P2] 融合点 3: the uncompressed path's keys get RoPE and are inserted).
"""
import numpy as np

from .rope import rope, ROPE_THETA

C4A = "c4a"
C128A = "c128a"
WINDOW = {C4A: (8, 4), C128A: (128, 128)}     # kind -> (window w, stride s)
RMS_EPS = 1e-6


def n_entries(T, kind):
    """Entries fully formed from T raw tokens: 0 if T < w, else floor((T - w) / s) + 1."""
    w, s = WINDOW[kind]
    return 0 if T < w else (T - w) // s + 1


def entry_span(i, kind):
    """First and last raw position covered by entry i."""
    w, s = WINDOW[kind]
    return s * i, s * i + w - 1


def entry_position(i, kind):
    """RoPE position of entry i: the last raw token it covers."""
    return entry_span(i, kind)[1]


def gate(z):
    """Softmax over the window (axis 0) of the window's logits, float64: z [w] (one weight per token) or
    z [w][d] (per channel: a softmax down every column)."""
    z = np.asarray(z, dtype=np.float64)
    e = np.exp(z - np.max(z, axis=0))
    return e / np.sum(e, axis=0)


def rms_norm(u, gamma=None, eps=RMS_EPS):
    """u / sqrt(mean(u^2) + eps), times gamma if given."""
    u = np.asarray(u, dtype=np.float64)
    v = u / np.sqrt(np.mean(u * u) + eps)
    return v if gamma is None else v * np.asarray(gamma, dtype=np.float64)


def compress_entry(x_win, z_win, pos, rope_dim, gamma=None, eps=RMS_EPS, theta=ROPE_THETA):
    """One compressed entry: R_pos(RMSNorm(sum_j g_j x_j)) with g = softmax(z_win); z_win [w] (scalar gate) or
    [w][d] (per-channel gate, g_j a vector multiplying x_j element by element)."""
    g = gate(z_win)
    if g.ndim == 1:
        g = g[:, None]
    u = np.sum(g * np.asarray(x_win, dtype=np.float64), axis=0)
    return rope(rms_norm(u, gamma, eps), pos, rope_dim, theta)


def compress_tokens(x, z, kind, rope_dim, gamma=None, eps=RMS_EPS, theta=ROPE_THETA):
    """All entries formed from raw tokens x [T][d] with logits z [T] or [T][d] (bulk path)."""
    w, s = WINDOW[kind]
    x = np.asarray(x, dtype=np.float64)
    n = n_entries(x.shape[0], kind)
    out = np.empty((n, x.shape[1]), dtype=np.float64)
    for i in range(n):
        a = s * i
        out[i] = compress_entry(x[a:a + w], z[a:a + w], a + w - 1, rope_dim, gamma, eps, theta)
    return out


class RollingState:
    """Per-request residual: the last w raw tokens and logits, slot = position mod w (logits [w], or [w][d]
    for the per-channel gate)."""

    def __init__(self, kind, dim, ring_x=None, ring_z=None, per_channel=False):
        self.kind = kind
        w, _ = WINDOW[kind]
        self.x = np.zeros((w, dim)) if ring_x is None else np.array(ring_x, dtype=np.float64)
        zshape = (w, dim) if per_channel else (w,)
        self.z = np.zeros(zshape) if ring_z is None else np.array(ring_z, dtype=np.float64)

    def step(self, x_p, z_p, p, rope_dim, gamma=None, eps=RMS_EPS, theta=ROPE_THETA):
        """Append token p; return (i, entry) when p closes entry i, else None."""
        w, s = WINDOW[self.kind]
        self.x[p % w] = x_p
        self.z[p % w] = z_p
        if p + 1 < w or (p + 1 - w) % s != 0:
            return None
        i = (p + 1 - w) // s
        slots = [(q % w) for q in range(p - w + 1, p + 1)]
        return i, compress_entry(self.x[slots], self.z[slots], p, rope_dim, gamma, eps, theta)


def swa_rows(x, positions, rope_dim, theta=ROPE_THETA):
    """Sliding-window rows s_p = R_p x_p for raw tokens x [n][d] at positions [n]."""
    return rope(x, np.asarray(positions), rope_dim, theta)
