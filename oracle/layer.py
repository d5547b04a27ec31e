"""The layer step's stages over paged pools, shaped like the library's calls (oracle; test infrastructure only).

[P2] 全景图 (decode flow), steps C-E: compress -> RMSNorm -> RoPE -> cache insert and
SWA insertion; indexer scores -> top-K; main attention over the top-K compressed
entries plus the local window; inverse RoPE on the output.  [P2] 设计 1 / [P1] §2.2:
every cache is paged in 256-raw-position logical blocks through per-request tables.

A pool here holds decoded float64 rows (bf16 storage) or e4m3 codes plus a per-row
fp32 scale (fp8 storage), viewed as [num_blocks * rows_per_block, dim].  Writes round
to the storage format with this package's codecs, exactly as a stored row reads back.
"""
import numpy as np

from . import codecs, paging
from .attention import sparse_attention, window_positions, quantize_output
from .compress import RollingState, WINDOW, C4A, swa_rows
from .indexer import index_scores as _index_scores, visible_entries
from .rope import ROPE_THETA
from .topk import topk as _topk

BF16 = "bf16"
FP8 = "fp8_e4m3"
FP4 = "fp4_e2m1"


class Pool:
    """A paged cache pool: ``data`` [num_blocks * epb, dim], ``scale`` [num_blocks * epb] for fp8.

    bf16 pools hold either float64 values or the raw uint16 bit patterns (decoded on read); fp4 pools hold
    packed e2m1 bytes [num_blocks * epb, dim / 2] and a scale per row.
    """

    def __init__(self, epb, dtype, data, scale=None):
        self.epb = epb
        self.dtype = dtype
        self.data = data
        self.scale = scale
        self.bits = dtype == BF16 and data.dtype == np.uint16

    @property
    def num_blocks(self):
        return self.data.shape[0] // self.epb

    def read(self, table_row, ids):
        """Decoded float64 rows for logical ids."""
        rows = paging.physical_rows(table_row, ids, self.epb, self.num_blocks)
        if self.dtype == BF16:
            if self.bits:
                return codecs.bf16_decode(self.data[rows])
            return np.asarray(self.data[rows], dtype=np.float64)
        if self.dtype == FP4:
            return codecs.fp4_dequantize_rows(self.data[rows], self.scale[rows])
        return codecs.fp8_dequantize_rows(self.data[rows], self.scale[rows])

    def read_codes(self, table_row, ids):
        """Raw (codes, scale) of fp8 rows for logical ids."""
        rows = paging.physical_rows(table_row, ids, self.epb, self.num_blocks)
        return self.data[rows], self.scale[rows]

    def write(self, table_row, ids, values):
        """Round float64 rows to the storage format and store them at logical ids."""
        rows = paging.physical_rows(table_row, ids, self.epb, self.num_blocks)
        values = np.atleast_2d(np.asarray(values, dtype=np.float64))
        if self.dtype == BF16:
            self.data[rows] = codecs.bf16_encode(values) if self.bits else codecs.bf16_round(values)
        elif self.dtype == FP4:
            codes, scale = codecs.fp4_quantize_rows(values)
            self.data[rows] = codes
            self.scale[rows] = scale
        else:
            codes, scale = codecs.fp8_quantize_rows(values)
            self.data[rows] = codes
            self.scale[rows] = scale


def compress(kind, start_pos, x_new, z_new, states, rope_dim, out_pool, out_bt,
             swa_pool=None, swa_bt=None, gamma=None, eps=1e-6, theta=ROPE_THETA, record=None):
    """Append new raw tokens per request, emitting every entry they close.

    start_pos [B]; x_new[r] [n_r][d] and z_new[r] [n_r] (or [n_r][d], per-channel gate) hold request r's new tokens at
    positions start_pos[r] .. start_pos[r] + n_r - 1; states[r] is its RollingState,
    updated in place.  Entry i goes to ``out_pool`` logical row i; with an SWA pool,
    token p goes to its logical row p as R_p x_p.  Returns the emitted entry ids per request.
    With a dict ``record``, the float64 rows before storage rounding are also kept there:
    record[("entry", r, i)] and record[("swa", r, p)].
    """
    emitted = []
    for r in range(len(start_pos)):
        got = []
        for j in range(len(z_new[r])):
            p = int(start_pos[r]) + j
            res = states[r].step(x_new[r][j], z_new[r][j], p, rope_dim, gamma, eps, theta)
            if res is not None:
                i, entry = res
                out_pool.write(out_bt[r], [i], entry)
                got.append(i)
                if record is not None:
                    record[("entry", r, i)] = entry
            if swa_pool is not None:
                row = swa_rows(np.asarray(x_new[r][j])[None], [p], rope_dim, theta)
                swa_pool.write(swa_bt[r], [p], row)
                if record is not None:
                    record[("swa", r, p)] = row[0]
        emitted.append(got)
    return emitted


def index_scores(q_codes, q_scale, w, q_pos, q_req, key_pool, bt, kind=C4A, rows=None):
    """Scores of each query (or of the listed ``rows``) against its request's visible entries.

    Returns ({row: float64 [n_vis]}, {row: n_vis}).
    """
    rows = range(len(q_pos)) if rows is None else rows
    out, nvis = {}, {}
    for q in rows:
        m, r = int(q_pos[q]), int(q_req[q])
        n = visible_entries(m, kind)
        codes, scale = key_pool.read_codes(bt[r], np.arange(n))
        if key_pool.dtype == FP4:
            codes = codecs.fp4_unpack(codes)
        out[q] = _index_scores(q_codes[q], q_scale[q], w[q], codes, scale, n,
                               key_format="e2m1" if key_pool.dtype == FP4 else "e4m3")
        nvis[q] = n
    return out, nvis


def topk(scores_row, n_valid, k):
    """Top-k of one score row (see oracle.topk)."""
    return _topk(scores_row, n_valid, k)


def sparse_attn(q, q_pos, q_req, kind, topk_ids, main_pool, main_bt, swa_pool, swa_bt,
                window, sm_scale, rope_dim, theta=ROPE_THETA, rows=None):
    """Attention output of each query (or of the listed ``rows``).

    topk_ids[q] lists logical entry ids (-1 = none); ``topk_ids is None`` means every
    visible entry (the c128a dense case).  Returns ({row: out [H][d]}, {row: lse [H]}).
    """
    rows = range(len(q_pos)) if rows is None else rows
    out, lse = {}, {}
    for qi in rows:
        m, r = int(q_pos[qi]), int(q_req[qi])
        if topk_ids is None:
            ids = np.arange(visible_entries(m, kind))
        else:
            ids = np.asarray(topk_ids[qi])
            ids = ids[ids >= 0]
        comp = main_pool.read(main_bt[r], ids) if len(ids) else np.zeros((0, q.shape[-1]))
        win = swa_pool.read(swa_bt[r], window_positions(m, window))
        keys = np.concatenate([comp, win], axis=0)
        out[qi], lse[qi] = sparse_attention(q[qi], keys, m, rope_dim, sm_scale, theta)
    return out, lse


def sparse_attn_q8(q, q_pos, q_req, kind, topk_ids, main_pool, main_bt, swa_pool, swa_bt, window, sm_scale,
                   rope_dim, theta=ROPE_THETA, rows=None):
    """sparse_attn with the output in fp8 (quantize_output): ({row: (codes [H][d], scales [H][d/128])},
    {row: lse [H]}, {row: out [H][d] float64 before quantisation})."""
    out, lse = sparse_attn(q, q_pos, q_req, kind, topk_ids, main_pool, main_bt, swa_pool, swa_bt, window, sm_scale,
                           rope_dim, theta, rows)
    return {r: quantize_output(o) for r, o in out.items()}, lse, out


def ring_contents(states):
    """(x [B][w][d], z [B][w] or [B][w][d]) of a list of RollingStates, slot = position mod w."""
    return np.stack([s.x for s in states]), np.stack([s.z for s in states])


__all__ = ["Pool", "BF16", "FP8", "FP4", "compress", "index_scores", "topk", "sparse_attn", "sparse_attn_q8",
           "ring_contents", "WINDOW"]
