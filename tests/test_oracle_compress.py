"""Pins of the oracle's compressor and paging: the pages' entry counts, spans and block
geometry, closed forms of the gate, the bulk == incremental identity, and table translation."""
import math
import os

import numpy as np
import pytest

from oracle import compress as C, paging, rope as R, codecs
from oracle.layer import Pool, BF16, FP8, compress as layer_compress

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if line:
            out.append(line.split())
    return out


def test_entry_counts_golden():
    for kind, T, n in _rows("entry_counts.txt"):
        assert C.n_entries(int(T), kind) == int(n)
    # "about T/4" and "T/128" for every T that is a whole number of 256-position blocks
    for T in (256, 4096, 65536, 1 << 20):
        assert C.n_entries(T, C.C4A) == T // 4 - 1
        assert C.n_entries(T, C.C128A) == T // 128
    assert C.n_entries(7, C.C4A) == 0 and C.n_entries(8, C.C4A) == 1
    assert C.n_entries(127, C.C128A) == 0 and C.n_entries(128, C.C128A) == 1


def test_spans_golden_and_rope_position():
    for i, first, last in _rows("c4a_spans.txt"):
        assert C.entry_span(int(i), C.C4A) == (int(first), int(last))
        assert C.entry_position(int(i), C.C4A) == int(last)
    assert C.entry_span(0, C.C128A) == (0, 127)


def test_block_geometry_golden():
    want = {k: int(v) for k, v in _rows("block_geometry.txt")}
    assert paging.entries_per_block(C.WINDOW[C.C4A][1]) == want["c4a"]
    assert paging.entries_per_block(C.WINDOW[C.C128A][1]) == want["c128a"]
    assert paging.entries_per_block(1) == want["swa"]
    # every entry of a block starts inside that block's 256 raw positions
    for kind in (C.C4A, C.C128A):
        s = C.WINDOW[kind][1]
        epb = paging.entries_per_block(s)
        for i in range(3 * epb):
            assert (s * i) // 256 == i // epb


def test_gate_is_softmax_brute_force():
    z = [0.3, -1.2, 2.5, 0.0, 0.7, -0.1, 1.1, -3.0]
    e = [math.exp(v) for v in z]
    want = [v / sum(e) for v in e]
    assert np.allclose(C.gate(np.array(z)), want, rtol=1e-14)


def test_equal_logits_give_normalised_window_mean():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((8, 64))
    out = C.compress_entry(x, np.full(8, 0.37), pos=7, rope_dim=16)
    mean = x.mean(axis=0)
    want = R.rope(mean / math.sqrt(float(np.dot(mean, mean)) / 64 + 1e-6), 7, 16)
    assert np.allclose(out, want, atol=1e-12)


def test_dominant_logit_selects_one_token():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((8, 64))
    z = np.zeros(8)
    z[5] = 800.0
    out = C.compress_entry(x, z, pos=11, rope_dim=16)
    t = x[5]
    want = R.rope(t / math.sqrt(float(np.dot(t, t)) / 64 + 1e-6), 11, 16)
    assert np.allclose(out, want, atol=1e-12)


def test_rms_of_entry_before_rope_is_one():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((128, 512))
    u = C.rms_norm(C.gate(rng.standard_normal(128)) @ x, eps=0.0)
    assert abs(math.sqrt(np.mean(u * u)) - 1.0) < 1e-12


@pytest.mark.parametrize("kind,T", [(C.C4A, 203), (C.C128A, 515)])
def test_incremental_equals_bulk_bitwise(kind, T):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((T, 32))
    z = rng.standard_normal(T)
    bulk = C.compress_tokens(x, z, kind, rope_dim=8)
    st = C.RollingState(kind, 32)
    got = {}
    for p in range(T):
        res = st.step(x[p], z[p], p, rope_dim=8)
        if res is not None:
            got[res[0]] = res[1]
    assert sorted(got) == list(range(len(bulk)))
    for i, e in got.items():
        assert np.array_equal(e, bulk[i])


def test_paging_translation_and_unmapped_blocks():
    table = np.array([5, 2, -1, 0])
    epb = 64
    ids = np.array([0, 63, 64, 130, 200])
    with pytest.raises(paging.PagingError):
        paging.physical_rows(table, ids, epb, num_blocks=6)       # id 130 lies in unmapped block 2
    rows = paging.physical_rows(table, np.array([0, 63, 64, 127, 192, 255]), epb, num_blocks=6)
    assert list(rows) == [320, 383, 128, 191, 0, 63]
    with pytest.raises(paging.PagingError):
        paging.physical_rows(np.array([7]), [0], epb, num_blocks=6)  # block beyond the pool
    with pytest.raises(paging.PagingError):
        paging.physical_rows(table, [256], epb, num_blocks=6)        # beyond the table


def test_layer_compress_chunk_with_state_matches_bulk():
    """A chunk appended after cached tokens (state ring + new tokens) gives the bulk entries."""
    rng = np.random.default_rng(5)
    d, T0, n = 32, 37, 50
    x = codecs.bf16_round(rng.standard_normal((T0 + n, d)))
    z = rng.standard_normal(T0 + n)
    bulk = C.compress_tokens(x, z, C.C4A, rope_dim=8)
    # the ring holds the cached tokens' last 8 positions, slot = position mod 8
    ring_x = np.zeros((8, d))
    ring_z = np.zeros(8)
    for p in range(T0 - 8, T0):
        ring_x[p % 8], ring_z[p % 8] = x[p], z[p]
    st = C.RollingState(C.C4A, d, ring_x, ring_z)
    epb = 64
    pool = Pool(epb, BF16, np.zeros((2 * epb, d)))
    table = np.array([[1]])
    emitted = layer_compress(C.C4A, [T0], [x[T0:]], [z[T0:]], [st], 8, pool, table)
    first = C.n_entries(T0, C.C4A)
    assert emitted[0] == list(range(first, C.n_entries(T0 + n, C.C4A)))
    for i in emitted[0]:
        assert np.array_equal(pool.read(table[0], [i])[0], codecs.bf16_round(bulk[i]))
    for p in range(T0 + n - 8, T0 + n):                       # ring now holds the last 8 tokens
        assert np.array_equal(st.x[p % 8], x[p])


def test_layer_compress_fp8_pool_and_swa_rows():
    rng = np.random.default_rng(6)
    d = 16
    x = rng.standard_normal((12, d))
    z = rng.standard_normal(12)
    st = C.RollingState(C.C4A, d)
    pool = Pool(64, FP8, np.zeros((64, d), dtype=np.uint8), np.zeros(64))
    swa = Pool(256, BF16, np.zeros((256, d)))
    layer_compress(C.C4A, [0], [x], [z], [st], 8, pool, np.array([[0]]), swa, np.array([[0]]))
    e1 = C.compress_entry(x[4:12], z[4:12], 11, 8)
    codes, scale = codecs.fp8_quantize_rows(e1[None])
    assert np.array_equal(pool.data[1], codes[0]) and pool.scale[1] == scale[0]
    assert np.array_equal(swa.data[9], codecs.bf16_round(R.rope(x[9], 9, 8)))


# ---- per-channel gate (a variant: one logit per raw token and channel, a softmax down every channel) ----

def test_per_channel_gate_brute_force():
    """u_c = sum_j exp(z_jc) / sum_k exp(z_kc) * x_jc, written out with scalar loops on a tiny window."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((8, 5))
    z = rng.standard_normal((8, 5)) * 2.0
    u = np.zeros(5)
    for c in range(5):
        den = sum(math.exp(z[k, c]) for k in range(8))
        u[c] = sum(math.exp(z[j, c]) / den * x[j, c] for j in range(8))
    want = R.rope(u / math.sqrt(float(np.dot(u, u)) / 5 + 1e-6), 7, 0)
    got = C.compress_entry(x, z, pos=7, rope_dim=0)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-13)
    g = C.gate(z)
    assert g.shape == (8, 5) and np.allclose(g.sum(axis=0), 1.0, rtol=1e-14)


def test_per_channel_gate_with_equal_columns_is_the_scalar_gate():
    """Logits that are the same in every channel of a token give the scalar gate's entry (up to the order in
    which numpy sums a window: a one-dimensional sum and a column sum round differently in the last bit)."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((8, 64))
    zs = rng.standard_normal(8)
    scalar = C.compress_entry(x, zs, pos=15, rope_dim=16)
    per_channel = C.compress_entry(x, np.repeat(zs[:, None], 64, axis=1), pos=15, rope_dim=16)
    assert np.allclose(scalar, per_channel, rtol=1e-13, atol=1e-14)


def test_per_channel_gate_picks_a_token_per_channel():
    """A dominant logit in channel c selects token j_c for that channel only: different channels take their
    values from different tokens."""
    rng = np.random.default_rng(13)
    x = rng.standard_normal((8, 16))
    z = np.zeros((8, 16))
    pick = np.arange(16) % 8
    z[pick, np.arange(16)] = 800.0
    t = x[pick, np.arange(16)]
    want = t / math.sqrt(float(np.dot(t, t)) / 16 + 1e-6)
    assert np.allclose(C.compress_entry(x, z, pos=3, rope_dim=0), want, atol=1e-12)


@pytest.mark.parametrize("kind,T", [(C.C4A, 203), (C.C128A, 300)])
def test_per_channel_incremental_equals_bulk_bitwise(kind, T):
    rng = np.random.default_rng(14)
    x = rng.standard_normal((T, 32))
    z = rng.standard_normal((T, 32))
    bulk = C.compress_tokens(x, z, kind, rope_dim=8)
    st = C.RollingState(kind, 32, per_channel=True)
    got = {}
    for p in range(T):
        res = st.step(x[p], z[p], p, rope_dim=8)
        if res is not None:
            got[res[0]] = res[1]
    assert sorted(got) == list(range(len(bulk)))
    for i, e in got.items():
        assert np.array_equal(e, bulk[i])
