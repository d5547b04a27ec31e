"""Pins of the oracle's indexer, top-k and attention: brute force on tiny inputs, the
visibility rule, dense equivalence, translation invariance from inverse RoPE (with its
negative control), the m = 0 and single-key cases, and paged reads."""
import math

import numpy as np
import pytest

from oracle import codecs, compress as C, rope as R
from oracle.attention import sparse_attention, window_positions
from oracle.indexer import index_scores, visible_entries
from oracle.layer import Pool, BF16, sparse_attn
from oracle.topk import topk


def test_visibility_rule():
    # [P2] 机制四: the query at position 5 cannot see c128a entry 0, which covers 0..127
    assert visible_entries(5, C.C128A) == 0
    assert visible_entries(126, C.C128A) == 0 and visible_entries(127, C.C128A) == 1
    assert visible_entries(6, C.C4A) == 0 and visible_entries(7, C.C4A) == 1
    assert visible_entries(10, C.C4A) == 1 and visible_entries(11, C.C4A) == 2
    for m in range(300):
        n = visible_entries(m, C.C4A)
        assert all(C.entry_span(i, C.C4A)[1] <= m for i in range(n))
        assert C.entry_span(n, C.C4A)[1] > m


def test_window_is_128_positions_including_current():
    assert list(window_positions(0)) == [0]
    assert list(window_positions(200)) == list(range(73, 201))
    assert len(window_positions(10 ** 6)) == 128


def test_index_scores_brute_force():
    rng = np.random.default_rng(7)
    H, d, n = 3, 8, 11
    qc = codecs.e4m3_encode(rng.standard_normal((H, d)) * 4)
    kc = codecs.e4m3_encode(rng.standard_normal((n, d)) * 4)
    qs, ks, w = rng.uniform(0.5, 1.5, H), rng.uniform(0.5, 1.5, n), rng.uniform(0, 1, H)
    got = index_scores(qc, qs, w, kc, ks, n_visible=9)
    qv, kv = codecs.e4m3_decode(qc), codecs.e4m3_decode(kc)
    for i in range(n):
        if i >= 9:
            assert got[i] == -math.inf
            continue
        want = 0.0
        for h in range(H):
            dot = sum(float(qv[h, c]) * float(kv[i, c]) for c in range(d))
            want += w[h] * max(0.0, qs[h] * ks[i] * dot)
        assert abs(got[i] - want) <= 1e-12 * max(1.0, abs(want))


def test_index_scores_relu_zeroes_negative_heads():
    q = codecs.e4m3_encode(np.array([[1.0, 1.0], [-1.0, -1.0]]))
    k = codecs.e4m3_encode(np.array([[2.0, 2.0], [-2.0, -2.0]]))
    s = index_scores(q, [1.0, 1.0], [0.25, 0.75], k, [1.0, 1.0], n_visible=2)
    assert list(s) == [0.25 * 4.0, 0.75 * 4.0]


def _brute_topk(s, n_valid, k):
    order = sorted(range(n_valid), key=lambda i: (-s[i], i))
    chosen = sorted(order[:k])
    return chosen + [-1] * (k - len(chosen))


@pytest.mark.parametrize("seed", range(12))
def test_topk_brute_force_with_ties(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 65))
    k = int(rng.integers(1, 17))
    s = rng.integers(0, 5, size=n).astype(np.float64)            # forces many ties
    if seed % 3 == 0:
        s[:] = 2.0                                               # all equal
    n_valid = int(rng.integers(0, n + 1))
    assert list(topk(s, n_valid, k)) == _brute_topk(list(s), n_valid, k)


def test_topk_all_visible_is_identity_set():
    s = np.random.default_rng(9).standard_normal(40)
    assert list(topk(s, 40, 64)) == list(range(40)) + [-1] * 24


def _dense_attention(q, keys, m, rope_dim, scale):
    """Textbook softmax attention with K = V and a final R_m^-1, written with loops."""
    H, d = q.shape
    out = np.zeros((H, d))
    for h in range(H):
        logits = [scale * float(np.dot(q[h], kk)) for kk in keys]
        mx = max(logits)
        e = [math.exp(l - mx) for l in logits]
        tot = sum(e)
        o = sum((ei / tot) * kk for ei, kk in zip(e, keys))
        for j in range(rope_dim // 2):                            # explicit 2x2 inverse rotations
            a = -m * 10000.0 ** (-2 * j / rope_dim)
            i0 = d - rope_dim + 2 * j
            x0, x1 = o[i0], o[i0 + 1]
            o[i0], o[i0 + 1] = x0 * math.cos(a) - x1 * math.sin(a), x0 * math.sin(a) + x1 * math.cos(a)
        out[h] = o
    return out


def _layer_pools(x, z, kind, d, rope_dim, shift=0):
    """Pools and tables holding compressed entries and SWA rows of raw tokens x at positions shift + p."""
    T = x.shape[0]
    w, s = C.WINDOW[kind]
    # entries formed at shifted positions: entry i covers shift + s*i ... (shift is a multiple of 256)
    ent = C.compress_tokens(x, z, kind, rope_dim)
    ent = R.rope(R.rope(ent, [C.entry_position(i, kind) for i in range(len(ent))], rope_dim, inverse=True),
                 [shift + C.entry_position(i, kind) for i in range(len(ent))], rope_dim)
    epb = 256 // s
    nblk = (shift + T + 255) // 256
    main = Pool(epb, BF16, np.zeros((nblk * epb, d)))
    swa = Pool(256, BF16, np.zeros((nblk * 256, d)))
    perm = np.random.default_rng(11).permutation(nblk)
    table = perm[None, :]
    off = shift // s
    main.data[[perm[(off + i) // epb] * epb + (off + i) % epb for i in range(len(ent))]] = ent
    rows = R.rope(x, shift + np.arange(T), rope_dim)
    swa.data[[perm[(shift + p) // 256] * 256 + (shift + p) % 256 for p in range(T)]] = rows
    return main, swa, table, off


def test_dense_equivalence_when_k_covers_all_visible():
    rng = np.random.default_rng(12)
    d, r, T, H = 32, 8, 300, 4
    x, z = rng.standard_normal((T, d)), rng.standard_normal(T)
    main, swa, table, _ = _layer_pools(x, z, C.C4A, d, r)
    m = T - 1
    q = R.rope(rng.standard_normal((1, H, d)), m, r)
    n = visible_entries(m, C.C4A)
    ids = np.arange(n)[None, :]
    scale = 1 / math.sqrt(d)
    got, _ = sparse_attn(q, [m], [0], C.C4A, ids, main, table, swa, table, 128, scale, r)
    keys = list(main.read(table[0], np.arange(n))) + list(swa.read(table[0], window_positions(m)))
    assert np.allclose(got[0], _dense_attention(q[0], keys, m, r, scale), atol=1e-12)
    got_none, _ = sparse_attn(q, [m], [0], C.C4A, None, main, table, swa, table, 128, scale, r)
    assert np.allclose(got_none[0], got[0], atol=1e-14)


@pytest.mark.parametrize("kind", [C.C4A, C.C128A])
def test_translation_invariance_and_negative_control(kind):
    rng = np.random.default_rng(13)
    d, r, T, H = 64, 16, 700, 4
    x, z = rng.standard_normal((T, d)), rng.standard_normal(T)
    q_raw = rng.standard_normal((1, H, d))
    scale = 1 / math.sqrt(d)
    outs, raw = [], []
    for shift in (0, 256 * 37):
        main, swa, table, off = _layer_pools(x, z, kind, d, r, shift)
        m = shift + T - 1
        q = R.rope(q_raw, m, r)
        n = C.n_entries(T, kind)
        ids = (off + np.arange(n))[None, :]
        o, _ = sparse_attn(q, [m], [0], kind, ids, main, table, swa, table, 128, scale, r)
        outs.append(o[0])
        keys = np.concatenate([main.read(table[0], ids[0]), swa.read(table[0], window_positions(m))])
        raw.append(sparse_attention(q[0], keys, m, r, scale, inverse_rope=False)[0])
    assert np.max(np.abs(outs[0] - outs[1])) < 1e-9
    assert np.max(np.abs(raw[0] - raw[1])) > 1e-3                 # without R_m^-1 the output moves


def test_first_position_attends_only_itself():
    rng = np.random.default_rng(14)
    d, r = 32, 8
    x = rng.standard_normal((1, d))
    swa = Pool(256, BF16, np.zeros((256, d)))
    swa.data[0] = R.rope(x[0], 0, r)
    main = Pool(64, BF16, np.zeros((64, d)))
    q = rng.standard_normal((1, 3, d))
    out, lse = sparse_attn(q, [0], [0], C.C4A, np.full((1, 4), -1), main, np.array([[0]]),
                           swa, np.array([[0]]), 128, 0.1, r)
    assert np.allclose(out[0], np.broadcast_to(x[0], (3, d)), atol=1e-14)
    assert np.allclose(lse[0], 0.1 * (q[0] @ swa.data[0]))


def test_single_key_output_is_key_unrotated():
    rng = np.random.default_rng(15)
    k = rng.standard_normal(16)
    o, _ = sparse_attention(rng.standard_normal((2, 16)), R.rope(k, 900, 8)[None], 900, 8, 0.5)
    assert np.allclose(o, np.broadcast_to(k, (2, 16)), atol=1e-12)


# ---- fp8 output (inverse RoPE + fp8 quantisation, [P2] 融合点 2) -----------------------------------------
def test_quantize_output_blocks_are_independent_and_saturate_at_448():
    from oracle.attention import quantize_output
    from oracle.codecs import e4m3_decode
    rng = np.random.default_rng(9)
    o = rng.standard_normal((3, 512))
    o[0, 5] = 1000.0                                   # a large value in block 0 of head 0 only
    codes, scale = quantize_output(o)
    assert codes.shape == (3, 512) and scale.shape == (3, 4)
    # each block's scale is its own amax / 448 (fp32): the outlier does not touch blocks 1-3
    for h in range(3):
        for b in range(4):
            blk = o[h, 128 * b:128 * (b + 1)]
            assert scale[h, b] == np.float32(np.max(np.abs(blk)) / 448.0)
    # the block's largest magnitude maps to the largest code, +-448
    assert e4m3_decode(codes[0, 5:6])[0] == 448.0
    assert np.max(np.abs(e4m3_decode(codes[1, :128]))) == 448.0
    # dequantised within half an e4m3 step: relative 2^-4 for normals (absolute 2^-10 * scale below 2^-6)
    deq = e4m3_decode(codes).reshape(3, 4, 128) * scale[..., None]
    err = np.abs(deq.reshape(3, 512) - o)
    bound = np.maximum(np.abs(o) * 2.0 ** -4, np.repeat(scale, 128, axis=1) * 2.0 ** -10)
    assert np.all(err <= bound * (1 + 1e-9))


def test_quantize_output_zero_block_and_negative_zero():
    from oracle.attention import quantize_output
    o = np.zeros((1, 512))
    o[0, 128:] = 1.0
    o[0, 200] = -0.0
    o[0, 300] = -1e-30                                 # rounds to zero, keeps its sign
    codes, scale = quantize_output(o)
    assert scale[0, 0] == 1.0 and np.all(codes[0, :128] == 0)   # all-zero block: scale 1, codes +0
    assert codes[0, 300] == 0x80                                  # -0 code
    assert np.all(scale[0, 1:] == np.float32(1.0 / 448.0))


def test_sparse_attn_q8_is_the_quantised_sparse_attn():
    """The layer call's fp8 output equals quantize_output of the float64 output it returns beside it."""
    from oracle import layer as OL
    from oracle.attention import quantize_output
    rng = np.random.default_rng(3)
    epb = 64
    main = OL.Pool(epb, OL.BF16, rng.standard_normal((4 * epb, 512)))
    swa = OL.Pool(256, OL.BF16, rng.standard_normal((2 * 256, 512)))
    bt = np.array([[2, 0, 3, 1]])
    sbt = np.array([[1, 0]])
    q = rng.standard_normal((1, 8, 512))
    topk = np.array([[3, 7, 11, -1]])
    q8, lse, out = OL.sparse_attn_q8(q, [300], [0], "c4a", topk, main, bt, swa, sbt, 128, 512 ** -0.5, 64)
    codes, scales = q8[0]
    want_c, want_s = quantize_output(out[0])
    assert np.array_equal(codes, want_c) and np.array_equal(scales, want_s)


# ---- query prep ([P2] 融合点 3: the Q-norm beside the key RoPE and insert) ----------------------------------

def test_query_prep_brute_force():
    """Per head: divide by sqrt(mean(q^2) + eps), then rotate each pair of the last rope_dim dims by m * f_j,
    written with scalar loops on a tiny case."""
    import math
    from oracle.attention import query_prep
    from oracle.rope import inv_freq
    rng = np.random.default_rng(31)
    q = rng.standard_normal((2, 8))
    m, rd, eps = 37, 4, 1e-6
    f = inv_freq(rd)
    want = np.zeros_like(q)
    for h in range(2):
        ms = sum(float(x) * float(x) for x in q[h]) / 8
        v = [float(x) / math.sqrt(ms + eps) for x in q[h]]
        for j in range(rd // 2):
            a = m * f[j]
            i0 = 8 - rd + 2 * j
            x0, x1 = v[i0], v[i0 + 1]
            v[i0], v[i0 + 1] = x0 * math.cos(a) - x1 * math.sin(a), x0 * math.sin(a) + x1 * math.cos(a)
        want[h] = v
    assert np.allclose(query_prep(q, m, rd), want, rtol=1e-12, atol=1e-13)


def test_query_prep_norm_scale_invariance_and_gamma():
    from oracle.attention import query_prep
    rng = np.random.default_rng(32)
    q = rng.standard_normal((64, 512)) * 3.0
    out = query_prep(q, 1000, 64, eps=0.0)
    assert np.allclose(np.sqrt(np.mean(out * out, axis=-1)), 1.0, atol=1e-12)     # the rotation keeps the RMS
    assert np.allclose(query_prep(7.5 * q, 1000, 64, eps=0.0), out, atol=1e-12)   # a scale drops out
    assert np.allclose(query_prep(q, 1000, 64, gamma=np.full(512, 2.0), eps=0.0), 2.0 * out, atol=1e-12)


def test_query_prep_scores_depend_on_relative_position():
    """<query_prep(q, m), R_n k> depends on m - n only (the query is rotated at its own position)."""
    from oracle.attention import query_prep
    from oracle.rope import rope
    rng = np.random.default_rng(33)
    q = rng.standard_normal((4, 64))
    k = rng.standard_normal(64)
    s1 = query_prep(q, 500, 32) @ rope(k, 480, 32)
    s2 = query_prep(q, 90500, 32) @ rope(k, 90480, 32)
    s3 = query_prep(q, 500, 32) @ rope(k, 470, 32)
    assert np.allclose(s1, s2, atol=1e-9)
    assert not np.allclose(s1, s3, atol=1e-3)                                     # negative control
