"""Pins of the oracle's codecs and RoPE against the OCP OFP8 table, torch's library
conversions, closed forms and the rotation-group identities of the inverse-RoPE derivation."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import codecs, rope as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if line:
            rows.append(line.split())
    return rows


def test_e4m3_golden_ocp_table():
    for val, code in _golden_rows("e4m3_ocp.txt"):
        v, c = float(val), int(code, 16)
        assert int(codecs.e4m3_encode(np.array([v]))[0]) == c, val
        assert codecs.e4m3_decode(np.array([c], dtype=np.uint8))[0] == v, code


def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = codecs.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2                                   # S.1111.111 only
    assert np.array_equal(ours[~nan], lib[~nan])


def test_e4m3_encode_matches_torch_rne():
    g = torch.Generator().manual_seed(5)
    x = torch.cat([torch.randn(200000, generator=g) * s for s in (0.003, 0.1, 1.0, 30.0, 120.0)])
    x = torch.clamp(x, -448.0, 448.0)
    lib = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = codecs.e4m3_encode(x.double().numpy())
    assert np.array_equal(ours, lib)


def test_e4m3_round_half_even_and_saturation():
    # 1.0625 lies half-way between 1.0 (M=0) and 1.125 (M=1): the even mantissa wins
    assert codecs.e4m3_round(np.array([1.0625]))[0] == 1.0
    assert codecs.e4m3_round(np.array([1.1875]))[0] == 1.25
    # subnormal midpoint 1.5 * 2^-9 -> 2 * 2^-9
    assert codecs.e4m3_round(np.array([1.5 * 2 ** -9]))[0] == 2 * 2 ** -9
    # saturating conversion: beyond the largest finite value stays at +-448
    assert list(codecs.e4m3_round(np.array([460.0, 500.0, -1e6]))) == [448.0, 448.0, -448.0]


def test_e4m3_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    back = codecs.e4m3_encode(codecs.e4m3_decode(codes))
    assert np.array_equal(back, codes)


def test_bf16_round_matches_torch():
    g = torch.Generator().manual_seed(6)
    x = torch.randn(300000, generator=g, dtype=torch.float32) * 7.0
    lib = x.to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(codecs.bf16_round(x.double().numpy()), lib)
    # tie: 1 + 2^-8 is half-way between 1 and 1 + 2^-7 -> even significand (1.0)
    assert codecs.bf16_round(np.array([1.0 + 2 ** -8]))[0] == 1.0
    assert codecs.bf16_round(np.array([1.0 + 3 * 2 ** -8]))[0] == 1.0 + 2 ** -6


def test_bf16_bits_codec_matches_torch():
    g = torch.Generator().manual_seed(8)
    x = torch.randn(100000, generator=g, dtype=torch.float32) * 3.0
    bits = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(codecs.bf16_decode(bits), x.to(torch.bfloat16).double().numpy())
    assert np.array_equal(codecs.bf16_encode(x.double().numpy()), bits)


def test_fp8_row_quantisation():
    v = np.array([[0.5, -3.0, 1.25, 0.0], [0.0, 0.0, 0.0, 0.0]])
    codes, scale = codecs.fp8_quantize_rows(v)
    assert scale[0] == np.float32(3.0 / 448.0) and scale[1] == 1.0
    assert codes[0, 1] == 0xFE                              # the amax element maps to -448
    assert np.all(codes[1] == 0)
    back = codecs.fp8_dequantize_rows(codes, scale)
    assert np.max(np.abs(back[0] - v[0])) <= 3.0 / 16       # e4m3 keeps 4 significant bits


def test_rope_inv_freq_closed_form():
    f = R.inv_freq(64, 10000.0)
    assert f[0] == 1.0
    assert abs(f[1] / 10000.0 ** (-2 / 64) - 1) < 1e-15
    assert abs(f[31] / 10000.0 ** (-62 / 64) - 1) < 1e-15


def test_rope_rotates_interleaved_pairs_of_last_dims():
    d, r, p = 16, 8, 3.0
    for j in range(r // 2):
        e = np.zeros(d)
        e[d - r + 2 * j] = 1.0
        out = R.rope(e, p, r)
        ang = p * 10000.0 ** (-2 * j / r)
        want = np.zeros(d)
        want[d - r + 2 * j] = math.cos(ang)
        want[d - r + 2 * j + 1] = math.sin(ang)
        assert np.allclose(out, want, atol=1e-15)
    v = np.arange(d, dtype=np.float64)
    assert np.array_equal(R.rope(v, 7, r)[: d - r], v[: d - r])   # no RoPE on the first d - r dims


def test_rope_group_identities():
    rng = np.random.default_rng(0)
    v = rng.standard_normal((5, 512))
    a, b = 1234, 98765
    assert np.allclose(R.rope(R.rope(v, a, 64), a, 64, inverse=True), v, atol=1e-12)
    assert np.allclose(R.rope(R.rope(v, a, 64), b, 64), R.rope(v, a + b, 64), atol=1e-9)
    assert np.allclose(np.linalg.norm(R.rope(v, b, 64), axis=1), np.linalg.norm(v, axis=1))
    # R_m^T R_n = R_(n-m): the score depends on relative position only
    q, k = v[0], v[1]
    s1 = R.rope(q, 500, 64) @ R.rope(k, 300, 64)
    s2 = R.rope(q, 500 + 777, 64) @ R.rope(k, 300 + 777, 64)
    assert abs(s1 - s2) < 1e-10


# ---- fp4 e2m1 (the fp4 indexer cache) --------------------------------------------------------------------
def _e2m1_golden():
    rows = []
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "e2m1_ocp.txt")):
        if line.strip() and not line.startswith("#"):
            c, v = line.split()
            rows.append((int(c), float(v)))
    return rows


def test_e2m1_decode_matches_the_ocp_table():
    from oracle.codecs import e2m1_decode
    g = _e2m1_golden()
    assert len(g) == 16
    for c, v in g:
        got = e2m1_decode(np.array([c]))[0]
        assert got == v and np.signbit(got) == np.signbit(v), (c, got, v)


def test_e2m1_round_trip_midpoints_and_saturation():
    from oracle.codecs import e2m1_decode, e2m1_encode, e2m1_round
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(e2m1_encode(e2m1_decode(codes)), codes)                 # every code (with -0)
    # ties to even: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -5.0, -0.25])
    assert list(e2m1_round(x)) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, -4.0, -0.0]
    # just off the midpoints: nearest
    eps = 1e-9
    assert list(e2m1_round(np.array([0.25 + eps, 2.5 + eps, 5.0 - eps]))) == [0.5, 3.0, 4.0]
    # saturation to +-6 and the sign of a negative zero
    assert list(e2m1_round(np.array([6.9, 1e9, -7.0]))) == [6.0, 6.0, -6.0]
    assert e2m1_encode(np.array([-1e-9]))[0] == 0x8


def test_fp4_pack_order_and_row_quantisation():
    from oracle.codecs import fp4_pack, fp4_unpack, fp4_quantize_rows, fp4_dequantize_rows, e2m1_decode
    c = np.array([[1, 2, 3, 15]], dtype=np.uint8)
    p = fp4_pack(c)
    assert list(p[0]) == [0x21, 0xF3]                       # element 2j in the low nibble
    assert np.array_equal(fp4_unpack(p), c)
    rng = np.random.default_rng(4)
    v = rng.standard_normal((20, 128)) * np.exp(rng.uniform(-2, 2, (20, 1)))
    packed, scale = fp4_quantize_rows(v)
    assert packed.shape == (20, 64)
    assert np.all(scale == (np.max(np.abs(v), axis=1) / 6.0).astype(np.float32))
    deq = fp4_dequantize_rows(packed, scale)
    # the largest magnitude of each row maps to +-6; every element within half a step of the e2m1 grid
    assert np.all(np.max(np.abs(e2m1_decode(fp4_unpack(packed))), axis=1) == 6.0)
    u = np.abs(v / scale[:, None])
    half = np.where(u < 2, 0.25, np.where(u < 4, 0.5, 1.0))
    assert np.all(np.abs(deq / scale[:, None] - v / scale[:, None]) <= half + 1e-12)


def test_index_scores_with_fp4_keys_brute_force():
    """The indexer score with e2m1 keys: a brute-force loop over heads and dims of the decoded values."""
    from oracle.indexer import index_scores
    from oracle.codecs import e2m1_decode, e4m3_decode
    rng = np.random.default_rng(6)
    H, d, n = 4, 32, 9
    qc = rng.integers(0, 0x7F, (H, d)).astype(np.uint8)
    kc = rng.integers(0, 16, (n, d)).astype(np.uint8)
    qs, ks, w = rng.uniform(0.1, 1, H), rng.uniform(0.1, 1, n), rng.uniform(0, 1, H)
    got = index_scores(qc, qs, w, kc, ks, 7, key_format="e2m1")
    for i in range(n):
        want = -np.inf
        if i < 7:
            want = 0.0
            for h in range(H):
                dot = sum(e4m3_decode(qc[h, c]) * e2m1_decode(kc[i, c]) for c in range(d))
                want += w[h] * max(0.0, qs[h] * ks[i] * dot)
        assert (got[i] == want) if i >= 7 else abs(got[i] - want) <= 1e-12 * max(1.0, abs(want)), i
