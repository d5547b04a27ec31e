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
