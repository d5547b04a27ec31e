"""CPU pins of the parity helpers that judge e4m3 rows: a correct rounding passes, a wrong code or scale
fails, and a value on a rounding midpoint accepts either neighbour (the only latitude the check gives)."""
import numpy as np

from oracle.codecs import fp8_quantize_rows, e4m3_decode, e4m3_encode
import torch

from _parity import fp8_row_violations, e4m3_half_spacing, check_rows, pool_absmax, attn_bound, assert_attn_close


def test_half_spacing_matches_the_grid():
    grid = np.sort(e4m3_decode(np.arange(0x7F, dtype=np.uint8)))
    for lo, hi in zip(grid[:-1], grid[1:]):
        mid = 0.5 * (lo + hi)
        # just inside the upper cell: its half spacing is the distance to the lower midpoint or more
        assert e4m3_half_spacing(np.nextafter(hi, 0.0)) >= (hi - lo) / 2 - 1e-15
        assert e4m3_half_spacing(mid) * 2 >= (hi - lo) - 1e-15


def test_correct_rounding_passes_and_wrong_codes_fail():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((40, 128)) * np.exp(rng.uniform(-3, 3, (40, 1)))
    codes, scale = fp8_quantize_rows(v)
    bad_el, bad_rows = fp8_row_violations(codes, scale, v)
    assert len(bad_el) == 0 and len(bad_rows) == 0
    # one code moved to its neighbour away from any midpoint: caught
    wrong = codes.copy()
    u = v / scale[:, None]
    j = np.argmin(np.abs(np.abs(u[0]) - 100.0))          # a mid-cell value near 100
    wrong[0, j] = wrong[0, j] + 1 if (wrong[0, j] & 0x7F) < 0x7E else wrong[0, j] - 1
    bad_el, _ = fp8_row_violations(wrong, scale, v)
    assert [tuple(x) for x in bad_el] == [(0, j)]
    # a wrong sign: caught
    wrong = codes.copy()
    k = int(np.argmax(np.abs(u[1])))
    wrong[1, k] ^= 0x80
    bad_el, _ = fp8_row_violations(wrong, scale, v)
    assert (1, k) in [tuple(x) for x in bad_el]
    # a scale off by 1e-3: the row is reported
    _, bad_rows = fp8_row_violations(codes, scale * (1 + 1e-3), v)
    assert len(bad_rows) == len(v)


def test_midpoint_accepts_either_neighbour():
    scale = np.array([1.0])
    for lo_code in (0x40, 0x48, 0x5A, 0x05):          # normals of several binades and a subnormal
        lo, hi = e4m3_decode(np.array([lo_code, lo_code + 1], dtype=np.uint8))
        mid = 0.5 * (lo + hi)
        v = np.full((1, 4), mid)
        v[0, 1:] = [1.0, 2.0, 448.0]                  # amax = 448 keeps the scale at 1
        for c in (lo_code, lo_code + 1):
            codes = e4m3_encode(v)
            codes[0, 0] = c
            bad_el, bad_rows = fp8_row_violations(codes, scale, v)
            assert len(bad_el) == 0 and len(bad_rows) == 0, (lo_code, c)
        codes = e4m3_encode(v)
        codes[0, 0] = lo_code + 2                     # two cells away: rejected
        assert len(fp8_row_violations(codes, scale, v)[0]) == 1


def test_check_rows_is_per_row():
    rng = np.random.default_rng(5)
    want = rng.standard_normal((50, 64))
    got = want.copy()
    got[17] *= 1.05                                   # one row 5% off: the whole-case norm would hide it
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 1e-2
    try:
        check_rows(got, want)
    except AssertionError as e:
        assert e.args[0][1] == 17
    else:
        raise AssertionError("a 5% row error passed the per-row check")


def test_pool_absmax_equals_the_decoded_maximum():
    """e4m3 magnitudes grow with a code's low 7 bits, so the largest low-7-bit code of a row decodes to the
    row's largest magnitude; checked against decoding every code."""
    mags = np.abs(e4m3_decode(np.arange(0x7F, dtype=np.uint8)))
    assert np.all(np.diff(mags) > 0)
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 256, (50, 64), dtype=np.uint8)
    codes[codes & 0x7F == 0x7F] = 0x10                      # no NaN codes in a pool
    scale = rng.uniform(0.5, 1.5, 50)
    want = float(np.max(np.abs(e4m3_decode(codes) * scale[:, None])))
    assert pool_absmax((torch.from_numpy(codes), torch.from_numpy(scale))) == want
    bf = torch.from_numpy(rng.standard_normal((30, 8))).to(torch.bfloat16)
    assert pool_absmax((bf, None), (torch.from_numpy(codes), torch.from_numpy(scale))) == max(
        want, float(bf.float().abs().max()))


def test_attention_bound_catches_a_wrong_weight():
    """An output off by one key's weight error of a few percent fails the element bound; rounding-sized
    perturbations of the weights pass."""
    rng = np.random.default_rng(6)
    v = rng.standard_normal((640, 512))
    p = rng.uniform(0, 1, 640)
    w = p / p.sum()
    o = w @ v
    vmax = np.abs(v).max()
    wr = p * (1 + rng.uniform(-2.0 ** -9, 2.0 ** -9, 640))
    assert_attn_close(wr / wr.sum() @ v, o, vmax)            # bf16-sized weight errors pass
    bad = p.copy()
    bad[int(np.argmax(p))] *= 1.5                            # one key's weight wrong by half
    try:
        assert_attn_close(bad / bad.sum() @ v, o, vmax)
    except AssertionError:
        pass
    else:
        raise AssertionError("a wrong weight passed the attention bound")
    assert np.all(attn_bound(o, vmax) > 0)
