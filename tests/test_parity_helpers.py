"""CPU pins of the parity helpers that judge e4m3 rows: a correct rounding passes, a wrong code or scale
fails, and a value on a rounding midpoint accepts either neighbour (the only latitude the check gives)."""
import numpy as np

from oracle.codecs import fp8_quantize_rows, e4m3_decode, e4m3_encode
from _parity import fp8_row_violations, e4m3_half_spacing, check_rows


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
