"""Parity helpers: feed the oracle the same seeded bytes the CUDA path used, compare with the
stated tolerances.

Tolerances (fixed in the tests that use them):
  * indices, gathers, rolling state: bit-exact;
  * top-k sets: identical except elements whose oracle score lies within 1e-3 relative of the
    oracle's k-th score;
  * attention outputs: element-wise within 2^-6.5 * vmax + 2^-9 * |o| (vmax: the largest |value| of the key
    pools), and rel-L2 <= 1e-2 over a case (bf16 / fp8 data).  The kernel rounds each probability to bf16
    (relative error <= u = 2^-9) before P V and divides by the sum of those rounded probabilities, so the
    output is a convex combination of key rows whose weights are perturbed by at most 2u relative: the
    error is <= 2u * max_j |v_j - o| <= 4u * vmax per dimension; the inverse rotation mixes a pair of dims
    (a factor sqrt 2), and the bf16 store adds half an ulp, <= u * |o|;
  * compressor rows and indexer scores: rel-L2 <= 1e-2, for every row (entry, or query's score row);
  * e4m3 rows (fp8 pools): an e4m3 code decides an integer from a float, so each code is checked as a
    correct round-to-nearest of the oracle's float64 value divided by the row scale (up to a relative
    slack of 1e-4 of that value: the GPU's fp32 value may sit on the other side of a rounding midpoint),
    and the row scale as amax/448 within 1e-5 relative;
  * e2m1 rows (fp4 indexer pools): the same, on the e2m1 grid, with the row scale amax/6.
"""
import numpy as np
import torch

from oracle import layer as OL, compress as OC
from oracle.codecs import (fp8_dequantize_rows, fp8_row_scale, e4m3_decode, fp4_dequantize_rows, fp4_row_scale,
                           fp4_unpack, e2m1_decode)

ATTN_REL_L2 = 1e-2
ROW_REL_L2 = 1e-2
TOPK_TIE_REL = 1e-3


def np64(t):
    """A torch tensor (any device) as numpy: bf16/fp32 -> float64, integers unchanged."""
    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16, torch.float32, torch.float64):
        return t.to(torch.float64).numpy()
    return t.numpy()


def attn_bound(W, vmax):
    """Element-wise bound on |kernel - oracle| for an attention output W (module docstring)."""
    return 2.0 ** -6.5 * vmax + 2.0 ** -9 * np.abs(W)


def assert_attn_close(got, W, vmax):
    """Attention output within attn_bound element by element and within ATTN_REL_L2 overall."""
    err = np.abs(np.asarray(got, np.float64) - W)
    excess = err - attn_bound(W, vmax)
    worst = np.unravel_index(int(np.argmax(excess)), excess.shape)
    assert excess[worst] <= 0.0, ("attention element", worst, float(err[worst]), float(attn_bound(W, vmax)[worst]))
    e = rel_l2(got, W)
    assert e <= ATTN_REL_L2, ("attention rel-L2", e)


def pool_absmax(*pools):
    """Largest |value| over key pools given as (data, scale) device tensors: bf16 rows (scale None) or e4m3
    codes with a scale per row.  e4m3 magnitudes grow with the code's low 7 bits, so each row's largest
    magnitude is the decode of its largest low-7-bit code."""
    m = 0.0
    for data, scale in pools:
        if data.dtype == torch.bfloat16:
            m = max(m, float(data.detach().abs().max().float()))
        else:
            top = (data.detach() & 0x7F).amax(dim=-1).cpu().numpy()
            m = max(m, float(np.max(e4m3_decode(top) * np.abs(np64(scale)))))
    return m


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def to_device(case, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in case.items()}


def oracle_pool(data, scale, epb, fmt=None):
    """An oracle Pool over (copies of) a case's pool tensors (fmt "fp4": packed e2m1 bytes)."""
    if fmt == "fp4":
        return OL.Pool(epb, OL.FP4, data.detach().cpu().numpy().copy(), np64(scale).copy())
    if data.dtype == torch.bfloat16:
        return OL.Pool(epb, OL.BF16, data.detach().cpu().view(torch.int16).numpy().view(np.uint16).copy())
    return OL.Pool(epb, OL.FP8, data.detach().cpu().numpy().copy(), np64(scale).copy())


def idx_pool(case):
    """The oracle Pool over a case's indexer key pool."""
    return oracle_pool(case["idx_data"], case["idx_scale"], 64, case["spec"].idx_dtype)


def rolling_states(case, which="main"):
    """Oracle RollingStates from a case's state ring (slot = position mod w)."""
    spec = case["spec"]
    xs = np64(case["state_x" if which == "main" else "state_xi"])
    zs = np64(case["state_z" if which == "main" else "state_zi"])
    slots = np64(case["state_slot"])
    return [OC.RollingState(spec.kind, xs.shape[-1], xs[slots[r]], zs[slots[r]]) for r in range(spec.batch)]


def new_tokens(case, which="main"):
    cu = np64(case["cu_new"])
    x = np64(case["x_new" if which == "main" else "xi_new"])
    z = np64(case["z_new" if which == "main" else "zi_new"])
    return [x[cu[r]:cu[r + 1]] for r in range(len(cu) - 1)], [z[cu[r]:cu[r + 1]] for r in range(len(cu) - 1)]


def pool_rows(data, scale, rows, fmt=None):
    """Decoded float64 rows of a (device) pool at physical row ids."""
    d = data.detach().cpu()
    if d.dtype == torch.bfloat16:
        return np64(d[rows])
    if fmt == "fp4":
        return fp4_dequantize_rows(d[rows].numpy(), np64(scale.detach().cpu()[rows]))
    return fp8_dequantize_rows(d[rows].numpy(), np64(scale.detach().cpu()[rows]))


def topk_sets_match(gpu_idx, oracle_scores, n_valid, k):
    """Top-k set equality with the near-tie exemption; returns (ok, n_differing)."""
    want = set(int(i) for i in OL.topk(oracle_scores, n_valid, k) if i >= 0)
    got = set(int(i) for i in gpu_idx if i >= 0)
    if got == want:
        return True, 0
    s = np.asarray(oracle_scores[:n_valid], np.float64)
    kth = np.sort(s)[::-1][min(k, n_valid) - 1]
    tol = TOPK_TIE_REL * max(abs(kth), 1e-30)
    diff = got ^ want
    ok = all(abs(s[i] - kth) <= tol for i in diff if 0 <= i < n_valid) and len(got) == len(want)
    return ok, len(diff)


FP8_VALUE_SLACK = 1e-4
FP8_SCALE_REL = 1e-5


def e4m3_half_spacing(a):
    """Half the e4m3 grid spacing at magnitude a: subnormals 2^-10, normals 2^(floor(log2 a) - 4)."""
    a = np.asarray(a, np.float64)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return np.where(a < 2.0 ** -6, 2.0 ** -10, 2.0 ** (e - 4))


def fp8_row_violations(codes, scale, values, value_slack=FP8_VALUE_SLACK, scale_rel=FP8_SCALE_REL):
    """Elements of e4m3 rows (codes uint8 [n][d], fp32 scale [n]) that are not a correct rounding of the
    float64 values [n][d] / scale (up to a relative slack of the value); and rows whose scale is not amax/448
    within scale_rel.  Returns (bad_elements, bad_rows)."""
    FP8_VALUE_SLACK_ = value_slack
    codes = np.asarray(codes, np.uint8)
    scale = np.asarray(scale, np.float64)
    values = np.asarray(values, np.float64)
    want_scale = fp8_row_scale(values)
    bad_rows = np.nonzero(np.abs(scale - want_scale) > scale_rel * want_scale)[0]
    u = values / scale[:, None]
    dec = e4m3_decode(codes)
    a = np.abs(u)
    sat = a >= 448.0
    err = np.abs(dec - u)
    ok = err <= e4m3_half_spacing(np.minimum(a, 448.0)) + FP8_VALUE_SLACK_ * a + 1e-12
    ok = np.where(sat, np.abs(dec) == 448.0, ok) & ((dec == 0) | (np.sign(dec) == np.sign(u)) | (a < 2.0 ** -10))
    return np.argwhere(~ok), bad_rows


FP4_VALUE_SLACK = 1e-4
FP4_SCALE_REL = 1e-5


def e2m1_half_spacing(a):
    """Half the e2m1 grid spacing of the cell holding magnitude a: 0.25 below 2, 0.5 in [2, 4), 1 from 4."""
    a = np.asarray(a, np.float64)
    return np.where(a < 2.0, 0.25, np.where(a < 4.0, 0.5, 1.0))


def fp4_row_violations(packed, scale, values, value_slack=FP4_VALUE_SLACK, scale_rel=FP4_SCALE_REL):
    """Elements of packed e2m1 rows (uint8 [n][d / 2], fp32 scale [n]) that are not a correct rounding of
    the float64 values [n][d] / scale (up to a relative slack of the value); and rows whose scale is not
    amax/6 within scale_rel.  Returns (bad_elements, bad_rows), element indices in unpacked order."""
    codes = fp4_unpack(np.asarray(packed, np.uint8))
    scale = np.asarray(scale, np.float64)
    values = np.asarray(values, np.float64)
    want_scale = fp4_row_scale(values)
    bad_rows = np.nonzero(np.abs(scale - want_scale) > scale_rel * want_scale)[0]
    u = values / scale[:, None]
    dec = e2m1_decode(codes)
    a = np.abs(u)
    err = np.abs(dec - u)
    ok = err <= e2m1_half_spacing(np.minimum(a, 6.0)) + value_slack * a + 1e-12
    ok = np.where(a >= 6.0, np.abs(dec) == 6.0, ok) & ((dec == 0) | (np.sign(dec) == np.sign(u)))
    return np.argwhere(~ok), bad_rows


def check_rows(got, want, tol=ROW_REL_L2, what="row"):
    """Per-row rel-L2 of float64 rows [n][d]; returns the worst (rel-L2, max abs)."""
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    worst, mabs = 0.0, 0.0
    for j in range(len(got)):
        e = rel_l2(got[j], want[j])
        assert e <= tol, (what, j, e)
        worst = max(worst, e)
        if got[j].size:
            mabs = max(mabs, float(np.max(np.abs(got[j] - want[j]))))
    return worst, mabs


def check_pool_rows(gdata, gscale, prows, values, stored, fmt=None):
    """GPU pool rows (physical ids) against the oracle: bf16 rows per-row rel-L2 against the oracle's stored
    (rounded) rows; e4m3 and e2m1 rows code by code against the oracle's float64 values before rounding."""
    if gdata.dtype == torch.bfloat16:
        return check_rows(pool_rows(gdata, gscale, prows), stored)
    d = gdata.detach().cpu()
    codes = d[prows].numpy()
    scale = np64(gscale.detach().cpu()[prows])
    if fmt == "fp4":
        bad_el, bad_rows = fp4_row_violations(codes, scale, values)
        assert len(bad_rows) == 0, ("e2m1 row scale", bad_rows[:8])
        assert len(bad_el) == 0, ("e2m1 code", bad_el[:8])
        # each element is already bounded by half its grid cell; the row error is reported, not re-bounded
        return check_rows(fp4_dequantize_rows(codes, scale), np.asarray(values), tol=np.inf, what="e2m1 row")
    bad_el, bad_rows = fp8_row_violations(codes, scale, values)
    assert len(bad_rows) == 0, ("e4m3 row scale", bad_rows[:8])
    assert len(bad_el) == 0, ("e4m3 code", bad_el[:8])
    deq = fp8_dequantize_rows(codes, scale)
    return check_rows(deq, np.asarray(values), tol=2.0 ** -4, what="e4m3 row within the format's bound")
