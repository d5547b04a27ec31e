"""Parity helpers: feed the oracle the same seeded bytes the CUDA path used, compare with the
stated tolerances.

Tolerances (fixed in the tests that use them):
  * indices, gathers, rolling state: bit-exact;
  * top-k sets: identical except elements whose oracle score lies within 1e-3 relative of the
    oracle's k-th score;
  * attention outputs: max abs <= 2e-2 and rel-L2 <= 1e-2 (bf16 / fp8 data);
  * compressor rows and indexer scores: rel-L2 <= 1e-2.
"""
import numpy as np
import torch

from oracle import layer as OL, compress as OC
from oracle.codecs import fp8_dequantize_rows

ATTN_MAX_ABS = 2e-2
ATTN_REL_L2 = 1e-2
ROW_REL_L2 = 1e-2
TOPK_TIE_REL = 1e-3


def np64(t):
    """A torch tensor (any device) as numpy: bf16/fp32 -> float64, integers unchanged."""
    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16, torch.float32, torch.float64):
        return t.to(torch.float64).numpy()
    return t.numpy()


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def to_device(case, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in case.items()}


def oracle_pool(data, scale, epb):
    """An oracle Pool over (copies of) a case's pool tensors."""
    if data.dtype == torch.bfloat16:
        return OL.Pool(epb, OL.BF16, data.detach().cpu().view(torch.int16).numpy().view(np.uint16).copy())
    return OL.Pool(epb, OL.FP8, data.detach().cpu().numpy().copy(), np64(scale).copy())


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


def pool_rows(data, scale, rows):
    """Decoded float64 rows of a (device) pool at physical row ids."""
    d = data.detach().cpu()
    if d.dtype == torch.bfloat16:
        return np64(d[rows])
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
