"""The C-ABI library builds, loads and exports every entry point that include/dsa.h declares;
host-side validation rejects bad arguments before anything reaches the GPU (no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from compressed_sparse_attention_c4a_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def _declared():
    text = open(os.path.join(ROOT, "include", "dsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n


def test_binding_exposes_the_same_names(lib):
    from compressed_sparse_attention_c4a_gb300 import dsa
    for n in _declared():
        assert callable(getattr(dsa, n)), n


def test_status_strings(lib):
    lib.dsa_status_string.restype = ctypes.c_char_p
    assert lib.dsa_status_string(0) == b"ok"
    assert b"device" in lib.dsa_status_string(4)
    assert lib.dsa_status_string(99) == b"unknown status"


def test_host_validation_rejects_before_launch(lib):
    P = ctypes.c_void_p
    # top-k: k outside 1..2048, ld not a multiple of 4
    lib.dsa_topk.argtypes = [ctypes.c_int32, P, ctypes.c_int32, P, ctypes.c_int32, P, P, P]
    assert lib.dsa_topk(4, P(16), 64, P(16), 0, P(16), None, None) == 1
    assert lib.dsa_topk(4, P(16), 66, P(16), 8, P(16), None, None) == 1
    assert lib.dsa_topk(0, None, 64, None, 8, None, None, None) == 0          # empty: a no-op
    # indexer: unsupported head count / dim
    lib.dsa_index_scores.argtypes = [ctypes.c_int32] * 3 + [P] * 5 + [ctypes.c_int32, P, P, P, ctypes.c_int32, P, P,
                                                                       P, P, P]
    assert lib.dsa_index_scores(1, 5, 128, *[P(16)] * 5, 1, P(16), P(16), P(16), 64, None, None, None, None, None) == 2
    assert lib.dsa_index_scores(1, 8, 96, *[P(16)] * 5, 1, P(16), P(16), P(16), 64, None, None, None, None, None) == 2
    # compress: bad kind, null pointers
    lib.dsa_compress.restype = ctypes.c_int32
    args = [ctypes.c_int32(7), ctypes.c_int32(1)] + [None] * 18
    assert lib.dsa_compress(*args) == 1
    args = [ctypes.c_int32(0), ctypes.c_int32(1), None, None, ctypes.c_int32(1)] + [None] * 15
    assert lib.dsa_compress(*args) == 1


def test_fused_topk_attention_host_validation(lib):
    """dsa_topk_sparse_attn_decode: the top-k output buffer is required, ld a multiple of 4, k in 1..2048, an
    empty batch a no-op; all decided on the host."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    P = ctypes.c_void_p
    bt = dsa.DsaBlockTable(64, 4, 4)
    main = dsa.DsaPool(256, None, 16, 64, 512, dsa.DSA_BF16)
    rope = dsa.DsaRope(64, 10000.0)
    f = dsa._lib.dsa_topk_sparse_attn_decode

    def call(batch=4, ld=64, k=8, topk_out=P(16), scores=P(16)):
        return f(batch, 64, P(16), P(16), 0, scores, ld, P(16), k, topk_out, ctypes.byref(main), ctypes.byref(bt),
                 ctypes.byref(main), ctypes.byref(bt), 128, 0.044, ctypes.byref(rope), P(16), None, None, 0, None,
                 None)
    assert call(topk_out=None) == dsa.DSA_ERR_INVALID_ARG
    assert call(ld=66) == dsa.DSA_ERR_INVALID_ARG
    assert call(k=0) == dsa.DSA_ERR_INVALID_ARG
    assert call(scores=P(20)) == dsa.DSA_ERR_INVALID_ARG        # scores not 16-byte aligned
    assert call(batch=0) == dsa.DSA_OK


def test_workspace_size_is_zero_for_unsupported_heads(lib):
    lib.dsa_attn_workspace_size.restype = ctypes.c_size_t
    assert lib.dsa_attn_workspace_size(32, 48, 640) == 0
    assert lib.dsa_attn_workspace_size(0, 64, 640) == 0


def test_attention_plan_host_only(lib):
    """The split plan is host arithmetic: valid without a GPU (the SM count falls back to a default)."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    hg, cl, ns, launches = dsa.dsa_attn_plan(32, 64, 640, "bf16")
    assert hg == 64 and cl in (1, 2, 4) and ns >= 1 and launches == (2 if ns > 1 else 1)
    hg, cl, ns, launches = dsa.dsa_attn_plan(4, 128, 8320, "bf16")
    assert hg == 64 and cl == 4 and ns > 1 and launches == 2
    assert dsa.dsa_attn_plan(8192, 64, 640, "bf16")[1:3] == (1, 1)        # many rows: one CTA per row
    P = ctypes.c_void_p
    lib.dsa_attn_plan.argtypes = [ctypes.c_int32] * 4 + [P]
    plan = (ctypes.c_int32 * 4)()
    assert lib.dsa_attn_plan(0, 64, 640, 0, plan) == 1
    assert lib.dsa_attn_plan(4, 48, 640, 0, plan) == 2
    assert lib.dsa_attn_plan(4, 64, 640, 7, plan) == 1


def test_topk_plan_host_only(lib):
    """The top-k dispatch is host arithmetic: valid without a GPU (the SM count falls back to a default of
    148, so 296 cluster CTAs are resident at once)."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    assert dsa.dsa_topk_plan(32, 16384, 512) == (0, 4, 512)       # few short rows: a 4-CTA cluster each
    assert dsa.dsa_topk_plan(100, 16384, 512) == (0, 1, 1024)     # many short rows: one CTA each
    assert dsa.dsa_topk_plan(200, 34816, 512) == (1, 1, 512)      # many long rows: one CTA per row
    assert dsa.dsa_topk_plan(120, 34816, 512) == (1, 2, 512)      # fewer rows: spread over two SMs
    assert dsa.dsa_topk_plan(16, 65536, 512) == (1, 4, 512)       # a row past 40,960 needs two parts at least
    assert dsa.dsa_topk_plan(1000, 65536, 512) == (1, 2, 512)
    assert dsa.dsa_topk_plan(1, 163840, 512) == (1, 4, 512)       # the longest row four parts hold
    P = ctypes.c_void_p
    lib.dsa_topk_plan.argtypes = [ctypes.c_int32] * 3 + [P]
    plan = (ctypes.c_int32 * 3)()
    assert lib.dsa_topk_plan(1, 163844, 512, plan) == 2            # DSA_ERR_UNSUPPORTED
    assert lib.dsa_topk_plan(1, 1026, 512, plan) == 1              # ld not a multiple of 4
    assert lib.dsa_topk_plan(1, 1024, 0, plan) == 1                # k < 1
    assert lib.dsa_topk_plan(1, 1024, 512, None) == 1


def test_static_attention_scratch_covers_every_plan_host_only(lib):
    """The allocation-free decode call needs dsa_attn_workspace_size() bytes of its fixed array.  A row's keys
    split over several clusters only while its clusters leave SMs idle, so the partials stay far below the
    array for any shape (rows x splits x clusters never exceed the SM count); the size check runs before any
    device call, and a shape that needs partials passes it (its next failure here is the missing device,
    or the NULL query, never DSA_ERR_UNSUPPORTED)."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    cap = dsa.dsa_attn_static_scratch_bytes()
    worst = 0
    for rows in list(range(1, 65)) + [100, 151, 152, 200, 4096]:
        for heads in (16, 32, 64, 128):
            for keys in (640, 2048 + 1024, 8192 + 128, 65536 + 128, 262144 + 128):
                worst = max(worst, dsa.dsa_attn_workspace_size(rows, heads, keys))
    assert 0 < worst <= cap
    main = dsa.DsaPool(16, None, 8, 64, 512, dsa.DSA_BF16)
    bt = dsa.DsaBlockTable(16, 4, 8)
    swa = dsa.DsaPool(16, None, 8, 256, 512, dsa.DSA_BF16)
    rope = dsa.rope(64)
    assert dsa.dsa_attn_workspace_size(4, 64, 512 + 128) > 0
    code = dsa._lib.dsa_sparse_attn_decode_static(4, 64, None, ctypes.c_void_p(16), 0, ctypes.c_void_p(16), 512,
                                                  ctypes.byref(main), ctypes.byref(bt), ctypes.byref(swa),
                                                  ctypes.byref(bt), 128, 0.0441941738, ctypes.byref(rope),
                                                  ctypes.c_void_p(16), None, None, None)
    assert code in (dsa.DSA_ERR_CUDA, dsa.DSA_ERR_INVALID_ARG)


def test_fp4_pool_checks_host_only(lib):
    """e2m1 pools: indexer keys at dim 128 only, a 32-byte aligned base, and no e2m1 window or attention pools."""
    from compressed_sparse_attention_c4a_gb300 import dsa
    P = ctypes.c_void_p
    bt = dsa.DsaBlockTable(64, 1, 4)
    scale = 256
    fn = lib.dsa_index_scores
    fn.argtypes = [ctypes.c_int32] * 3 + [P] * 5 + [ctypes.c_int32, P, P, P, ctypes.c_int32, P, P, P, P, P]

    def index(dim, base, dtype=dsa.DSA_FP4_E2M1):
        keys = dsa.DsaPool(base, scale, 4, 64, dim, dtype)
        return fn(1, 8, dim, *[P(16)] * 5, 1, ctypes.cast(ctypes.pointer(keys), P), ctypes.cast(ctypes.pointer(bt), P),
                  P(16), 64, None, None, None, None, None)

    assert index(64, 32) == dsa.DSA_ERR_UNSUPPORTED                  # fp4 keys: dim 128 only
    assert index(128, 48) == dsa.DSA_ERR_INVALID_ARG                 # 16- but not 32-byte aligned
    assert index(128, 32, dsa.DSA_BF16) == dsa.DSA_ERR_UNSUPPORTED   # bf16 keys
    lib.dsa_attn_plan.argtypes = [ctypes.c_int32] * 4 + [P]
    plan = (ctypes.c_int32 * 4)()
    assert lib.dsa_attn_plan(4, 64, 640, dsa.DSA_FP4_E2M1, plan) == dsa.DSA_ERR_UNSUPPORTED


def test_compress_rejects_rope_beyond_its_table_host_only(lib):
    """RoPE frequencies are a 32-pair table: rope_dim > 64 is DSA_ERR_UNSUPPORTED before any launch, for the one-cache
    call and for a job of the several-cache call; n_jobs outside 1 .. 4 is DSA_ERR_INVALID_ARG."""
    import torch
    from compressed_sparse_attention_c4a_gb300 import dsa
    P = ctypes.c_void_p
    rope = dsa.DsaRope(128, 10000.0)
    out = dsa.DsaPool(1 << 20, None, 4, 64, 128, dsa.DSA_BF16)
    bt = dsa.DsaBlockTable(64, 1, 4)
    args = [0, 1, P(16), P(16), 1, P(16), P(16), P(16), P(16), P(16), 4, None, ctypes.c_float(1e-6), ctypes.byref(rope),
            ctypes.byref(out), ctypes.byref(bt), None, None, None, None]
    assert dsa._lib.dsa_compress(*args) == dsa.DSA_ERR_UNSUPPORTED
    t = torch.zeros(16)
    job = dsa.compress_job(t, t, t, t, rope, out, bt)
    arr = (dsa.DsaCompressJob * 1)(job)
    assert dsa._lib.dsa_compress_jobs(0, 1, P(16), P(16), 1, P(16), 4, 1, arr, None, None, None) == dsa.DSA_ERR_UNSUPPORTED
    assert dsa._lib.dsa_compress_jobs(0, 1, P(16), P(16), 1, P(16), 4, 5, arr, None, None, None) == dsa.DSA_ERR_INVALID_ARG
    assert dsa._lib.dsa_compress_jobs(0, 1, P(16), P(16), 1, P(16), 4, 0, arr, None, None, None) == dsa.DSA_ERR_INVALID_ARG
    # a query job: rope_dim beyond the table, a dim the kernels do not take
    tq = torch.zeros((2, 4, 128), dtype=torch.bfloat16)
    pos = torch.zeros(2, dtype=torch.int32)
    qj = dsa.query_job(tq, tq, pos, rope)
    ok_job = (dsa.DsaCompressJob * 1)(dsa.compress_job(t, t, t, t, dsa.DsaRope(64, 1e4), out, bt))
    assert dsa._lib.dsa_compress_jobs(0, 1, P(16), P(16), 1, P(16), 4, 1, ok_job, ctypes.byref(qj), None,
                                      None) == dsa.DSA_ERR_UNSUPPORTED
    qj.dim = 96
    qj.rope = ctypes.pointer(dsa.DsaRope(64, 1e4))
    assert dsa._lib.dsa_compress_jobs(0, 1, P(16), P(16), 1, P(16), 4, 1, ok_job, ctypes.byref(qj), None,
                                      None) == dsa.DSA_ERR_UNSUPPORTED
