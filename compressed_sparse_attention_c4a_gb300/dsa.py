"""Python binding of libdsa.so (ctypes): argument marshalling only.

Every function has the name of the C entry point it calls and takes torch tensors (device memory)
plus Python ints/floats; all arithmetic runs in the library's CUDA kernels.  There is no fallback:
if libdsa.so is not built, importing this module raises.
"""
import ctypes
import os

import torch

# DSA_CHECKED=1 selects the bounds-checked build of the same kernels (libdsa_checked.so)
_CHECKED = os.environ.get("DSA_CHECKED") == "1"
_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdsa_checked.so" if _CHECKED else "libdsa.so")
if not os.path.exists(_PATH):
    raise ImportError(f"{_PATH} is not built; run `python -m compressed_sparse_attention_c4a_gb300.build"
                      f"{' --checked' if _CHECKED else ''}`")
_lib = ctypes.CDLL(_PATH)

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA, DSA_ERR_DEVICE_FAULT, DSA_ERR_TIMEOUT = range(6)
DSA_BF16, DSA_FP8_E4M3, DSA_FP4_E2M1 = 0, 1, 2
DSA_C4A, DSA_C128A = 0, 1
KIND = {"c4a": DSA_C4A, "c128a": DSA_C128A}

EXPORTS = ["dsa_status_string", "dsa_compress", "dsa_index_scores", "dsa_topk", "dsa_topk_plan", "dsa_attn_workspace_size",
           "dsa_sparse_attn_decode", "dsa_sparse_attn_prefill", "dsa_gather_rows", "dsa_sparse_attn_decode_static",
           "dsa_attn_static_scratch_bytes", "dsa_attn_plan", "dsa_debug_index_scores_stalled", "dsa_index_topk",
           "dsa_index_topk_workspace_size", "dsa_index_scores_counted", "dsa_topk_counted", "dsa_sparse_attn_q8",
           "dsa_compress_jobs", "dsa_topk_sparse_attn_decode"]


class DsaPool(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("num_blocks", ctypes.c_int32),
                ("rows_per_block", ctypes.c_int32), ("dim", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class DsaBlockTable(ctypes.Structure):
    _fields_ = [("table", ctypes.c_void_p), ("batch", ctypes.c_int32), ("max_blocks", ctypes.c_int32)]


class DsaRope(ctypes.Structure):
    _fields_ = [("rope_dim", ctypes.c_int32), ("theta", ctypes.c_double)]


class DsaCompressJob(ctypes.Structure):
    _fields_ = [("x_new", ctypes.c_void_p), ("logit_new", ctypes.c_void_p), ("state_x", ctypes.c_void_p),
                ("state_logit", ctypes.c_void_p), ("rms_gamma", ctypes.c_void_p), ("rms_eps", ctypes.c_float),
                ("rope", ctypes.POINTER(DsaRope)), ("out", ctypes.POINTER(DsaPool)),
                ("out_bt", ctypes.POINTER(DsaBlockTable)), ("swa", ctypes.POINTER(DsaPool)),
                ("swa_bt", ctypes.POINTER(DsaBlockTable)), ("gate_per_channel", ctypes.c_int32)]


class DsaQueryJob(ctypes.Structure):
    _fields_ = [("nq", ctypes.c_int32), ("heads", ctypes.c_int32), ("dim", ctypes.c_int32), ("q_raw", ctypes.c_void_p),
                ("q_out", ctypes.c_void_p), ("q_pos", ctypes.c_void_p), ("rms_gamma", ctypes.c_void_p),
                ("rms_eps", ctypes.c_float), ("rope", ctypes.POINTER(DsaRope))]


class DsaError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn}: {dsa_status_string(code)} ({code})")
        self.code = code


_P = ctypes.c_void_p
_I = ctypes.c_int32
_lib.dsa_status_string.restype = ctypes.c_char_p
_lib.dsa_status_string.argtypes = [_I]
_lib.dsa_attn_workspace_size.restype = ctypes.c_size_t
_lib.dsa_attn_workspace_size.argtypes = [_I, _I, _I]
_lib.dsa_attn_static_scratch_bytes.restype = ctypes.c_size_t
_lib.dsa_attn_static_scratch_bytes.argtypes = []
_lib.dsa_attn_plan.restype = ctypes.c_int32
_lib.dsa_attn_plan.argtypes = [_I, _I, _I, _I, _P]
_lib.dsa_index_topk_workspace_size.restype = ctypes.c_size_t
_lib.dsa_index_topk_workspace_size.argtypes = [_I]
_lib.dsa_topk_plan.restype = ctypes.c_int32
_lib.dsa_topk_plan.argtypes = [_I, _I, _I, _P]
for _name, _args in {
    "dsa_compress": [_I, _I, _P, _P, _I, _P, _P, _P, _P, _P, _I, _P, ctypes.c_float, _P, _P, _P, _P, _P, _P, _P],
    "dsa_compress_jobs": [_I, _I, _P, _P, _I, _P, _I, _I, _P, _P, _P, _P],
    "dsa_index_scores": [_I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P],
    "dsa_debug_index_scores_stalled": [_I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, ctypes.c_uint64, _P,
                                       _P],
    "dsa_topk": [_I, _P, _I, _P, _I, _P, _P, _P],
    "dsa_index_topk": [_I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _P, _I, _P, _P, ctypes.c_size_t, _P,
                       _P],
    "dsa_index_scores_counted": [_I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P],
    "dsa_topk_counted": [_I, _P, _I, _P, _I, _P, _P, _P, _P],
    "dsa_sparse_attn_decode": [_I, _I, _P, _P, _I, _P, _I, _P, _P, _P, _P, _I, ctypes.c_float, _P, _P, _P, _P,
                               ctypes.c_size_t, _P, _P],
    "dsa_sparse_attn_prefill": [_I, _I, _P, _P, _P, _I, _P, _I, _P, _P, _P, _P, _I, ctypes.c_float, _P, _P, _P,
                                _P, ctypes.c_size_t, _P, _P],
    "dsa_topk_sparse_attn_decode": [_I, _I, _P, _P, _I, _P, _I, _P, _I, _P, _P, _P, _P, _P, _I, ctypes.c_float, _P,
                                    _P, _P, _P, ctypes.c_size_t, _P, _P],
    "dsa_gather_rows": [_P, _P, _I, _P, _P, _P, _P, _P, _P],
    "dsa_sparse_attn_q8": [_I, _I, _P, _P, _P, _I, _P, _I, _P, _P, _P, _P, _I, ctypes.c_float, _P, _P, _P, _P, _P,
                           ctypes.c_size_t, _P, _P],
    "dsa_sparse_attn_decode_static": [_I, _I, _P, _P, _I, _P, _I, _P, _P, _P, _P, _I, ctypes.c_float, _P, _P, _P,
                                      _P, _P],
}.items():
    getattr(_lib, _name).restype = _I
    getattr(_lib, _name).argtypes = _args


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, code):
    if code != DSA_OK:
        raise DsaError(fn, code)


def dsa_status_string(code):
    return _lib.dsa_status_string(code).decode()


def pool(data, rows_per_block, scale=None, fmt=None):
    """A DsaPool over a tensor viewed as [num_blocks * rows_per_block, row] (bf16, uint8 e4m3, or with
    fmt="fp4" uint8 bytes of two e2m1 codes each, so that dim = 2 * row)."""
    rows = data.numel() // data.shape[-1]
    assert rows % rows_per_block == 0
    if fmt == "fp4":
        assert data.dtype == torch.uint8
        dtype, dim = DSA_FP4_E2M1, 2 * data.shape[-1]
    else:
        dtype = DSA_BF16 if data.dtype == torch.bfloat16 else DSA_FP8_E4M3
        dim = data.shape[-1]
    return DsaPool(data.data_ptr(), None if scale is None else scale.data_ptr(), rows // rows_per_block,
                   rows_per_block, dim, dtype)


def block_table(table):
    """A DsaBlockTable over an int32 [batch][max_blocks] tensor."""
    return DsaBlockTable(table.data_ptr(), table.shape[0], table.shape[1])


def rope(rope_dim=64, theta=10000.0):
    return DsaRope(rope_dim, theta)


def dsa_compress(kind, cu_new, start_pos, max_new, x_new, logit_new, state_x, state_logit, state_slot,
                 rope_cfg, out, out_bt, swa=None, swa_bt=None, rms_gamma=None, rms_eps=1e-6, dev_status=None,
                 stream=None):
    code = _lib.dsa_compress(KIND.get(kind, kind), start_pos.numel(), _ptr(cu_new), _ptr(start_pos), int(max_new),
                             _ptr(x_new), _ptr(logit_new), _ptr(state_x), _ptr(state_logit), _ptr(state_slot),
                             state_x.shape[0], _ptr(rms_gamma), float(rms_eps), ctypes.byref(rope_cfg),
                             ctypes.byref(out), ctypes.byref(out_bt),
                             None if swa is None else ctypes.byref(swa),
                             None if swa_bt is None else ctypes.byref(swa_bt), _ptr(dev_status), _stream(stream))
    _check("dsa_compress", code)


def compress_job(x_new, logit_new, state_x, state_logit, rope_cfg, out, out_bt, swa=None, swa_bt=None,
                 rms_gamma=None, rms_eps=1e-6, per_channel=False):
    """One cache's arguments of dsa_compress_jobs (the struct keeps the rope, pool and table objects alive).
    per_channel: logits per raw token and channel (logit_new [n][dim], state_logit [slots][w][dim])."""
    return DsaCompressJob(x_new.data_ptr(), logit_new.data_ptr(), state_x.data_ptr(), state_logit.data_ptr(),
                          None if rms_gamma is None else rms_gamma.data_ptr(), float(rms_eps), ctypes.pointer(rope_cfg),
                          ctypes.pointer(out), ctypes.pointer(out_bt), None if swa is None else ctypes.pointer(swa),
                          None if swa_bt is None else ctypes.pointer(swa_bt), 1 if per_channel else 0)


def query_job(q_raw, q_out, q_pos, rope_cfg, rms_gamma=None, rms_eps=1e-6):
    """The query job of dsa_compress_jobs: q_raw, q_out [nq][heads][dim] bf16 (q_out may be q_raw)."""
    nq, heads, dim = q_raw.shape
    return DsaQueryJob(nq, heads, dim, q_raw.data_ptr(), q_out.data_ptr(), q_pos.data_ptr(),
                       None if rms_gamma is None else rms_gamma.data_ptr(), float(rms_eps), ctypes.pointer(rope_cfg))


def dsa_compress_jobs(kind, cu_new, start_pos, max_new, state_slot, num_slots, jobs, dev_status=None, stream=None,
                      query=None):
    arr = (DsaCompressJob * len(jobs))(*jobs) if jobs else None
    code = _lib.dsa_compress_jobs(KIND.get(kind, kind), start_pos.numel(), _ptr(cu_new), _ptr(start_pos), int(max_new),
                                  _ptr(state_slot), int(num_slots), len(jobs), arr,
                                  None if query is None else ctypes.byref(query), _ptr(dev_status), _stream(stream))
    _check("dsa_compress_jobs", code)


def dsa_index_scores(q8, q_scale, w, q_pos, q_req, q_group, keys, bt, scores, n_visible=None, dev_status=None,
                     stream=None, fresh_pos=None, work=None):
    nq, heads, dim = q8.shape
    code = _lib.dsa_index_scores(nq, heads, dim, _ptr(q8), _ptr(q_scale), _ptr(w), _ptr(q_pos), _ptr(q_req),
                                 int(q_group), ctypes.byref(keys), ctypes.byref(bt), _ptr(scores), scores.shape[1],
                                 _ptr(n_visible), _ptr(fresh_pos), _ptr(work), _ptr(dev_status), _stream(stream))
    _check("dsa_index_scores", code)


def dsa_debug_index_scores_stalled(q8, q_scale, w, q_pos, q_req, q_group, keys, bt, scores, wait_limit_ns,
                                   n_visible=None, dev_status=None, stream=None):
    """Test hook: the indexer launch with every copy withheld, so its bounded waits run out after
    ``wait_limit_ns`` (see include/dsa.h)."""
    nq, heads, dim = q8.shape
    code = _lib.dsa_debug_index_scores_stalled(nq, heads, dim, _ptr(q8), _ptr(q_scale), _ptr(w), _ptr(q_pos),
                                               _ptr(q_req), int(q_group), ctypes.byref(keys), ctypes.byref(bt),
                                               _ptr(scores), scores.shape[1], _ptr(n_visible), int(wait_limit_ns),
                                               _ptr(dev_status), _stream(stream))
    _check("dsa_debug_index_scores_stalled", code)


def dsa_index_topk_workspace_size(nq):
    return int(_lib.dsa_index_topk_workspace_size(int(nq)))


def dsa_index_topk(q8, q_scale, w, q_pos, q_req, q_group, keys, bt, scores, k, idx_out, workspace, n_visible=None,
                   dev_status=None, stream=None, fresh_pos=None):
    """Indexer scores with the per-query top-k fused in (see include/dsa.h); ``workspace`` a zero-filled
    device buffer of at least dsa_index_topk_workspace_size(nq) bytes."""
    nq, heads, dim = q8.shape
    code = _lib.dsa_index_topk(nq, heads, dim, _ptr(q8), _ptr(q_scale), _ptr(w), _ptr(q_pos), _ptr(q_req),
                               int(q_group), ctypes.byref(keys), ctypes.byref(bt), _ptr(scores), scores.shape[1],
                               _ptr(n_visible), _ptr(fresh_pos), int(k), _ptr(idx_out), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream))
    _check("dsa_index_topk", code)


def dsa_index_scores_counted(q8, q_scale, w, q_pos, q_req, q_group, keys, bt, scores, counts, n_visible=None,
                             dev_status=None, stream=None, fresh_pos=None, work=None):
    """dsa_index_scores that also counts each row's level-1 top-k histogram into ``counts`` (zero-filled)."""
    nq, heads, dim = q8.shape
    code = _lib.dsa_index_scores_counted(nq, heads, dim, _ptr(q8), _ptr(q_scale), _ptr(w), _ptr(q_pos), _ptr(q_req),
                                         int(q_group), ctypes.byref(keys), ctypes.byref(bt), _ptr(scores),
                                         scores.shape[1], _ptr(n_visible), _ptr(fresh_pos), _ptr(work), _ptr(counts),
                                         _ptr(dev_status), _stream(stream))
    _check("dsa_index_scores_counted", code)


def dsa_topk_counted(scores, n_valid, k, idx_out, counts, dev_status=None, stream=None):
    """dsa_topk starting from the counts dsa_index_scores_counted made (and clearing them)."""
    code = _lib.dsa_topk_counted(scores.shape[0], _ptr(scores), scores.shape[1], _ptr(n_valid), int(k), _ptr(idx_out),
                                 _ptr(counts), _ptr(dev_status), _stream(stream))
    _check("dsa_topk_counted", code)


def dsa_topk(scores, n_valid, k, idx_out, dev_status=None, stream=None):
    code = _lib.dsa_topk(scores.shape[0], _ptr(scores), scores.shape[1], _ptr(n_valid), int(k), _ptr(idx_out),
                         _ptr(dev_status), _stream(stream))
    _check("dsa_topk", code)


def dsa_attn_workspace_size(nq, heads, max_keys):
    return int(_lib.dsa_attn_workspace_size(int(nq), int(heads), int(max_keys)))


def dsa_topk_plan(nq, ld, k):
    """(kernel: 0 registers / 1 cluster, CTAs per row, threads per CTA) of the top-k call."""
    plan = (ctypes.c_int32 * 3)()
    _check("dsa_topk_plan", _lib.dsa_topk_plan(int(nq), int(ld), int(k), plan))
    return tuple(int(x) for x in plan)


def dsa_attn_plan(nq, heads, max_keys, dtype="bf16"):
    """(heads per CTA, CTAs per cluster, key splits per row, kernels per call) of the attention call."""
    plan = (ctypes.c_int32 * 4)()
    code = _lib.dsa_attn_plan(int(nq), int(heads), int(max_keys), {"bf16": DSA_BF16, "fp8": DSA_FP8_E4M3}.get(dtype, dtype),
                              plan)
    _check("dsa_attn_plan", code)
    return tuple(int(x) for x in plan)


def dsa_sparse_attn_decode(q, q_pos, kind, topk, k, main, main_bt, swa, swa_bt, window, sm_scale, rope_cfg, out,
                           lse=None, workspace=None, dev_status=None, stream=None):
    B, H, _ = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    code = _lib.dsa_sparse_attn_decode(B, H, _ptr(q), _ptr(q_pos), KIND.get(kind, kind), _ptr(topk), int(k),
                                       ctypes.byref(main), ctypes.byref(main_bt), ctypes.byref(swa),
                                       ctypes.byref(swa_bt), int(window), float(sm_scale), ctypes.byref(rope_cfg),
                                       _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, _ptr(dev_status),
                                       _stream(stream))
    _check("dsa_sparse_attn_decode", code)


def dsa_topk_sparse_attn_decode(q, q_pos, kind, scores, n_visible, k, topk_out, main, main_bt, swa, swa_bt, window,
                                sm_scale, rope_cfg, out, lse=None, workspace=None, dev_status=None, stream=None):
    """dsa_topk of (scores, n_visible, k) into topk_out, then dsa_sparse_attn_decode over it (one kernel when the
    work split allows)."""
    B, H, _ = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    code = _lib.dsa_topk_sparse_attn_decode(B, H, _ptr(q), _ptr(q_pos), KIND.get(kind, kind), _ptr(scores),
                                            scores.shape[1], _ptr(n_visible), int(k), _ptr(topk_out),
                                            ctypes.byref(main), ctypes.byref(main_bt), ctypes.byref(swa),
                                            ctypes.byref(swa_bt), int(window), float(sm_scale), ctypes.byref(rope_cfg),
                                            _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, _ptr(dev_status),
                                            _stream(stream))
    _check("dsa_topk_sparse_attn_decode", code)


def dsa_sparse_attn_prefill(q, q_pos, q_req, kind, topk, k, main, main_bt, swa, swa_bt, window, sm_scale, rope_cfg,
                            out, lse=None, workspace=None, dev_status=None, stream=None):
    nq, H, _ = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    code = _lib.dsa_sparse_attn_prefill(nq, H, _ptr(q), _ptr(q_pos), _ptr(q_req), KIND.get(kind, kind), _ptr(topk),
                                        int(k), ctypes.byref(main), ctypes.byref(main_bt), ctypes.byref(swa),
                                        ctypes.byref(swa_bt), int(window), float(sm_scale), ctypes.byref(rope_cfg),
                                        _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, _ptr(dev_status),
                                        _stream(stream))
    _check("dsa_sparse_attn_prefill", code)


def dsa_sparse_attn_q8(q, q_pos, q_req, kind, topk, k, main, main_bt, swa, swa_bt, window, sm_scale, rope_cfg, out,
                       out_scale, lse=None, workspace=None, dev_status=None, stream=None):
    """Attention with the output in e4m3 and an amax/448 scale per 128-dim block (see include/dsa.h); q_req None
    for decode rows."""
    nq, H, _ = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    code = _lib.dsa_sparse_attn_q8(nq, H, _ptr(q), _ptr(q_pos), _ptr(q_req), KIND.get(kind, kind), _ptr(topk), int(k),
                                   ctypes.byref(main), ctypes.byref(main_bt), ctypes.byref(swa), ctypes.byref(swa_bt),
                                   int(window), float(sm_scale), ctypes.byref(rope_cfg), _ptr(out), _ptr(out_scale),
                                   _ptr(lse), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check("dsa_sparse_attn_q8", code)


def dsa_gather_rows(pool_, bt, req, ids, out, out_scale=None, dev_status=None, stream=None):
    code = _lib.dsa_gather_rows(ctypes.byref(pool_), ctypes.byref(bt), ids.numel(), _ptr(req), _ptr(ids), _ptr(out),
                                _ptr(out_scale), _ptr(dev_status), _stream(stream))
    _check("dsa_gather_rows", code)


def dsa_attn_static_scratch_bytes():
    return int(_lib.dsa_attn_static_scratch_bytes())


def dsa_sparse_attn_decode_static(q, q_pos, kind, topk, k, main, main_bt, swa, swa_bt, window, sm_scale, rope_cfg,
                                  out, lse=None, dev_status=None, stream=None):
    """dsa_sparse_attn_decode for callers that cannot allocate: split-K partials go to the library's
    fixed per-device scratch array instead of a caller workspace (see include/dsa.h)."""
    B, H, _ = q.shape
    code = _lib.dsa_sparse_attn_decode_static(B, H, _ptr(q), _ptr(q_pos), KIND.get(kind, kind), _ptr(topk), int(k),
                                              ctypes.byref(main), ctypes.byref(main_bt), ctypes.byref(swa),
                                              ctypes.byref(swa_bt), int(window), float(sm_scale),
                                              ctypes.byref(rope_cfg), _ptr(out), _ptr(lse), _ptr(dev_status),
                                              _stream(stream))
    _check("dsa_sparse_attn_decode_static", code)
