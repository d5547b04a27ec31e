"""The allocation-free decode attention call against the workspace call.

dsa_sparse_attn_decode_static serves callers that cannot allocate device memory (a serving loop that
forbids cudaMalloc on its hot path, a host whose device memory all belongs to its own arena, a plugin
that only receives input and output pointers): it keeps its split-K partials in a fixed array inside
the library instead of a caller workspace.  Two calls in a row, with different shapes, must each match
dsa_sparse_attn_decode on the same inputs within the attention tolerances; the second call sees the
first call's leftovers in the shared array.

This file is collected last on purpose: if it fails, a run that stops at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_c4a_gb300 import dsa, synth
from compressed_sparse_attention_c4a_gb300.step import LayerStep, SM_SCALE
from _parity import assert_attn_close, pool_absmax, np64

pytestmark = pytest.mark.gpu


def _compare_static_to_workspace(spec):
    step = LayerStep(synth.make_case(spec, "cuda"))
    step.run()                                      # compress, index, top-k, attention via the workspace call
    torch.cuda.synchronize()
    assert step.workspace is not None, "the case must split keys over CTAs (uses scratch)"
    ref, ref_lse = step.out.clone(), step.lse.clone()
    out = torch.full_like(step.out, float("nan"))
    lse = torch.full_like(step.lse, float("nan"))
    c = step.case
    dsa.dsa_sparse_attn_decode_static(c["q"], c["q_pos"], step.kind, step.topk if step.has_index else None,
                                      spec.topk if step.has_index else 0, step.main, step.main_bt, step.swa,
                                      step.swa_bt, spec.window, SM_SCALE, step.rope_main, out, lse,
                                      dev_status=step.status)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    got, want = np64(out), np64(ref)
    assert_attn_close(got, want, pool_absmax((c["main_data"], c["main_scale"]), (c["swa_data"], c["swa_scale"])))
    assert np.max(np.abs(np64(lse) - np64(ref_lse))) <= 1e-3


def test_static_scratch_matches_workspace_call_twice():
    assert dsa.dsa_attn_static_scratch_bytes() == 32 << 20
    # first call: c4a decode over top-k entries plus the window (keys split over several CTAs)
    _compare_static_to_workspace(synth.CaseSpec("noalloc_c4a", cached=[1000, 2999, 777, 4095], new=[1] * 4,
                                                seed=31))
    # second call, right after: another shape (c128a, dense over entries) in the same shared array
    _compare_static_to_workspace(synth.CaseSpec("noalloc_c128a", kind="c128a", cached=[60000, 1279, 127],
                                                new=[1] * 3, idx_heads=0, topk=0, seed=32))

