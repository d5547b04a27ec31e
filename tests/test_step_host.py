"""Host-side logic of the layer step (no GPU): the per-request bound that tells the indexer which key
pages this step's compressor may still be writing."""
import numpy as np
import pytest

from compressed_sparse_attention_c4a_gb300 import synth
from compressed_sparse_attention_c4a_gb300.step import LayerStep
from oracle.indexer import visible_entries


@pytest.mark.parametrize("cached", [[0, 1, 6, 7, 8, 9, 10, 11, 12], [1000, 2999, 4095, 4096, 65535, 65536]])
def test_fresh_from_is_entries_complete_before_the_new_tokens(cached):
    """fresh_from[r] = entries whose last raw token precedes request r's first new token (c4a: entry i
    ends at 4i + 7): those the compressor of this step cannot write."""
    spec = synth.CaseSpec("fresh", cached=cached, new=[1] * len(cached), seed=5)
    case = synth.make_case(spec, "cpu")
    step = LayerStep(case)
    start = case["start_pos"].numpy()
    want = np.array([visible_entries(int(p) - 1, "c4a") if p > 0 else 0 for p in start])
    assert np.array_equal(step.fresh_from.numpy(), want)


def test_fresh_from_absent_without_an_indexer_compressor():
    spec = synth.CaseSpec("nofresh", cached=[0], new=[700], heads=16, idx_heads=4, idx_dim=64, index_compress=False,
                          seed=12)
    step = LayerStep(synth.make_case(spec, "cpu"))
    assert step.fresh_from is None
