"""Host-side logic of the layer step (no GPU): the indexer learns where this step's compressor starts, so
that it can score the key pages the compressor cannot write before that compressor ends."""
import torch

from compressed_sparse_attention_c4a_gb300 import synth
from compressed_sparse_attention_c4a_gb300.step import LayerStep


def test_fresh_pos_is_the_compressor_start():
    """fresh_pos[r] is the first new raw position of request r, the one the compressor call starts from."""
    cached = [0, 1, 6, 7, 8, 9, 1000, 4095, 4096, 65535]
    spec = synth.CaseSpec("fresh", cached=cached, new=[1] * len(cached), seed=5)
    case = synth.make_case(spec, "cpu")
    step = LayerStep(case)
    assert torch.equal(step.fresh_pos, case["start_pos"])
    assert step.fresh_pos.tolist() == cached


def test_fresh_pos_absent_without_an_indexer_compressor():
    spec = synth.CaseSpec("nofresh", cached=[0], new=[700], heads=16, idx_heads=4, idx_dim=64, index_compress=False,
                          seed=12)
    step = LayerStep(synth.make_case(spec, "cpu"))
    assert step.fresh_pos is None
