"""Plain, slow CPU oracle for one compressed-sparse-attention (c4a / c128a) layer step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or calls this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it.  It shares no code, header,
table or constant generator with the CUDA library; it reads the same seeded input
bytes and nothing else.

Everything is computed in float64 with numpy.  Stored values (bf16 cache rows,
e4m3 indexer codes) are decoded with this package's own codecs, written from the
bf16 bit layout and the OCP OFP8 specification.

Sources (web pages on the method; cited by page title and section):
  [P1] "DeepSeek DSA、DeepSeek V4与vLLM Hybrid KV Cache详解" (gentlecold.top)
  [P2] "DeepSeek V4 稀疏注意力完全解剖" (zoe.im)

Modules, in the order the layer step runs them:
  codecs     bf16 / e4m3 rounding, decoding, per-row fp8 scaling
  rope       rotary position embedding on the last ``rope_dim`` dims
  paging     256-position logical blocks and block-table translation
  compress   c4a / c128a compressor (gate, weighted sum, RMSNorm, RoPE), SWA insert
  indexer    lightning-indexer scores with the causal visibility rule
  topk       per-query top-k with lowest-index tie-break
  attention  MQA attention over top-k entries + sliding window, inverse RoPE
  layer      the ABI-shaped stages over paged pools (what the GPU calls compute)

Parity status: every function is pinned by a ``-m "not gpu"`` test against a
closed form, a library routine, a brute force or an invariant; none is
"parity unpinned".
"""
