"""CPU oracle for KV-shared prompt prefill: TEST INFRASTRUCTURE ONLY.

Plain, slow, readable numpy (fp32, with fp64 where a step is computed once
per table) restatement of what the prefill pass computes.  Only the tests,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import it.  The product path (the CUDA library and
its Python binding) never imports, links or calls anything in here, and this
package imports nothing from the product path: the two share no code.  The
only common module is the seeded input generator, which holds no arithmetic
of the method.

Sources (web pages, by title and section):
- "llama.cpp Gemma 4 prefill KV graph optimization" (devotd.net news, zh-hans
  and ko versions), section 1: KV-shared layers write no K/V and reuse an
  earlier layer's cache; before the first such layer the token rows that no
  output needs are pruned; intermediate ubatches skip those layers and the
  last ubatch carries one row; per-layer-embedding scaling; the pruning
  predicate listing (n_layer_kv_from_start, single sequence, no embeddings).
  Section 3's closing paragraph: outputs identical to the unpruned graph.
- "PicoLM KV Cache persistence" (xxqk.cn news 668802), "file" paragraph: the
  cache file holds a magic "KVCP", metadata (cached positions, layers, KV
  dim), then FP16 keys of the first N positions, then FP16 values; "rules"
  paragraph: layers / KV-dim mismatches are refused, the cached position count
  may not exceed the context length.

Where the pages leave the architecture open, the oracle takes the plainest
readings the rest supports: a pre-norm decoder with RMSNorm gains (1 + g),
half-split RoPE, GELU in its tanh form, the per-layer-embedding block
x += W_pp (gelu(W_pg x) * ple) after the FFN, no embedding scale and a tied
head.  Every function here is pinned by the tests to something outside it
(hand-written values, closed forms, a published error bound, float64
brute-force loops, the pages' worked size).  What no pin can confirm is the
choice of those readings itself: the pages fix no architecture, so the
brute-force models check that the oracle computes the readings correctly,
not that a particular checkpoint would use them.
"""
from .prefill import (  # noqa: F401
    OracleContext,
    attention,
    gelu_tanh,
    kv_image_bytes,
    prune_shared,
    q4_0_decode,
    rmsnorm,
    rope_neox,
    silu,
)
