"""Independent fp64 CPU oracle for paged grouped-query attention with fused RoPE-and-append.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously-correct restatement of
what the hot path computes.  Only the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  It shares no
code with the CUDA library (``paged_kv_gqa_14_gb300``) and neither imports the other.

Sources restated here (page title, section):

* "mini_engine" README, "What it does": a Qwen3 decoder with grouped-query attention and
  RoPE, served from a paged KV cache with block tables; chunked prefill under a token budget.
* "mini_engine" README, "Where the gap comes from": attention gathers the KV blocks into
  contiguous tensors before the softmax -- the semantics the oracle keeps on purpose.
* "mini_engine" README, "Next: fused kernels": fused RoPE, fused QKV split + KV-cache write.
* "09 -- Mini Inference Engine (The Capstone)", "Week 4 -- Paged KV cache": one big pool of
  ``num_blocks x block_size`` slots, block_size 16, per-sequence block table
  (logical block i -> physical block id), attention that gathers through the block table.
* "09 -- Mini Inference Engine (The Capstone)", "Week 3 -- Continuous batching": prefill and
  decode sequences of varying lengths mixed in one batch.

Pinned by ``tests/test_oracle_*.py`` (brute force, closed forms, invariants, library
special cases).  Every function here is pinned; none is "parity unpinned".
"""

from .bf16 import bf16_bits_to_f64, f64_to_bf16_bits
from .rope import rope_inv_freq, rope64
from .append import kv_append, positions_and_slots
from .attention import (
    paged_attention,
    gather_sequence_kv,
    attention_partial,
    merge_partials,
    classify_spans,
)
from .brute import brute_rope, brute_kv_append, brute_paged_attention

__all__ = [
    "bf16_bits_to_f64",
    "f64_to_bf16_bits",
    "rope_inv_freq",
    "rope64",
    "kv_append",
    "positions_and_slots",
    "paged_attention",
    "gather_sequence_kv",
    "attention_partial",
    "merge_partials",
    "classify_spans",
    "brute_rope",
    "brute_kv_append",
    "brute_paged_attention",
]
