"""Paged grouped-query attention over a ragged prefill/decode batch, fp64 (test infrastructure only).

Follows:

* "mini_engine" README, "What it does": grouped-query attention; chunked prefill under
  max_num_batched_tokens.
* "mini_engine" README, "Where the gap comes from": attention gathers the KV blocks --
  the oracle does exactly that: gather through the block table into contiguous K/V, then
  plain softmax attention.
* "09 -- Mini Inference Engine (The Capstone)", "Week 4 -- Paged KV cache": per-sequence
  block table, logical block i -> physical block id; "rewrite attention to gather from
  block table".
* "09 -- Mini Inference Engine (The Capstone)", "Week 3 -- Continuous batching": a batch
  mixes prefill and decode sequences of varying lengths.

Readings taken where the pages are silent:

* ``context_lens[b]`` counts every key of sequence b, including the span's new tokens.
* The span of sequence b is rows ``[query_start_loc[b], query_start_loc[b+1])`` of q and
  out.  Row r of an n-row span is the token at position ``ctx - n + r`` and attends to keys
  ``0 .. ctx - n + r`` (causal, aligned to the end of the context).  A decode step is a span
  of one row that sees the whole context.
* q head h reads kv head ``h // (Hq / Hkv)`` (contiguous groups).
* Rows of out that no span covers are left as NaN by the oracle (the kernels leave them
  untouched).
"""

import numpy as np

from .bf16 import bf16_bits_to_f64

SPAN_NONE = 0
SPAN_DECODE = 1
SPAN_PREFILL = 2


def classify_spans(query_start_loc, context_lens, block_size=16):
    """Per sequence: the span kind and the number of KV pages the step reads.

    kind is SPAN_NONE for an empty span, SPAN_DECODE for a span of one new token, and
    SPAN_PREFILL for a longer (chunked-prefill) span -- the mixed batch of "Week 3".
    pages = ceil(ctx / block_size) ("Week 4": a sequence holds ceil(len / 16) blocks).
    """
    qsl = np.asarray(query_start_loc).astype(np.int64)
    ctx = np.asarray(context_lens).astype(np.int64)
    spans = qsl[1:] - qsl[:-1]
    kind = np.where(spans == 0, SPAN_NONE, np.where(spans == 1, SPAN_DECODE, SPAN_PREFILL))
    pages = np.where(spans == 0, 0, -(-ctx // block_size))
    return kind.astype(np.int32), pages.astype(np.int64), spans


def gather_sequence_kv(k_cache, v_cache, block_table_row, ctx):
    """Gather one sequence's first ``ctx`` keys/values into contiguous fp64 [ctx, Hkv, d]."""
    block_size = k_cache.shape[1]
    nblk = -(-int(ctx) // block_size)
    ids = np.asarray(block_table_row[:nblk]).astype(np.int64)
    hkv, d = k_cache.shape[2], k_cache.shape[3]
    K = bf16_bits_to_f64(k_cache[ids].reshape(nblk * block_size, hkv, d)[:ctx])
    V = bf16_bits_to_f64(v_cache[ids].reshape(nblk * block_size, hkv, d)[:ctx])
    return K, V


def paged_attention(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale):
    """out[t, h] = softmax(scale * q[t, h] . K^T over the visible keys) . V, in fp64.

    q:             uint16 [T, Hq, d]  (bf16, already rotated)
    k_cache/v_cache: uint16 [num_blocks, block_size, Hkv, d]
    block_tables:  int [B, max_blocks]
    context_lens:  int [B]
    query_start_loc: int [B + 1]
    Returns float64 [T, Hq, d].
    """
    q = np.asarray(q, dtype=np.uint16)
    T, Hq, d = q.shape
    hkv = k_cache.shape[2]
    if Hq % hkv:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    group = Hq // hkv
    qsl = np.asarray(query_start_loc).astype(np.int64)
    ctxs = np.asarray(context_lens).astype(np.int64)
    out = np.full((T, Hq, d), np.nan)
    for b in range(len(ctxs)):
        start, end = int(qsl[b]), int(qsl[b + 1])
        n = end - start
        if n == 0:
            continue
        ctx = int(ctxs[b])
        if ctx < n:
            raise ValueError(f"sequence {b}: context {ctx} shorter than its span {n}")
        K, V = gather_sequence_kv(k_cache, v_cache, block_tables[b], ctx)
        Q = bf16_bits_to_f64(q[start:end])
        for h in range(Hq):
            kh = h // group
            S = scale * (Q[:, h, :] @ K[:, kh, :].T)  # [n, ctx]
            for r in range(n):
                last = ctx - n + r  # causal: keys 0..last are visible
                s = S[r, : last + 1]
                p = np.exp(s - s.max())
                p /= p.sum()
                out[start + r, h] = p @ V[: last + 1, kh, :]
    return out


def attention_partial(qvec, K, V, scale):
    """Softmax statistics of one query row over a subset of keys.

    Returns (m, l, acc) with m = max score, l = sum exp(s - m), acc = sum exp(s - m) v:
    the state a split of the keys carries before the splits are merged.
    """
    s = scale * (K @ qvec)
    m = s.max()
    e = np.exp(s - m)
    return m, e.sum(), e @ V


def merge_partials(ms, ls, accs):
    """Combine split states into the softmax output.

    With M = max_s m_s:  out = sum_s e^{m_s - M} acc_s / sum_s e^{m_s - M} l_s.
    Equals the softmax over the union of the splits' keys (log-sum-exp rescaling).
    """
    ms = np.asarray(ms, dtype=np.float64)
    w = np.exp(ms - ms.max())
    num = sum(wi * np.asarray(a, dtype=np.float64) for wi, a in zip(w, accs))
    den = float(np.dot(w, np.asarray(ls, dtype=np.float64)))
    return num / den

