"""Fused RoPE-and-append in fp64 (test infrastructure only).

Follows:

* "mini_engine" README, "Next: fused kernels": "Fused RoPE" and "Fused QKV split and
  KV-cache write" -- the new token's q and k are rotated and its k, v written into the cache.
* "09 -- Mini Inference Engine (The Capstone)", "Week 4 -- Paged KV cache": the pool is one
  buffer of num_blocks x block_size slots with block_size 16; a sequence's logical block i
  lives in physical block ``block_table[i]``.

Reading of the slot mapping (the pages give the pool, not the index formula): slot s names
row ``s % block_size`` of physical block ``s // block_size``, i.e. the flat row s of the
pool viewed as ``[num_blocks * block_size, num_kv_heads, head_dim]``.  A negative slot is
padding and writes nothing.  Storage is bf16: rotated values are rounded to nearest-even
once, from fp64.
"""

import numpy as np

from .bf16 import bf16_bits_to_f64, f64_to_bf16_bits
from .rope import rope64


def kv_append(q, k, v, positions, slot_mapping, k_cache, v_cache, rope_theta):
    """Return ``(q_rot, k_cache_new, v_cache_new)`` as bf16 bit patterns.

    q:            uint16 [T, Hq, d]   new queries (bf16)
    k, v:         uint16 [T, Hkv, d]  new keys / values (bf16)
    positions:    int    [T]          absolute position of each new token
    slot_mapping: int    [T]          destination slot, < 0 means "skip"
    k_cache, v_cache: uint16 [num_blocks, block_size, Hkv, d]; not modified (copies returned)

    q_rot = bf16(rope(q)); for every t with slot s >= 0 the cache row (s // bs, s % bs)
    becomes bf16(rope(k[t])) in the K cache and exactly v[t] in the V cache.  Every other
    cache row is returned unchanged.
    """
    q = np.asarray(q, dtype=np.uint16)
    k = np.asarray(k, dtype=np.uint16)
    v = np.asarray(v, dtype=np.uint16)
    pos = np.asarray(positions).astype(np.int64)
    slots = np.asarray(slot_mapping).astype(np.int64)
    block_size = k_cache.shape[1]

    # rotation in fp64, one position per token, broadcast over the heads
    q_rot64 = rope64(bf16_bits_to_f64(q), pos[:, None], rope_theta)
    k_rot64 = rope64(bf16_bits_to_f64(k), pos[:, None], rope_theta)
    k_rot = f64_to_bf16_bits(k_rot64)

    kc = np.array(k_cache, dtype=np.uint16, copy=True)
    vc = np.array(v_cache, dtype=np.uint16, copy=True)
    for t in range(q.shape[0]):
        s = int(slots[t])
        if s < 0:
            continue
        blk, off = divmod(s, block_size)
        kc[blk, off] = k_rot[t]
        vc[blk, off] = v[t]
    return f64_to_bf16_bits(q_rot64), kc, vc


def positions_and_slots(query_start_loc, context_lens, block_tables, block_size, num_tokens):
    """Where each new token sits and which pool slot it is written to, from the scheduler's
    tables ("09 -- Mini Inference Engine (The Capstone)", "Week 4 -- Paged KV cache": logical
    block i of a sequence is physical block ``block_table[i]``; the reading of the slot number
    as above).  Token t of sequence b's span (rows ``[qsl[b], qsl[b+1])``, n of them, over a
    context of ctx keys that counts the span) sits at position ``p = ctx - n + (t - qsl[b])``
    and goes to slot ``block_tables[b][p // bs] * bs + p % bs``.  Tokens outside every span
    get position 0 and slot -1.  Returns int64 arrays (positions, slots) of length num_tokens.
    """
    qsl = np.asarray(query_start_loc).astype(np.int64)
    ctx = np.asarray(context_lens).astype(np.int64)
    positions = np.zeros(int(num_tokens), dtype=np.int64)
    slots = np.full(int(num_tokens), -1, dtype=np.int64)
    for b in range(len(ctx)):
        n = int(qsl[b + 1] - qsl[b])
        for r in range(n):
            t = int(qsl[b]) + r
            p = int(ctx[b]) - n + r
            positions[t] = p
            slots[t] = int(block_tables[b][p // block_size]) * block_size + p % block_size
    return positions, slots
