"""Pure-Python brute force of the same definitions (test infrastructure only).

Every value is handled one scalar at a time with Python floats (IEEE fp64) and the ``math``
module; block-table lookups are explicit integer arithmetic per key.  Only for tiny inputs
(a few sequences, contexts of tens of tokens, small head_dim).  It exists to pin the
vectorised oracle: a transposed operand, a wrong gather index or a dropped term in one of
the two shows up as a disagreement.

Same readings as ``oracle.rope``, ``oracle.append`` and ``oracle.attention``.
"""

import math
import struct


def _bf16_to_float(bits):
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def brute_rope(vec, pos, theta):
    """Rotate one head vector (a list of Python floats) to position ``pos``."""
    d = len(vec)
    half = d // 2
    out = [0.0] * d
    for i in range(half):
        freq = float(theta) ** (-2.0 * i / d)
        ang = float(pos) * freq
        c, s = math.cos(ang), math.sin(ang)
        a, b = vec[i], vec[i + half]
        out[i] = a * c - b * s
        out[i + half] = b * c + a * s
    return out


def brute_kv_append(k, v, positions, slot_mapping, k_cache, v_cache, rope_theta):
    """Return {(block, offset, kv_head): (k_rot as floats, v as bf16 bits)} for written rows.

    k, v: nested lists / arrays of bf16 bits [T][Hkv][d].  ``k_cache`` only supplies the
    block size (its dim 1).  No rounding to bf16 here: the caller compares against the
    oracle's stored bf16 with the rounding tolerance.
    """
    block_size = len(k_cache[0])
    written = {}
    for t in range(len(k)):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        blk = slot // block_size
        off = slot - blk * block_size
        for h in range(len(k[t])):
            kv = [_bf16_to_float(x) for x in k[t][h]]
            written[(blk, off, h)] = (brute_rope(kv, positions[t], rope_theta), list(v[t][h]))
    return written


def brute_paged_attention(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale):
    """Explicit loops over (sequence, row, q head, key, dim).  Returns nested lists [T][Hq][d]."""
    T = len(q)
    Hq = len(q[0])
    d = len(q[0][0])
    block_size = len(k_cache[0])
    hkv = len(k_cache[0][0])
    group = Hq // hkv
    out = [[[float("nan")] * d for _ in range(Hq)] for _ in range(T)]
    for b in range(len(context_lens)):
        start = int(query_start_loc[b])
        n = int(query_start_loc[b + 1]) - start
        ctx = int(context_lens[b])
        for r in range(n):
            t = start + r
            last = ctx - n + r
            for h in range(Hq):
                kh = h // group
                qv = [_bf16_to_float(x) for x in q[t][h]]
                scores = []
                for j in range(last + 1):
                    phys = int(block_tables[b][j // block_size])
                    off = j % block_size
                    kj = k_cache[phys][off][kh]
                    dot = 0.0
                    for i in range(d):
                        dot += qv[i] * _bf16_to_float(kj[i])
                    scores.append(scale * dot)
                mx = max(scores)
                w = [math.exp(s - mx) for s in scores]
                z = sum(w)
                for i in range(d):
                    acc = 0.0
                    for j in range(last + 1):
                        phys = int(block_tables[b][j // block_size])
                        acc += w[j] * _bf16_to_float(v_cache[phys][j % block_size][kh][i])
                    out[t][h][i] = acc / z
    return out
