"""Write the stored expected values under tests/golden/ from the oracle alone.

Run from the repository root:  python tests/golden/make_golden.py
The inputs come from the seeded generator (paged_kv_gqa_14_gb300.workloads); the expected
values come only from oracle/.  Nothing here touches the CUDA library.
"""

import hashlib
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from paged_kv_gqa_14_gb300 import workloads as W  # noqa: E402


def digest(*arrays):
    h = hashlib.sha256()
    for a in arrays:
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def tiny_decode():
    bt = W.config(1)
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping,
                                     bt.k_cache, bt.v_cache, bt.rope_theta)
    out = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens,
                                 bt.query_start_loc, bt.scale)
    return {
        "what": "tiny decode workload (4 seqs, contexts 1/17/33/100, 4 q / 2 kv heads, d 64): "
                "oracle kv_append then oracle paged_attention",
        "source": "mini_engine README 'What it does' (GQA + RoPE, paged KV cache); "
                  "09 -- Mini Inference Engine (The Capstone) 'Week 4 -- Paged KV cache'",
        "input_sha256": digest(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache,
                               bt.v_cache, bt.block_tables, bt.context_lens, bt.query_start_loc),
        "q_rot_bits": q_rot.astype(int).tolist(),
        "k_cache_sha256": digest(kc),
        "v_cache_sha256": digest(vc),
        "out": [[[float(x) for x in row] for row in tok] for tok in out],
    }


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_decode_oracle.json")
    with open(path, "w") as f:
        json.dump(tiny_decode(), f, indent=0)
    print("wrote", path)
