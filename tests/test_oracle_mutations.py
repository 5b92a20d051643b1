"""The pins are sharp: plausible mistakes planted in a copy of the oracle fail them.

Each case rewrites one line of an oracle module's source (a flipped sign, a wrong index,
a transposed pair layout, a dropped scale, a lost causal bound, a swapped gather order),
loads the mutant as a separate module, and checks that the independent reference the pins
use -- brute force, the complex-rotation form, the library SDPA -- disagrees with it.  The
real oracle is never modified.
"""

import importlib.util
import os

import numpy as np
import pytest

import oracle
from paged_kv_gqa_14_gb300 import workloads as W

ORACLE_DIR = os.path.dirname(os.path.abspath(oracle.__file__))


def _mutant(module, old, new):
    path = os.path.join(ORACLE_DIR, module + ".py")
    src = open(path).read()
    assert src.count(old) == 1, f"mutation anchor not unique in {module}: {old!r}"
    spec = importlib.util.spec_from_loader(f"oracle._mutant_{module}", loader=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    exec(compile(src.replace(old, new), path + " (mutant)", "exec"), mod.__dict__)
    return mod


ROPE_MUTANTS = [
    ("x1 * c - x2 * s", "x1 * c + x2 * s"),
    ("x2 * c + x1 * s", "x2 * c - x1 * s"),
    ("(-2.0 * i / head_dim)", "(-1.0 * i / head_dim)"),
    ("x1 = x[..., :half]\n    x2 = x[..., half:]", "x1 = x[..., 0::2]\n    x2 = x[..., 1::2]"),
]


@pytest.mark.parametrize("old,new", ROPE_MUTANTS)
def test_rope_pins_catch_mutant(old, new):
    m = _mutant("rope", old, new)
    rng = np.random.default_rng(0)
    x = rng.standard_normal(64)
    caught = False
    for p in [1, 17, 300]:
        ref = oracle.brute_rope(list(x), p, 1e4)
        if not np.allclose(m.rope64(x, np.float64(p), 1e4), ref, atol=1e-9):
            caught = True
    assert caught


ATTN_MUTANTS = [
    ("kh = h // group", "kh = h % hkv"),
    ("last = ctx - n + r  #", "last = ctx - 1  #"),
    ("S = scale * (Q[:, h, :]", "S = (Q[:, h, :]"),
    ("ids = np.asarray(block_table_row[:nblk])", "ids = np.sort(np.asarray(block_table_row[:nblk]))"),
    ("out[start + r, h] = p @ V[: last + 1, kh, :]", "out[start + r, h] = p @ V[: last + 1, 0, :]"),
    ("Q = bf16_bits_to_f64(q[start:end])", "Q = bf16_bits_to_f64(q[start:end])[::-1]"),
]


@pytest.mark.parametrize("old,new", ATTN_MUTANTS)
def test_attention_pins_catch_mutant(old, new):
    m = _mutant("attention", old, new)
    caught = False
    for seed in range(6):
        bt = W.random_case(seed, max_ctx=36, head_dims=(8,), groups=(2, 3), kv_heads=(2,))
        q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping,
                                         bt.k_cache, bt.v_cache, bt.rope_theta)
        ref = np.array(oracle.brute_paged_attention(q_rot.tolist(), kc.tolist(), vc.tolist(),
                                                    bt.block_tables.tolist(), bt.context_lens.tolist(),
                                                    bt.query_start_loc.tolist(), bt.scale))
        try:
            got = m.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens,
                                    bt.query_start_loc, bt.scale)
        except Exception:
            caught = True
            break
        if not (np.all(np.isfinite(got)) and np.max(np.abs(got - ref)) < 1e-12):
            caught = True
            break
    assert caught


APPEND_MUTANTS = [
    ("blk, off = divmod(s, block_size)", "off, blk = divmod(s, block_size)"),
    ("vc[blk, off] = v[t]", "vc[blk, off] = k[t]"),
    ("if s < 0:\n            continue", "if s < -1:\n            continue"),
    ("k_rot64 = rope64(bf16_bits_to_f64(k), pos[:, None], rope_theta)",
     "k_rot64 = bf16_bits_to_f64(k)"),
]


@pytest.mark.parametrize("old,new", APPEND_MUTANTS)
def test_append_pins_catch_mutant(old, new):
    m = _mutant("append", old, new)
    bt = W.make_batch([5, 40, 17], [1, 1, 1], 4, 2, 16, 10, seed=3)
    slots = bt.slot_mapping.copy()
    slots[2] = -1
    try:
        q_rot, kc, vc = m.kv_append(bt.q, bt.k, bt.v, bt.positions, slots, bt.k_cache,
                                    bt.v_cache, bt.rope_theta)
    except Exception:
        return
    written = oracle.brute_kv_append(bt.k.tolist(), bt.v.tolist(), bt.positions.tolist(),
                                     slots.tolist(), bt.k_cache, bt.v_cache, bt.rope_theta)
    touched = np.zeros(bt.k_cache.shape[:3], dtype=bool)
    ok = True
    for (blk, off, h), (krot, vbits) in written.items():
        touched[blk, off, h] = True
        got = oracle.bf16_bits_to_f64(kc[blk, off, h])
        ok &= bool(np.all(np.abs(got - np.array(krot)) <= 2.0**-7 * np.abs(krot) + 1e-30))
        ok &= bool(np.array_equal(vc[blk, off, h], np.array(vbits, dtype=np.uint16)))
    ok &= bool(np.array_equal(kc[~touched], bt.k_cache[~touched]))
    ok &= bool(np.array_equal(vc[~touched], bt.v_cache[~touched]))
    assert not ok
