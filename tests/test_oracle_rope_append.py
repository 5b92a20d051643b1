"""Pins for the oracle's bf16 storage, RoPE and KV append (CPU only).

Each check compares the oracle against something other than itself: exhaustive bf16
patterns, a library conversion, closed forms, invariants every rotary embedding satisfies,
and a pure-Python brute force.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_14_gb300 import workloads as W


# ----------------------------------------------------------------------------- bf16 storage
def test_bf16_roundtrip_all_finite_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_bits_to_f64(bits)
    finite = np.isfinite(vals)
    back = oracle.f64_to_bf16_bits(vals[finite])
    assert np.array_equal(back, bits[finite])
    # the infinities map back too
    inf = np.isinf(vals)
    assert np.array_equal(oracle.f64_to_bf16_bits(vals[inf]), bits[inf])


def test_bf16_rounding_matches_torch_on_fp32_values():
    # for values that fp32 holds exactly there is no double rounding, so a library
    # fp32 -> bf16 conversion (nearest-even) must agree bit for bit
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(200_000).astype(np.float32),
        (rng.standard_normal(50_000) * 1e-38).astype(np.float32),  # subnormal range
        (rng.standard_normal(50_000) * 1e30).astype(np.float32),
        np.float32([1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8, -1.0 - 2.0**-8, 3.3895314e38]),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_ties_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: the even neighbour is 1
    assert oracle.f64_to_bf16_bits(1.0 + 2.0**-8) == 0x3F80
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert oracle.f64_to_bf16_bits(1.0 + 3 * 2.0**-8) == 0x3F82
    # just above the tie rounds up
    assert oracle.f64_to_bf16_bits(1.0 + 2.0**-8 + 2.0**-30) == 0x3F81


# ----------------------------------------------------------------------------------- RoPE
def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).standard_normal((5, 3, 64))
    assert np.array_equal(oracle.rope64(x, np.zeros((5, 1)), 1e6), x)


def test_rope_matches_complex_rotation_form():
    # rotate-half RoPE is a complex multiplication of z_i = x_i + j x_{i+d/2} by
    # exp(j * pos * theta^(-2i/d)); evaluate that form with numpy's complex exp
    rng = np.random.default_rng(2)
    for d, theta in [(2, 1e4), (8, 1e4), (64, 1e6), (128, 1e6)]:
        x = rng.standard_normal((4, d))
        pos = np.array([0, 1, 37, 8191], dtype=np.float64)
        z = x[:, : d // 2] + 1j * x[:, d // 2 :]
        freq = np.exp(-np.log(theta) * (2.0 * np.arange(d // 2) / d))
        zr = z * np.exp(1j * pos[:, None] * freq[None, :])
        ref = np.concatenate([zr.real, zr.imag], axis=1)
        got = oracle.rope64(x, pos, theta)
        assert np.allclose(got, ref, rtol=0, atol=1e-11)


def test_rope_first_pair_turns_by_position_radians():
    # pair 0 has frequency theta^0 = 1: unit vector e_0 goes to (cos p, sin p) on (0, d/2)
    d = 16
    e0 = np.zeros(d)
    e0[0] = 1.0
    for p in [1, 2, 100]:
        r = oracle.rope64(e0, np.float64(p), 1e4)
        assert abs(r[0] - math.cos(p)) < 1e-15 and abs(r[d // 2] - math.sin(p)) < 1e-15
        assert np.count_nonzero(np.abs(r) > 1e-15) <= 2


def test_rope_pair_wavelengths():
    # pair i returns to its start after pos = 2*pi*theta^(2i/d): pins the exponent -2i/d
    d, theta = 32, 1e4
    rng = np.random.default_rng(3)
    x = rng.standard_normal(d)
    for i in [1, 5, 15]:
        period = 2 * math.pi * theta ** (2 * i / d)
        r = oracle.rope64(x, np.float64(period), theta)
        assert abs(r[i] - x[i]) < 1e-9 * max(1, period) and abs(r[i + d // 2] - x[i + d // 2]) < 1e-9 * max(1, period)


def test_rope_preserves_pair_norms_and_relative_position():
    rng = np.random.default_rng(4)
    d = 64
    q = rng.standard_normal(d)
    k = rng.standard_normal(d)
    rq = oracle.rope64(q, np.float64(1234), 1e6)
    half = d // 2
    assert np.allclose(rq[:half] ** 2 + rq[half:] ** 2, q[:half] ** 2 + q[half:] ** 2, atol=1e-12)
    # <R_m q, R_n k> depends on m - n only
    dots = [
        np.dot(oracle.rope64(q, np.float64(m), 1e6), oracle.rope64(k, np.float64(m - 7), 1e6))
        for m in [7, 20, 500, 4000]
    ]
    assert np.allclose(dots, dots[0], atol=1e-9)


def test_rope_matches_brute_force():
    rng = np.random.default_rng(5)
    for d in [2, 8, 64]:
        x = rng.standard_normal(d)
        for p in [0, 3, 999]:
            got = oracle.rope64(x, np.float64(p), 1e6)
            ref = oracle.brute_rope(list(x), p, 1e6)
            assert np.allclose(got, ref, atol=1e-12, rtol=0)


# ----------------------------------------------------------------------------- KV append
def _ulp_bf16(x):
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.maximum(x, 2.0**-126))
    return np.ldexp(1.0, e - 8)


@pytest.mark.parametrize("seed", range(6))
def test_kv_append_matches_brute_force(seed):
    bt = W.random_case(seed, max_ctx=40)
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping,
                                     bt.k_cache, bt.v_cache, bt.rope_theta)
    written = oracle.brute_kv_append(bt.k.tolist(), bt.v.tolist(), bt.positions.tolist(),
                                     bt.slot_mapping.tolist(), bt.k_cache, bt.v_cache, bt.rope_theta)
    touched = np.zeros(bt.k_cache.shape[:3], dtype=bool)
    for (blk, off, h), (krot, vbits) in written.items():
        touched[blk, off, h] = True
        got = oracle.bf16_bits_to_f64(kc[blk, off, h])
        # stored K is the fp64 rotation rounded once to bf16: within half an ulp
        assert np.all(np.abs(got - np.array(krot)) <= 0.5 * _ulp_bf16(krot) + 1e-300)
        assert np.array_equal(vc[blk, off, h], np.array(vbits, dtype=np.uint16))
    # every other cache row is bit-identical (NaN poison compared as bits)
    assert np.array_equal(kc[~touched], bt.k_cache[~touched])
    assert np.array_equal(vc[~touched], bt.v_cache[~touched])
    # q rotation agrees with the brute-force rotation
    q64 = oracle.bf16_bits_to_f64(bt.q)
    for t in range(bt.q.shape[0]):
        for h in range(bt.q.shape[1]):
            ref = np.array(oracle.brute_rope(list(q64[t, h]), int(bt.positions[t]), bt.rope_theta))
            got = oracle.bf16_bits_to_f64(q_rot[t, h])
            assert np.all(np.abs(got - ref) <= 0.5 * _ulp_bf16(ref) + 1e-300)


def test_kv_append_skips_negative_slots_and_keeps_position_zero_exact():
    bt = W.make_batch([1, 20], [1, 1], 4, 2, 16, 8, seed=11)
    slots = bt.slot_mapping.copy()
    slots[1] = -1
    pos = bt.positions.copy()
    pos[0] = 0
    _, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, pos, slots, bt.k_cache, bt.v_cache, 1e6)
    blk, off = divmod(int(slots[0]), 16)
    assert np.array_equal(kc[blk, off], bt.k[0])  # RoPE at position 0 is the identity
    assert np.array_equal(vc[blk, off], bt.v[0])
    # the skipped token's slot stays poisoned
    b2, o2 = divmod(int(bt.slot_mapping[1]), 16)
    assert np.array_equal(kc[b2, o2], bt.k_cache[b2, o2])
    assert np.array_equal(vc[b2, o2], bt.v_cache[b2, o2])


def test_append_then_single_key_attention_returns_v():
    # a one-token context: the appended row is the only key, so the output is that v exactly
    bt = W.make_batch([1, 1, 1], [1, 1, 1], 6, 3, 32, 5, seed=12)
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping,
                                     bt.k_cache, bt.v_cache, bt.rope_theta)
    out = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens,
                                 bt.query_start_loc, bt.scale)
    G = 2
    for t in range(3):
        for h in range(6):
            assert np.array_equal(out[t, h], oracle.bf16_bits_to_f64(bt.v[t, h // G]))


def test_positions_and_slots_on_a_hand_example():
    # block size 4; sequence 0: 6 keys, a 2-row span (positions 4, 5) in logical block 1 ->
    # physical 7; sequence 1: empty span; sequence 2: 3 keys, one decode row (position 2) in
    # logical block 0 -> physical 2; a trailing token no span covers
    tables = np.array([[3, 7], [5, -1], [2, -1]])
    pos, slots = oracle.positions_and_slots([0, 2, 2, 3], [6, 9, 3], tables, 4, 4)
    assert pos.tolist() == [4, 5, 2, 0]
    assert slots.tolist() == [7 * 4 + 0, 7 * 4 + 1, 2 * 4 + 2, -1]


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_positions_and_slots_reproduce_the_workloads(index):
    # the generator places the new tokens as a scheduler would; its explicit positions and
    # slots agree with the derivation from the tables, and every slot is inside the pool and
    # unique
    bt = W.config(index, poison=False)
    pos, slots = oracle.positions_and_slots(bt.query_start_loc, bt.context_lens, bt.block_tables,
                                            bt.block_size, bt.num_tokens)
    assert np.array_equal(pos, bt.positions) and np.array_equal(slots, bt.slot_mapping)
    assert np.all((slots >= 0) & (slots < bt.num_blocks * bt.block_size))
    assert len(set(slots.tolist())) == len(slots)


def test_positions_and_slots_follow_the_block_table_not_the_position():
    # permuting the physical blocks moves the slots with them; positions do not change
    bt = W.config(2, poison=False)
    perm = np.random.default_rng(1).permutation(bt.num_blocks)
    tables = np.where(bt.block_tables >= 0, perm[np.maximum(bt.block_tables, 0)], -1)
    pos, slots = oracle.positions_and_slots(bt.query_start_loc, bt.context_lens, tables, bt.block_size,
                                            bt.num_tokens)
    assert np.array_equal(pos, bt.positions)
    blk, off = np.divmod(bt.slot_mapping, bt.block_size)
    assert np.array_equal(slots, perm[blk] * bt.block_size + off)
