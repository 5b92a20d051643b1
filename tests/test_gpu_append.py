"""kv_append on the GPU against the fp64 oracle: bit-exact slot placement and V copy,
untouched rows bit-unchanged (NaN poison included), rotated K and q within one bf16 ulp
plus the fp32 rotation's absolute error (``tests.gpu_util.rope_tol``)."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_14_gb300 import ops
from paged_kv_gqa_14_gb300 import workloads as W
from tests.gpu_util import Dev, bf16_to_dev, dev_to_bits, idx_to_dev, rope_tol

pytestmark = pytest.mark.gpu


def _check_append(bt, d):
    d.append()
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache,
                                     bt.v_cache, bt.rope_theta)
    gk = dev_to_bits(d.k_cache)
    gv = dev_to_bits(d.v_cache)
    # V: every row bit-identical (written rows are copies, the rest untouched)
    assert np.array_equal(gv, vc)
    # K: untouched rows bit-identical; written rows within the rotation tolerance (one bf16
    # ulp, plus the fp32 absolute error where the rotation cancels)
    written = np.zeros(bt.k_cache.shape[:2], dtype=bool)
    src = {}
    for t, s in enumerate(bt.slot_mapping):
        if s >= 0:
            written[s // 16, s % 16] = True
            src[(s // 16, s % 16)] = t
    assert np.array_equal(gk[~written], kc[~written])
    rows = sorted(src)
    kref = oracle.bf16_bits_to_f64(np.stack([kc[r] for r in rows]))
    kgot = oracle.bf16_bits_to_f64(np.stack([gk[r] for r in rows]))
    kin = np.stack([bt.k[src[r]] for r in rows])
    assert np.all(np.abs(kgot - kref) <= rope_tol(kin, kref))
    qgot = oracle.bf16_bits_to_f64(dev_to_bits(d.q))
    qref = oracle.bf16_bits_to_f64(q_rot)
    assert np.all(np.abs(qgot - qref) <= rope_tol(bt.q, qref))
    return (kgot != kref).mean()


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_append_matches_oracle_on_workloads(index):
    bt = W.config(index)
    frac_off = _check_append(bt, Dev(bt))
    assert frac_off < 0.01  # 1-ulp differences are rare rounding ties, not a pattern


@pytest.mark.parametrize("d,theta", [(128, 1.0e6), (64, 1.0e4), (64, 0.5), (128, 0.1)])
def test_append_large_positions(d, theta):
    # positions up to 2^24: the kernel takes each angle modulo one turn in 64-bit fixed point;
    # the oracle's fp64 angle is exact to p f_i 2^-53 rad there (2^-28 for f_i <= 1; a base
    # below one turns a pair by up to 1 / theta rad per position: under 2^-25 at theta 0.1), well
    # inside the rotation tolerance
    bt = W.make_batch([3] * 16, [1] * 16, 16, 8 if d == 128 else 4, d, 20, seed=21, rope_theta=theta)
    bt.positions = np.array([0, 1, 2, 31, 999, 1000, 65535, 65536, 123457, 1_000_003, 4_000_037,
                             2**22 + 3, 7_777_777, 2**23 - 1, 2**24 - 5, 2**24], dtype=np.int64)
    _check_append(bt, Dev(bt))


@pytest.mark.parametrize("seed", range(6))
def test_append_random_shapes(seed):
    bt = W.random_case(seed, head_dims=(64, 128), groups=(1, 2, 3, 7), kv_heads=(1, 2, 4, 8))
    _check_append(bt, Dev(bt))


@pytest.mark.parametrize("d,hq,hkv", [(128, 16, 8), (64, 14, 2), (128, 28, 4)])
def test_append_large_step_matches_oracle(d, hq, hkv):
    # 3000 new tokens in one step (about 20 per SM), every 97th a padding token with slot -1
    rng = np.random.default_rng(d + hq)
    ctx = rng.integers(1, 40, size=3000)
    pages = int(sum(-(-int(c) // 16) for c in ctx))
    bt = W.make_batch(ctx, [1] * 3000, hq, hkv, d, pages + 2, seed=d + hq)
    bt.slot_mapping = bt.slot_mapping.copy()
    bt.slot_mapping[::97] = -1
    _check_append(bt, Dev(bt))


def test_append_skips_negative_slots_and_flags_out_of_range():
    bt = W.make_batch([5, 20, 33, 2], [1, 1, 1, 1], 8, 4, 128, 12, seed=3)
    slots = bt.slot_mapping.copy()
    slots[1] = -1  # padding token
    slots[2] = 12 * 16 + 5  # past the pool: must be skipped and flagged
    d = Dev(bt)
    d.slots = idx_to_dev(slots)
    ops.get_device_error()  # clear
    d.append()
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0x1
    gk, gv = dev_to_bits(d.k_cache), dev_to_bits(d.v_cache)
    for t in (1, 2):
        b, o = divmod(int(bt.slot_mapping[t]), 16)
        assert np.array_equal(gk[b, o], bt.k_cache[b, o])
        assert np.array_equal(gv[b, o], bt.v_cache[b, o])
    for t in (0, 3):
        b, o = divmod(int(slots[t]), 16)
        assert np.array_equal(gv[b, o], bt.v[t])


def test_append_position_zero_is_exact_copy():
    bt = W.make_batch([1, 1], [1, 1], 4, 2, 64, 4, seed=9)
    d = Dev(bt)
    d.append()
    gk = dev_to_bits(d.k_cache)
    for t in range(2):
        b, o = divmod(int(bt.slot_mapping[t]), 16)
        assert np.array_equal(gk[b, o], bt.k[t])
    assert np.array_equal(dev_to_bits(d.q), bt.q)


@pytest.mark.parametrize("index", [1, 3, 5])
def test_append_with_device_side_slots_matches_explicit_slots(index):
    # positions and slots derived on the GPU from the tables equal the scheduler's, and the
    # caches and q come out bit-identical to the explicit-slot call
    bt = W.config(index)
    ref = Dev(bt)
    ref.append()
    d = Dev(bt)
    pos = torch.full((bt.num_tokens,), -7, dtype=torch.int64, device="cuda")
    slots = torch.full((bt.num_tokens,), -7, dtype=torch.int64, device="cuda")
    ops.kv_append_paged(d.q, d.k, d.v, d.block_tables, d.context_lens, d.qsl, d.k_cache, d.v_cache,
                        bt.rope_theta, positions_out=pos, slot_mapping_out=slots)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    want_pos, want_slots = oracle.positions_and_slots(bt.query_start_loc, bt.context_lens, bt.block_tables,
                                                      bt.block_size, bt.num_tokens)
    assert np.array_equal(pos.cpu().numpy(), want_pos)
    assert np.array_equal(slots.cpu().numpy(), want_slots)
    for a, b in ((d.k_cache, ref.k_cache), (d.v_cache, ref.v_cache), (d.q, ref.q)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_device_side_slots_skip_tokens_outside_spans():
    bt = W.make_batch([20, 33, 5, 90], [3, 0, 5, 1], 8, 4, 64, 16, seed=14)
    T = bt.num_tokens
    # two extra trailing tokens that no span covers
    q = np.concatenate([bt.q, bt.q[:2]])
    k = np.concatenate([bt.k, bt.k[:2]])
    v = np.concatenate([bt.v, bt.v[:2]])
    d = Dev(bt)
    d.q, d.k, d.v = bf16_to_dev(q), bf16_to_dev(k), bf16_to_dev(v)
    pos = torch.zeros(T + 2, dtype=torch.int64, device="cuda")
    slots = torch.zeros(T + 2, dtype=torch.int64, device="cuda")
    ops.kv_append_paged(d.q, d.k, d.v, d.block_tables, d.context_lens, d.qsl, d.k_cache, d.v_cache,
                        bt.rope_theta, positions_out=pos, slot_mapping_out=slots)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    want_pos, want_slots = oracle.positions_and_slots(bt.query_start_loc, bt.context_lens, bt.block_tables,
                                                      bt.block_size, T + 2)
    assert np.array_equal(slots.cpu().numpy(), want_slots)
    assert np.array_equal(pos.cpu().numpy(), want_pos)
    assert np.all(slots.cpu().numpy()[T:] == -1)
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache, bt.v_cache,
                                     bt.rope_theta)
    assert np.array_equal(dev_to_bits(d.v_cache), vc)


def test_append_reads_strided_views_of_a_packed_qkv_buffer():
    bt = W.make_batch([17, 40, 3], [1, 1, 1], 16, 8, 128, 10, seed=4)
    T, hq, hkv, dd = bt.num_tokens, 16, 8, 128
    packed = np.zeros((T, (hq + 2 * hkv) * dd), dtype=np.uint16)
    packed[:, : hq * dd] = bt.q.reshape(T, -1)
    packed[:, hq * dd : (hq + hkv) * dd] = bt.k.reshape(T, -1)
    packed[:, (hq + hkv) * dd :] = bt.v.reshape(T, -1)
    P = bf16_to_dev(packed)
    q = P[:, : hq * dd].view(T, hq, dd)
    k = P[:, hq * dd : (hq + hkv) * dd].view(T, hkv, dd)
    v = P[:, (hq + hkv) * dd :].view(T, hkv, dd)
    d = Dev(bt)
    ops.kv_append(q, k, v, d.positions, d.slots, d.k_cache, d.v_cache, bt.rope_theta)
    ref = Dev(bt)
    ref.append()
    assert torch.equal(d.k_cache.view(torch.int16), ref.k_cache.view(torch.int16))
    assert torch.equal(d.v_cache.view(torch.int16), ref.v_cache.view(torch.int16))
    assert torch.equal(q.contiguous().view(torch.int16), ref.q.view(torch.int16))
    # k and v inside the packed buffer are untouched
    assert np.array_equal(dev_to_bits(P)[:, hq * dd :], packed[:, hq * dd :])
