"""Pools of 8-, 32-, 64- and 128-token blocks on the GPU.

"09 -- Mini Inference Engine (The Capstone)", "Design decisions you'll face": 16 tokens per
block for a first engine, the block size a tunable to measure later.  The kernels walk every
sequence in 16-token pages whatever the block size, so besides parity with the oracle (which
reads the block size off the pool's shape) the attention output must be bit-identical when
the same logical keys are stored with another block size.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_14_gb300 import ops
from paged_kv_gqa_14_gb300 import workloads as W
from tests.gpu_util import Dev, assert_close, dev_to_bits, rope_tol

pytestmark = pytest.mark.gpu

SIZES = [8, 32, 64, 128]


@pytest.fixture
def kernels():
    """Restore the process-wide kernel choices after a test that changes them."""
    yield
    ops.set_decode_kernel("auto")
    ops.set_prefill_kernel("auto")


def _oracle(bt):
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache, bt.v_cache,
                                     bt.rope_theta)
    ref = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc, bt.scale)
    return q_rot, kc, vc, ref


def _step(bt, d):
    d.append()
    out = d.attend()
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    return out


@pytest.mark.parametrize("bs", SIZES)
def test_append_places_rows_by_block_size(bs):
    bt = W.config(1, block_size=bs)
    d = Dev(bt)
    d.append()
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache, bt.v_cache,
                                     bt.rope_theta)
    assert np.array_equal(dev_to_bits(d.v_cache), vc)
    gk = dev_to_bits(d.k_cache)
    written = np.zeros(bt.k_cache.shape[:2], dtype=bool)
    for s in bt.slot_mapping:
        written[s // bs, s % bs] = True
    assert np.array_equal(gk[~written], kc[~written])
    kref = oracle.bf16_bits_to_f64(kc[written])
    kgot = oracle.bf16_bits_to_f64(gk[written])
    src = {int(s): t for t, s in enumerate(bt.slot_mapping)}
    order = [src[b * bs + o] for b, o in zip(*np.nonzero(written))]
    assert np.all(np.abs(kgot - kref) <= rope_tol(bt.k[order], kref))


@pytest.mark.parametrize("bs", SIZES)
@pytest.mark.parametrize("index", [1, 2])
def test_step_matches_oracle(bs, index):
    bt = W.config(index, block_size=bs)
    _, _, _, ref = _oracle(bt)
    out = _step(bt, Dev(bt))
    assert_close(out.float().cpu().numpy(), ref, f"config {index}, block size {bs}")


@pytest.mark.parametrize("bs", [8, 32])
@pytest.mark.parametrize("decode", ["simt", "tensor"])
@pytest.mark.parametrize("prefill", ["mma", "tcgen05"])
@pytest.mark.parametrize("seed", range(4))
def test_random_mixed_batches(bs, decode, prefill, seed, kernels):
    ops.set_decode_kernel(decode)
    ops.set_prefill_kernel(prefill)
    bt = W.random_case(seed + 300, max_seqs=6, max_ctx=300, head_dims=(64, 128), groups=(1, 2, 4, 7),
                       kv_heads=(1, 2, 4, 8), block_size=bs)
    if bt.q.shape[1] // bt.num_kv_heads > 8 or 8 % bt.num_kv_heads:
        pytest.skip("head counts outside the supported set")
    _, _, _, ref = _oracle(bt)
    out = _step(bt, Dev(bt))
    assert_close(out.float().cpu().numpy(), ref, f"seed {seed}, block size {bs}")


def _repack(bt, bs, seed):
    """The same logical keys and values stored in a pool of ``bs``-token blocks."""
    rng = np.random.default_rng(seed)
    B = bt.num_seqs
    ctx = bt.context_lens.astype(np.int64)
    nblk = -(-ctx // bs)
    width = max(1, -(-int(bt.block_tables.shape[1]) * 16 // bs))
    total = int(nblk.sum()) + 3
    perm = rng.permutation(total)
    old_bs = bt.k_cache.shape[1]
    hkv, d = bt.k_cache.shape[2], bt.k_cache.shape[3]
    kc = np.full((total, bs, hkv, d), 0x7FC0, dtype=np.uint16)  # NaN everywhere unused
    vc = kc.copy()
    table = np.full((B, width), -1, dtype=np.int32)
    cur = 0
    for b in range(B):
        table[b, : nblk[b]] = perm[cur : cur + nblk[b]]
        cur += nblk[b]
        for j in range(int(ctx[b])):
            ob, oo = bt.block_tables[b, j // old_bs], j % old_bs
            nb, no = table[b, j // bs], j % bs
            kc[nb, no] = bt.k_cache[ob, oo]
            vc[nb, no] = bt.v_cache[ob, oo]
    return kc, vc, table


@pytest.mark.parametrize("bs", SIZES)
@pytest.mark.parametrize("decode", ["simt", "tensor"])
@pytest.mark.parametrize("prefill", ["mma", "tcgen05"])
def test_output_bit_identical_across_block_sizes(bs, decode, prefill, kernels):
    # keys are visited in 16-token pages and 128-key tiles whatever the block size, so the
    # arithmetic and its order are the same: the outputs must agree bit for bit
    ops.set_decode_kernel(decode)
    ops.set_prefill_kernel(prefill)
    bt = W.make_batch([1, 17, 40, 100, 257, 300, 96], [1, 1, 1, 37, 1, 130, 96], 8, 4, 128, 80, seed=7,
                      poison=False)
    base = Dev(bt)
    base.append()
    torch.cuda.synchronize()
    # move the appended pool to the host, repack it, and attend over both layouts
    bt.k_cache = dev_to_bits(base.k_cache)
    bt.v_cache = dev_to_bits(base.v_cache)
    ref = base.attend()
    kc, vc, table = _repack(bt, bs, seed=bs)
    d = Dev(bt, q=dev_to_bits(base.q), k_cache=kc, v_cache=vc)
    d.block_tables = torch.from_numpy(table).cuda()
    out = d.attend()
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("bs", SIZES)
def test_device_side_slots(bs):
    bt = W.config(5, block_size=bs)
    ref = Dev(bt)
    ref.append()
    d = Dev(bt)
    pos = torch.full((bt.num_tokens,), -7, dtype=torch.int64, device="cuda")
    slots = torch.full((bt.num_tokens,), -7, dtype=torch.int64, device="cuda")
    ops.kv_append_paged(d.q, d.k, d.v, d.block_tables, d.context_lens, d.qsl, d.k_cache, d.v_cache, bt.rope_theta,
                        positions_out=pos, slot_mapping_out=slots)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    assert np.array_equal(slots.cpu().numpy(), bt.slot_mapping)
    assert np.array_equal(pos.cpu().numpy(), bt.positions)
    for a, b in ((d.k_cache, ref.k_cache), (d.v_cache, ref.v_cache), (d.q, ref.q)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("bs", [8, 64])
def test_context_past_table_row_is_flagged(bs):
    bt = W.make_batch([5 * bs, 3], [1, 1], 4, 2, 64, 8, seed=2, block_size=bs, max_blocks_per_seq=5)
    d = Dev(bt)
    d.context_lens = torch.tensor([5 * bs + 1, 3], dtype=torch.int32, device="cuda")
    ops.get_device_error()
    d.attend()
    assert ops.get_device_error() & 0x8
