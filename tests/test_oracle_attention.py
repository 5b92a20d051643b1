"""Pins for the oracle's paged attention (CPU only).

The oracle is compared with a pure-Python brute force, with a library routine on the
special cases that reduce to it (decode rows and from-scratch causal prefill equal
``torch.nn.functional.scaled_dot_product_attention`` in fp64 on the contiguous K/V), and
with closed forms and invariants: paged == contiguous, physical-id permutation invariance,
single-key output == v, equal scores -> mean of V, convex hull, GQA head map, causal
alignment of a chunk over earlier context, and the log-sum-exp merge identity.
"""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_14_gb300 import workloads as W


def _appended(bt):
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping,
                                     bt.k_cache, bt.v_cache, bt.rope_theta)
    return q_rot, kc, vc


def _run(bt, q_rot, kc, vc, block_tables=None):
    return oracle.paged_attention(q_rot, kc, vc, bt.block_tables if block_tables is None else block_tables,
                                  bt.context_lens, bt.query_start_loc, bt.scale)


@pytest.mark.parametrize("seed", range(8))
def test_oracle_matches_brute_force(seed):
    bt = W.random_case(seed, max_ctx=36, head_dims=(8, 16))
    q_rot, kc, vc = _appended(bt)
    out = _run(bt, q_rot, kc, vc)
    ref = np.array(oracle.brute_paged_attention(q_rot.tolist(), kc.tolist(), vc.tolist(),
                                                bt.block_tables.tolist(), bt.context_lens.tolist(),
                                                bt.query_start_loc.tolist(), bt.scale))
    assert np.all(np.isfinite(out))  # poisoned slots were never read
    assert np.max(np.abs(out - ref)) < 1e-12


def test_tiny_decode_config_matches_brute_force():
    bt = W.config(1)
    q_rot, kc, vc = _appended(bt)
    out = _run(bt, q_rot, kc, vc)
    ref = np.array(oracle.brute_paged_attention(q_rot.tolist(), kc.tolist(), vc.tolist(),
                                                bt.block_tables.tolist(), bt.context_lens.tolist(),
                                                bt.query_start_loc.tolist(), bt.scale))
    assert np.max(np.abs(out - ref)) < 1e-12


def _sdpa64(q, k, v, causal):
    """torch SDPA in fp64: q [n, Hq, d], k/v [ctx, Hkv, d] -> [n, Hq, d]."""
    G = q.shape[1] // k.shape[1]
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(np.repeat(k, G, axis=1)).permute(1, 0, 2)[None]
    vt = torch.from_numpy(np.repeat(v, G, axis=1)).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal,
                                                         scale=float(1.0 / np.sqrt(q.shape[2])))
    return o[0].permute(1, 0, 2).numpy()


def test_decode_rows_equal_library_sdpa_on_contiguous_kv():
    bt = W.config(2)
    q_rot, kc, vc = _appended(bt)
    bt.scale = 1.0 / 8.0  # d = 64
    out = _run(bt, q_rot, kc, vc)
    for b in [0, 5, 31]:
        K, V = oracle.gather_sequence_kv(kc, vc, bt.block_tables[b], bt.context_lens[b])
        t = bt.query_start_loc[b]
        ref = _sdpa64(oracle.bf16_bits_to_f64(q_rot[t : t + 1]), K, V, causal=False)
        assert np.max(np.abs(out[t : t + 1] - ref)) < 1e-12


def test_prefill_from_empty_context_equals_library_causal_sdpa():
    # a chunk over zero earlier tokens is textbook causal attention
    bt = W.make_batch([48, 7], [48, 7], 4, 2, 32, 10, seed=21)
    q_rot, kc, vc = _appended(bt)
    out = _run(bt, q_rot, kc, vc)
    for b in range(2):
        s, e = bt.query_start_loc[b], bt.query_start_loc[b + 1]
        K, V = oracle.gather_sequence_kv(kc, vc, bt.block_tables[b], bt.context_lens[b])
        ref = _sdpa64(oracle.bf16_bits_to_f64(q_rot[s:e]), K, V, causal=True)
        assert np.max(np.abs(out[s:e] - ref)) < 1e-12


def test_block_table_permutation_invariance_and_paged_equals_contiguous():
    bt = W.make_batch([40, 70, 16], [1, 5, 1], 4, 2, 16, 12, seed=22)
    q_rot, kc, vc = _appended(bt)
    out = _run(bt, q_rot, kc, vc)
    # lay every sequence's blocks out contiguously (identity-like table) in a fresh pool
    nb = bt.block_tables.shape[1]
    B = bt.num_seqs
    kc2 = np.full((B * nb,) + kc.shape[1:], W.NAN_BF16, dtype=np.uint16)
    vc2 = kc2.copy()
    bt2 = np.full_like(bt.block_tables, -1)
    for b in range(B):
        pages = -(-int(bt.context_lens[b]) // 16)
        for j in range(pages):
            kc2[b * nb + j] = kc[bt.block_tables[b, j]]
            vc2[b * nb + j] = vc[bt.block_tables[b, j]]
            bt2[b, j] = b * nb + j
    out2 = _run(bt, q_rot, kc2, vc2, block_tables=bt2)
    assert np.array_equal(out, out2)
    # and under a further random relabelling of the physical ids
    perm = np.random.default_rng(0).permutation(kc2.shape[0])
    kc3 = np.empty_like(kc2)
    vc3 = np.empty_like(vc2)
    kc3[perm] = kc2
    vc3[perm] = vc2
    bt3 = np.where(bt2 >= 0, perm[np.maximum(bt2, 0)], -1).astype(np.int32)
    out3 = _run(bt, q_rot, kc3, vc3, block_tables=bt3)
    assert np.array_equal(out, out3)


def test_single_key_output_is_v():
    bt = W.config(1)  # sequence 0 has a one-token context
    q_rot, kc, vc = _appended(bt)
    out = _run(bt, q_rot, kc, vc)
    G = bt.num_q_heads // bt.num_kv_heads
    for h in range(bt.num_q_heads):
        assert np.array_equal(out[0, h], oracle.bf16_bits_to_f64(bt.v[0, h // G]))


def test_equal_scores_give_mean_of_visible_values():
    bt = W.make_batch([33, 50], [1, 6], 4, 2, 16, 9, seed=23)
    q_rot, kc, vc = _appended(bt)
    zero_q = np.zeros_like(q_rot)
    out = _run(bt, zero_q, kc, vc)
    for b in range(2):
        s, e = bt.query_start_loc[b], bt.query_start_loc[b + 1]
        n, ctx = e - s, bt.context_lens[b]
        K, V = oracle.gather_sequence_kv(kc, vc, bt.block_tables[b], ctx)
        for r in range(n):
            last = ctx - n + r
            for h in range(4):
                assert np.allclose(out[s + r, h], V[: last + 1, h // 2].mean(axis=0), atol=1e-13, rtol=0)


def test_convex_hull():
    for seed in range(4):
        bt = W.random_case(100 + seed, max_ctx=60)
        q_rot, kc, vc = _appended(bt)
        out = _run(bt, q_rot, kc, vc)
        G = bt.num_q_heads // bt.num_kv_heads
        for b in range(bt.num_seqs):
            s, e = bt.query_start_loc[b], bt.query_start_loc[b + 1]
            n, ctx = e - s, bt.context_lens[b]
            K, V = oracle.gather_sequence_kv(kc, vc, bt.block_tables[b], ctx)
            for r in range(n):
                vis = V[: ctx - n + r + 1]
                for h in range(bt.num_q_heads):
                    lo = vis[:, h // G].min(axis=0)
                    hi = vis[:, h // G].max(axis=0)
                    o = out[s + r, h]
                    assert np.all(o >= lo - 1e-12) and np.all(o <= hi + 1e-12)


def test_gqa_head_map_is_contiguous_groups():
    # V of kv head j is the constant vector (j+1); q head h must output h // G + 1
    bt = W.make_batch([20, 37], [1, 3], 6, 3, 16, 8, seed=24)
    q_rot, kc, vc = _appended(bt)
    vc2 = vc.copy()
    for j in range(3):
        vc2[:, :, j, :] = oracle.f64_to_bf16_bits(np.full(16, j + 1.0))
    out = _run(bt, q_rot, kc, vc2)
    for h in range(6):
        assert np.allclose(out[:, h, :], h // 2 + 1.0, atol=1e-13)


def test_causal_alignment_of_chunk_over_earlier_context():
    # V rows are one-hot by key position and q = 0: row r of an n-row span over a context
    # of ctx keys must weight keys 0 .. ctx-n+r equally and every later key by exactly 0
    ctx, n, d = 29, 5, 32
    bt = W.make_batch([ctx], [n], 2, 1, d, 3, seed=25)
    q_rot, kc, vc = _appended(bt)
    vc2 = vc.copy()
    for j in range(ctx):
        blk = bt.block_tables[0, j // 16]
        onehot = np.zeros(d)
        onehot[j] = 1.0
        vc2[blk, j % 16, 0] = oracle.f64_to_bf16_bits(onehot)
    out = _run(bt, np.zeros_like(q_rot), kc, vc2)
    for r in range(n):
        last = ctx - n + r
        expect = np.zeros(d)
        expect[: last + 1] = 1.0 / (last + 1)
        for h in range(2):
            assert np.allclose(out[r, h], expect, atol=1e-15, rtol=0)


def test_scale_is_applied_to_scores():
    # doubling q (exact in bf16) and halving the scale leaves the output unchanged
    bt = W.make_batch([45], [3], 2, 1, 16, 4, seed=26)
    q_rot, kc, vc = _appended(bt)
    out = _run(bt, q_rot, kc, vc)
    q2 = oracle.f64_to_bf16_bits(2.0 * oracle.bf16_bits_to_f64(q_rot))
    out2 = oracle.paged_attention(q2, kc, vc, bt.block_tables, bt.context_lens,
                                  bt.query_start_loc, bt.scale / 2)
    assert np.max(np.abs(out - out2)) < 1e-14
    # and a different scale really changes it
    out3 = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens,
                                  bt.query_start_loc, bt.scale * 3)
    assert np.max(np.abs(out - out3)) > 1e-3


def test_merge_of_split_partials_equals_full_softmax():
    bt = W.config(2)
    q_rot, kc, vc = _appended(bt)
    out = _run(bt, q_rot, kc, vc)
    rng = np.random.default_rng(27)
    for b in [1, 7]:
        ctx = int(bt.context_lens[b])
        K, V = oracle.gather_sequence_kv(kc, vc, bt.block_tables[b], ctx)
        cuts = np.sort(rng.choice(np.arange(1, ctx), size=4, replace=False))
        edges = [0, *cuts.tolist(), ctx]
        t = bt.query_start_loc[b]
        for h in [0, 13]:
            qv = oracle.bf16_bits_to_f64(q_rot[t, h])
            parts = [oracle.attention_partial(qv, K[a:z, h // 7], V[a:z, h // 7], bt.scale)
                     for a, z in zip(edges[:-1], edges[1:])]
            merged = oracle.merge_partials([p[0] for p in parts], [p[1] for p in parts],
                                           [p[2] for p in parts])
            assert np.max(np.abs(merged - out[t, h])) < 1e-13


def test_classify_spans():
    kind, pages, spans = oracle.classify_spans([0, 1, 1, 9, 10], [17, 4, 40, 16])
    assert kind.tolist() == [oracle.attention.SPAN_DECODE, oracle.attention.SPAN_NONE,
                             oracle.attention.SPAN_PREFILL, oracle.attention.SPAN_DECODE]
    assert pages.tolist() == [2, 0, 3, 1]
    assert spans.tolist() == [1, 0, 8, 1]


def test_uncovered_rows_stay_nan():
    bt = W.make_batch([10, 12], [1, 1], 2, 1, 8, 4, seed=28)
    q_rot, kc, vc = _appended(bt)
    # sequence 1 gets an empty span: row 1 belongs to nobody
    qsl = np.array([0, 1, 1], dtype=np.int32)
    out = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, qsl, bt.scale)
    assert np.all(np.isfinite(out[0])) and np.all(np.isnan(out[1]))


@pytest.mark.parametrize("bs", [8, 32, 64, 128])
def test_block_size_does_not_change_the_result(bs):
    # "09 -- Mini Inference Engine (The Capstone)", "Week 4": a sequence's keys are its blocks'
    # rows in table order, so the same keys stored in blocks of another size give the same
    # attention (exactly: the oracle gathers the same fp64 values in the same order)
    bt = W.make_batch([1, 17, 40, 100, 130], [1, 1, 1, 37, 1], 4, 2, 16, 40, seed=3, poison=False)
    ref = oracle.paged_attention(bt.q, bt.k_cache, bt.v_cache, bt.block_tables, bt.context_lens,
                                 bt.query_start_loc, bt.scale)
    rng = np.random.default_rng(bs)
    ctx = bt.context_lens.astype(np.int64)
    nblk = -(-ctx // bs)
    total = int(nblk.sum()) + 2
    perm = rng.permutation(total)
    kc = np.full((total, bs) + bt.k_cache.shape[2:], 0x7FC0, dtype=np.uint16)  # NaN where unused
    vc = kc.copy()
    table = np.full((bt.num_seqs, int(nblk.max())), -1, dtype=np.int32)
    cur = 0
    for b in range(bt.num_seqs):
        table[b, : nblk[b]] = perm[cur : cur + nblk[b]]
        cur += nblk[b]
        for j in range(int(ctx[b])):
            kc[table[b, j // bs], j % bs] = bt.k_cache[bt.block_tables[b, j // 16], j % 16]
            vc[table[b, j // bs], j % bs] = bt.v_cache[bt.block_tables[b, j // 16], j % 16]
    got = oracle.paged_attention(bt.q, kc, vc, table, bt.context_lens, bt.query_start_loc, bt.scale)
    assert np.array_equal(got, ref)


def test_workload_block_size_variant_is_consistent():
    # a workload rebuilt over 32-token blocks: slots point into the tables, tables stay inside
    # the pool, and the pool keeps its size in tokens
    for bs in (8, 32):
        bt = W.config(1, block_size=bs, poison=False)
        base = W.config(1, poison=False)
        assert bt.k_cache.shape[1] == bs
        assert bt.num_blocks * bs == base.num_blocks * 16
        for t, (pos, s) in enumerate(zip(bt.positions, bt.slot_mapping)):
            b = int(np.searchsorted(bt.query_start_loc, t, side="right") - 1)
            assert s == bt.block_tables[b, pos // bs] * bs + pos % bs
        assert bt.block_tables.max() < bt.num_blocks
