"""paged_attention on the GPU against the fp64 oracle (max abs <= 2e-2, mean abs <= 2e-3),
on all five workloads at full size, random mixed micro-batches over every supported
shape, and the properties that hold at any size."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_14_gb300 import ops
from paged_kv_gqa_14_gb300 import workloads as W
from tests.gpu_util import (Dev, assert_close, bf16_to_dev, config_with_oracle, dev_to_bits, idx_to_dev)

pytestmark = pytest.mark.gpu


def _attend_oracle_inputs(bt, q_rot, kc, vc):
    d = Dev(bt, q=q_rot, k_cache=kc, v_cache=vc)
    out = d.attend()
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    return out.float().cpu().numpy(), d


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_attention_matches_oracle_on_workloads(index):
    bt, q_rot, kc, vc, ref = config_with_oracle(index)
    got, _ = _attend_oracle_inputs(bt, q_rot, kc, vc)
    assert_close(got, ref, bt.name)


@pytest.mark.parametrize("index", [1, 3, 5])
def test_full_step_append_then_attention(index):
    bt, q_rot, kc, vc, ref = config_with_oracle(index)
    d = Dev(bt)
    d.append()
    out = d.attend()
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    assert_close(out.float().cpu().numpy(), ref, bt.name + " (append + attention)")


@pytest.mark.parametrize("seed", range(12))
def test_random_mixed_batches(seed):
    bt = W.random_case(seed, max_seqs=6, max_ctx=300, head_dims=(64, 128), groups=(1, 2, 3, 4, 5, 6, 7, 8),
                       kv_heads=(1, 2, 4, 8))
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache,
                                     bt.v_cache, bt.rope_theta)
    ref = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc, bt.scale)
    got, _ = _attend_oracle_inputs(bt, q_rot, kc, vc)
    assert_close(got, ref, bt.name)


@pytest.fixture
def decode_kernel(request):
    ops.set_decode_kernel(request.param)
    yield request.param
    ops.set_decode_kernel("auto")


@pytest.mark.parametrize("decode_kernel", ["simt", "tensor"], indirect=True)
@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_both_decode_kernels_match_oracle(index, decode_kernel):
    bt, q_rot, kc, vc, ref = config_with_oracle(index)
    got, _ = _attend_oracle_inputs(bt, q_rot, kc, vc)
    assert_close(got, ref, f"{bt.name} decode={decode_kernel}")


@pytest.mark.parametrize("decode_kernel", ["simt", "tensor"], indirect=True)
@pytest.mark.parametrize("seed", range(100, 112))
def test_both_decode_kernels_random_shapes(seed, decode_kernel):
    bt = W.random_case(seed, max_seqs=8, max_ctx=400, head_dims=(64, 128), groups=(1, 2, 3, 4, 5, 6, 7, 8),
                       kv_heads=(1, 2, 4, 8), allow_prefill=False)
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache,
                                     bt.v_cache, bt.rope_theta)
    ref = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc, bt.scale)
    for ctas in (0, 3):
        ops.set_decode_ctas(ctas)
        try:
            got, _ = _attend_oracle_inputs(bt, q_rot, kc, vc)
        finally:
            ops.set_decode_ctas(0)
        assert_close(got, ref, f"{bt.name} decode={decode_kernel} ctas={ctas}")


@pytest.fixture
def prefill_kernel(request):
    ops.set_prefill_kernel(request.param)
    yield request.param
    ops.set_prefill_kernel("auto")


@pytest.mark.parametrize("prefill_kernel", ["mma", "tcgen05"], indirect=True)
def test_both_prefill_kernels_on_mixed_workload(prefill_kernel):
    bt, q_rot, kc, vc, ref = config_with_oracle(5)
    got, _ = _attend_oracle_inputs(bt, q_rot, kc, vc)
    assert_close(got, ref, f"{bt.name} prefill={prefill_kernel}")


@pytest.mark.parametrize("prefill_kernel", ["mma", "tcgen05"], indirect=True)
@pytest.mark.parametrize("case", [
    ([300, 40, 129], [300, 40, 129], 16, 8, 128),     # from-scratch chunks: ragged q tiles
    ([1000, 700, 2], [260, 129, 2], 16, 8, 128),      # chunks over earlier context, tiny span
    ([513, 64, 200], [257, 64, 1], 8, 8, 64),         # d 64, G 1, a decode row mixed in
    ([900, 333], [200, 333], 28, 4, 128),             # G 7
])
def test_both_prefill_kernels_on_long_chunks(prefill_kernel, case):
    ctx, spans, hq, hkv, d = case
    pages = sum(-(-c // 16) for c in ctx)
    bt = W.make_batch(ctx, spans, hq, hkv, d, pages + 5, seed=hash(tuple(ctx)) % 1000)
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache,
                                     bt.v_cache, bt.rope_theta)
    ref = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc, bt.scale)
    got, _ = _attend_oracle_inputs(bt, q_rot, kc, vc)
    assert_close(got, ref, f"prefill={prefill_kernel} ctx={ctx} spans={spans}")


@pytest.mark.parametrize("prefill_kernel", ["tcgen05"], indirect=True)
@pytest.mark.parametrize("group", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("d", [64, 128])
def test_tcgen05_prefill_every_group_size(prefill_kernel, group, d):
    # the tcgen05 tile stacks the G q heads of a kv head (floor(128 / G) positions x G rows):
    # every G, ragged tiles at both ends of a chunk, a second kv head, a decode row mixed in
    ctx, spans = [431, 150, 77], [301, 150, 1]
    pages = sum(-(-c // 16) for c in ctx)
    bt = W.make_batch(ctx, spans, 2 * group, 2, d, pages + 3, seed=70 + group)
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache,
                                     bt.v_cache, bt.rope_theta)
    ref = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc, bt.scale)
    got, _ = _attend_oracle_inputs(bt, q_rot, kc, vc)
    assert_close(got, ref, f"G={group} d={d}")


@pytest.mark.parametrize("prefill_kernel", ["mma", "tcgen05"], indirect=True)
@pytest.mark.parametrize("seed", range(200, 210))
def test_both_prefill_kernels_random_mixed(seed, prefill_kernel):
    bt = W.random_case(seed, max_seqs=5, max_ctx=500, head_dims=(64, 128), groups=(1, 2, 4, 7),
                       kv_heads=(1, 2, 4, 8))
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache,
                                     bt.v_cache, bt.rope_theta)
    ref = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc, bt.scale)
    got, _ = _attend_oracle_inputs(bt, q_rot, kc, vc)
    assert_close(got, ref, f"{bt.name} prefill={prefill_kernel}")


@pytest.mark.parametrize("ctas", [1, 7, 600])
def test_split_count_does_not_change_the_result(ctas):
    bt, q_rot, kc, vc, ref = config_with_oracle(3)
    auto, d = _attend_oracle_inputs(bt, q_rot, kc, vc)
    try:
        ops.set_decode_ctas(ctas)
        forced = d.attend().float().cpu().numpy()
    finally:
        ops.set_decode_ctas(0)
    assert_close(forced, ref, f"decode ctas={ctas}")
    assert np.abs(forced - auto).max() <= 2e-2


def test_physical_block_permutation_is_bit_identical():
    bt, q_rot, kc, vc, _ = config_with_oracle(2)
    got, _ = _attend_oracle_inputs(bt, q_rot, kc, vc)
    perm = np.random.default_rng(0).permutation(bt.num_blocks)
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = W.Batch(**{**bt.__dict__})
    bt2.block_tables = np.where(bt.block_tables >= 0, perm[np.maximum(bt.block_tables, 0)], -1).astype(np.int32)
    got2, _ = _attend_oracle_inputs(bt2, q_rot, kc2, vc2)
    assert np.array_equal(got, got2)


def test_single_key_context_returns_v_exactly():
    bt, q_rot, kc, vc, _ = config_with_oracle(1)  # sequence 0 has context 1
    _, d = _attend_oracle_inputs(bt, q_rot, kc, vc)
    out = dev_to_bits(d.attend())
    G = bt.num_q_heads // bt.num_kv_heads
    for h in range(bt.num_q_heads):
        assert np.array_equal(out[0, h], bt.v[0, h // G])


def test_last_prefill_row_equals_decode_at_same_context():
    # a 40-row chunk over 100 earlier tokens vs a one-row decode of its last token
    bt = W.make_batch([140], [40], 16, 8, 128, 12, seed=31)
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache,
                                     bt.v_cache, bt.rope_theta)
    pf, _ = _attend_oracle_inputs(bt, q_rot, kc, vc)
    bt_dec = W.Batch(**{**bt.__dict__})
    bt_dec.query_start_loc = np.array([0, 1], dtype=np.int32)
    dec, _ = _attend_oracle_inputs(bt_dec, q_rot[-1:], kc, vc)
    assert np.abs(pf[-1] - dec[0]).max() <= 2e-2


def test_empty_spans_and_uncovered_rows_are_untouched():
    bt = W.make_batch([30, 50, 20, 70], [1, 0, 5, 1], 8, 2, 64, 16, seed=32)
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache,
                                     bt.v_cache, bt.rope_theta)
    ref = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc, bt.scale)
    # one extra trailing row that no span covers
    q_ext = np.concatenate([q_rot, q_rot[:1]])
    d = Dev(bt, q=q_ext, k_cache=kc, v_cache=vc)
    sentinel = torch.full((bt.num_tokens + 1, 8, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    d.attend(out=sentinel)
    torch.cuda.synchronize()
    got = sentinel.float().cpu().numpy()
    assert_close(got[:-1], ref, "empty spans")
    assert np.all(got[-1] == 7.0)


def test_attention_on_strided_q_and_out():
    bt, q_rot, kc, vc, ref = config_with_oracle(1)
    T, hq, d = q_rot.shape
    wide = np.zeros((T, hq + 3, d), dtype=np.uint16)
    wide[:, 1 : hq + 1] = q_rot
    dd = Dev(bt, q=q_rot, k_cache=kc, v_cache=vc)
    qw = bf16_to_dev(wide)[:, 1 : hq + 1]
    outw = torch.zeros((T, hq + 2, d), dtype=torch.bfloat16, device="cuda")
    ops.paged_attention(qw, dd.k_cache, dd.v_cache, dd.block_tables, dd.context_lens, dd.qsl, bt.scale,
                        out=outw[:, 2:])
    assert_close(outw[:, 2:].float().cpu().numpy(), ref, "strided")
    assert torch.all(outw[:, :2] == 0)


def test_device_errors_are_flagged_not_faulted():
    bt = W.make_batch([30, 50, 20], [1, 1, 1], 8, 4, 128, 10, seed=33)
    d = Dev(bt)
    d.append()
    ops.get_device_error()  # clear
    bad = bt.block_tables.copy()
    bad[1, 1] = 10_000  # outside the pool: read redirected, bit set
    d.block_tables = idx_to_dev(bad)
    d.attend()
    torch.cuda.synchronize()
    assert ops.get_device_error() & 0x2
    d.block_tables = idx_to_dev(bt.block_tables)
    ctx = bt.context_lens.copy()
    ctx[2] = bt.block_tables.shape[1] * 16 + 1  # longer than its block-table row
    d.context_lens = idx_to_dev(ctx)
    d.attend()
    torch.cuda.synchronize()
    assert ops.get_device_error() & 0x8
    d.context_lens = idx_to_dev(bt.context_lens)
    qsl = bt.query_start_loc.copy()
    qsl[2] = qsl[1] - 1 if qsl[1] > 0 else 0  # non-monotone
    qsl[1] = qsl[1] + 1
    d.qsl = idx_to_dev(qsl.astype(np.int32))
    d.attend()
    torch.cuda.synchronize()
    assert ops.get_device_error() & 0x4
    # the context is still usable
    d.qsl = idx_to_dev(bt.query_start_loc)
    d.attend()
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0


def test_nan_poisoned_slots_never_leak():
    # every workload is generated with NaN in all unreferenced slots; full-size outputs are finite
    bt, q_rot, kc, vc, _ = config_with_oracle(5)
    got, _ = _attend_oracle_inputs(bt, q_rot, kc, vc)
    assert np.all(np.isfinite(got))


def test_cuda_graph_replay_matches_eager_step():
    # append + attention captured once in a CUDA graph: no host sync or allocation inside the
    # library, so replay reproduces the eager step bit for bit
    bt, _, _, _, ref = config_with_oracle(5)
    eager = Dev(bt)
    eager.append()
    out_e = eager.attend()
    d = Dev(bt)
    q_in = d.q.clone()
    out = torch.empty_like(d.q)
    ws = ops.alloc_workspace(bt.num_tokens, bt.num_seqs, bt.num_q_heads, bt.num_kv_heads, bt.head_dim,
                             bt.block_tables.shape[1])
    d.append()  # first calls do the one-time per-device set-up outside the capture
    d.q.copy_(q_in)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ops.kv_append(d.q, d.k, d.v, d.positions, d.slots, d.k_cache, d.v_cache, bt.rope_theta)
        ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.qsl, bt.scale,
                            out=out, workspace=ws)
    for _ in range(2):
        d.q.copy_(q_in)
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out_e.view(torch.int16))
    assert_close(out.float().cpu().numpy(), ref, "graph replay")


@pytest.mark.parametrize("prefill_kernel", ["mma", "tcgen05"], indirect=True)
@pytest.mark.parametrize("bs", [16, 128])
def test_long_contexts_and_largest_group(prefill_kernel, bs):
    # the largest shapes of the supported set: G = 8 (16 q / 2 kv heads), d 128, a 32768-token
    # decode context, a 1000-token chunk over 19000 earlier keys, a single-key sequence
    ctx, spans = [32768, 20000, 1], [1, 1000, 1]
    pages = sum(-(-c // bs) for c in ctx)
    bt = W.make_batch(ctx, spans, 16, 2, 128, pages + 4, seed=77, block_size=bs)
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache,
                                     bt.v_cache, bt.rope_theta)
    ref = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc, bt.scale)
    got, _ = _attend_oracle_inputs(bt, q_rot, kc, vc)
    assert_close(got, ref, f"long contexts, block size {bs}, prefill={prefill_kernel}")


@pytest.fixture
def overlap_setting():
    yield
    ops.set_overlap(True)


@pytest.mark.parametrize("case", ["mixed", "random", "prefill-heavy", "prefill-only"])
def test_prefill_beside_decode_matches_serial_order(case, overlap_setting):
    # the prefill tiles on their own share of the SMs (second stream) or before the decode on
    # all of them: the same per-item arithmetic, so the prefill rows agree bit for bit; the
    # decode rows are cut at other split points, so both are held to the oracle
    if case == "mixed":
        bt, q_rot, kc, vc, ref = config_with_oracle(5)
    else:
        if case == "random":
            ctx, spans = [40, 700, 1, 300, 2048, 64, 900], [40, 200, 1, 1, 130, 1, 1]
        elif case == "prefill-heavy":  # most SMs go to the prefill; three decodes
            ctx, spans = [3000, 2500, 4096, 700, 33, 1500], [512, 1000, 700, 1, 1, 1]
        else:  # no decode units at all
            ctx, spans = [800, 1200, 65], [800, 300, 65]
        pages = sum(-(-c // 16) for c in ctx)
        bt = W.make_batch(ctx, spans, 16, 8, 128, pages + 8, seed=11)
        q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache,
                                         bt.v_cache, bt.rope_theta)
        ref = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc,
                                     bt.scale)
    outs = {}
    for on in (True, False):
        ops.set_overlap(on)
        got, _ = _attend_oracle_inputs(bt, q_rot, kc, vc)
        assert_close(got, ref, f"{bt.name}, prefill beside decode {on}")
        outs[on] = got
    qsl = bt.query_start_loc
    rows = np.concatenate([np.arange(qsl[b], qsl[b + 1]) for b in range(bt.num_seqs) if qsl[b + 1] - qsl[b] > 1])
    assert len(rows) > 0
    assert np.array_equal(outs[True][rows], outs[False][rows])


def _visible_rows(bt):
    """(row, sequence, last visible key) for every row a span covers."""
    out = []
    qsl, ctx = bt.query_start_loc, bt.context_lens
    for b in range(bt.num_seqs):
        n = int(qsl[b + 1] - qsl[b])
        for r in range(n):
            out.append((int(qsl[b]) + r, b, int(ctx[b]) - n + r))
    return out


@pytest.mark.parametrize("prefill_kernel", ["mma", "tcgen05"], indirect=True)
def test_zero_query_gives_mean_of_visible_values(prefill_kernel):
    # q = 0: every visible key scores 0, so each row is the plain mean of the V rows it sees
    # (a decode row: the whole context; prefill row r of n: keys 0 .. ctx - n + r), on both
    # the decode and the prefill kernels, across page and tile boundaries
    ctx, spans = [1, 17, 300, 140, 64, 2100], [1, 1, 1, 40, 64, 300]
    pages = sum(-(-c // 16) for c in ctx)
    bt = W.make_batch(ctx, spans, 16, 8, 128, pages + 4, seed=41)
    _, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache, bt.v_cache,
                                 bt.rope_theta)
    q0 = np.zeros_like(bt.q)
    got, _ = _attend_oracle_inputs(bt, q0, kc, vc)
    G = bt.num_q_heads // bt.num_kv_heads
    ref = np.empty_like(got, dtype=np.float64)
    for row, b, last in _visible_rows(bt):
        _, V = oracle.gather_sequence_kv(kc, vc, bt.block_tables[b], int(bt.context_lens[b]))
        mean = V[: last + 1].mean(axis=0)  # [Hkv, d]
        ref[row] = np.repeat(mean, G, axis=0)
    assert_close(got, ref, f"q = 0, prefill={prefill_kernel}")


def test_outputs_lie_in_the_convex_hull_of_visible_values():
    # a softmax-weighted average: every output coordinate lies between the smallest and the
    # largest value of that V column over the keys the row sees (up to the bf16 rounding of the
    # output and fp32 accumulation: one bf16 ulp of the bound plus 1e-3)
    bt, q_rot, kc, vc, _ = config_with_oracle(5)
    got, _ = _attend_oracle_inputs(bt, q_rot, kc, vc)
    G = bt.num_q_heads // bt.num_kv_heads
    cache = {}
    worst = 0.0
    for row, b, last in _visible_rows(bt):
        if b not in cache:
            cache[b] = oracle.gather_sequence_kv(kc, vc, bt.block_tables[b], int(bt.context_lens[b]))[1]
        V = cache[b][: last + 1]
        lo = np.repeat(V.min(axis=0), G, axis=0)
        hi = np.repeat(V.max(axis=0), G, axis=0)
        slack = 1e-3 + np.maximum(np.abs(lo), np.abs(hi)) * 2.0**-8
        worst = max(worst, float(np.max(lo - got[row])), float(np.max(got[row] - hi)))
        assert np.all(got[row] >= lo - slack) and np.all(got[row] <= hi + slack), f"row {row}"
    assert worst <= 1e-2


def test_bounded_wait_runs_out_and_reports_timeout():
    # failure detection without a GPU fault: with the test-only fault injection the decode's
    # producer warp issues no copy and no barrier arrival, so its consumers' bounded waits run
    # out (about 2^31 SM clocks); the kernel sets PKV_DEVERR_TIMEOUT and finishes with nothing
    # in flight, and the next call on the same context is correct again
    import time

    bt, q_rot, kc, vc, ref = config_with_oracle(1)
    d = Dev(bt, q=q_rot, k_cache=kc, v_cache=vc)
    d.attend()
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    ops.set_fault_injection("decode_no_copies")
    try:
        t0 = time.perf_counter()
        d.attend()
        torch.cuda.synchronize()
        waited = time.perf_counter() - t0
    finally:
        ops.set_fault_injection(None)
    assert ops.get_device_error() == 0x10  # PKV_DEVERR_TIMEOUT, nothing else
    assert 0.2 < waited < 60.0
    got = d.attend().float().cpu().numpy()
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    assert_close(got, ref, "after a timed-out call")


@pytest.mark.parametrize("decode_kernel", ["simt", "tensor"], indirect=True)
@pytest.mark.parametrize("case", [
    ([40, 300, 17, 64], [0, 3, 0, 1]),   # as many tokens as sequences: a 3-row span beside empty ones
    ([50, 129, 33], [2, 0, 0]),          # fewer tokens than sequences
    ([2000, 5], [2, 0]),                 # a long context
])
def test_prefill_rows_without_more_tokens_than_sequences(case, decode_kernel):
    # num_tokens <= num_seqs: no prefill kernel is launched; the planner turns each row of a
    # longer span into a decode entry that sees its own causal context (keys 0 .. ctx - n + r)
    ctx, spans = case
    pages = sum(-(-c // 16) for c in ctx)
    bt = W.make_batch(ctx, spans, 16, 8, 128, pages + 4, seed=sum(ctx))
    assert bt.num_tokens <= bt.num_seqs
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache,
                                     bt.v_cache, bt.rope_theta)
    ref = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc, bt.scale)
    got, d = _attend_oracle_inputs(bt, q_rot, kc, vc)
    assert_close(got, ref, f"rows in the decode path, {case}, decode={decode_kernel}")
    # the plan: one decode entry per row, no prefill work entries
    ws = ops.alloc_workspace(bt.num_tokens, bt.num_seqs, bt.num_q_heads, bt.num_kv_heads, bt.head_dim,
                             bt.block_tables.shape[1])
    ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.qsl, bt.scale, workspace=ws)
    torch.cuda.synchronize()
    header = ws[:16].cpu().numpy().view(np.int32)[:4].tolist()
    assert header[0] == sum(spans) and header[3] == 0


@pytest.mark.parametrize("opts", [
    {"decode_kernel": "simt"}, {"decode_kernel": "tensor", "decode_ctas": 7},
    {"prefill_kernel": "mma"}, {"overlap": False}, {"overlap": True, "prefill_kernel": "tcgen05"},
])
def test_per_call_options_equal_the_process_settings(opts, overlap_setting):
    # pkv_paged_attention_ex: the same kernels and split as the process-wide settings give
    bt, q_rot, kc, vc, ref = config_with_oracle(5)
    d = Dev(bt, q=q_rot, k_cache=kc, v_cache=vc)
    got = ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.qsl, bt.scale,
                              options=opts)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    try:
        if "decode_kernel" in opts:
            ops.set_decode_kernel(opts["decode_kernel"])
        if "prefill_kernel" in opts:
            ops.set_prefill_kernel(opts["prefill_kernel"])
        if "overlap" in opts:
            ops.set_overlap(opts["overlap"])
        if "decode_ctas" in opts:
            ops.set_decode_ctas(opts["decode_ctas"])
        want = d.attend()
        torch.cuda.synchronize()
    finally:
        ops.set_decode_kernel("auto")
        ops.set_prefill_kernel("auto")
        ops.set_decode_ctas(0)
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    assert_close(got.float().cpu().numpy(), ref, f"options {opts}")


@pytest.mark.parametrize("index", [3, 5])
def test_early_planner_gives_the_same_plan(index):
    # PKV_ATTN_PLAN_EARLY after the step's kv_append (the use it is meant for): the same plan,
    # so the same kernels and bit-identical rows, and the oracle's result
    bt = W.config(index)
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache, bt.v_cache,
                                     bt.rope_theta)
    ref = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc, bt.scale)
    outs = []
    for opts in (None, {"plan_early": True}):
        d = Dev(bt)
        d.append()
        outs.append(ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.qsl, bt.scale,
                                        options=opts))
        torch.cuda.synchronize()
        assert ops.get_device_error() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert_close(outs[1].float().cpu().numpy(), ref, "early planner")


@pytest.mark.parametrize("index,block_size,overlap", [(1, 16, None), (2, 16, None), (3, 16, None), (4, 16, None),
                                                      (5, 16, None), (5, 16, False), (3, 8, None), (5, 128, None)])
def test_early_streaming_gives_the_same_rows(index, block_size, overlap):
    # PKV_ATTN_STREAM_EARLY right after the step's kv_append: the decode copies the pages without
    # a new key while the append may still run; the rows are bit-identical to the plain call's
    # and match the oracle, over three steps back to back (in the serial order, overlap False,
    # the prefill kernel sits between the planner and the decode)
    bt = W.config(index, block_size=block_size)
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache, bt.v_cache,
                                     bt.rope_theta)
    ref = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc, bt.scale)
    outs = []
    for opts in ({"overlap": overlap}, {"overlap": overlap, "stream_early": True}):
        d = Dev(bt)
        for _ in range(3):
            d.q.copy_(bf16_to_dev(bt.q))
            d.append()
            got = ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.qsl, bt.scale,
                                      options=opts)
        torch.cuda.synchronize()
        assert ops.get_device_error() == 0
        outs.append(got)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert_close(outs[1].float().cpu().numpy(), ref, "early streaming")


def test_early_streaming_with_rows_of_longer_spans():
    # no more tokens than sequences but some spans of two or three rows: their rows are decode
    # entries whose new keys start before their last page, so the decode waits before any page
    ctx = [40, 33, 17, 64, 5, 100, 16, 31]
    spans = [2, 0, 1, 3, 0, 1, 0, 1]
    bt = W.make_batch(ctx, spans, 8, 2, 64, 64, seed=5)
    assert bt.num_tokens <= bt.num_seqs
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache, bt.v_cache,
                                     bt.rope_theta)
    ref = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc, bt.scale)
    outs = []
    for opts in (None, {"stream_early": True}):
        d = Dev(bt)
        d.append()
        outs.append(ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.qsl, bt.scale,
                                        options=opts))
        torch.cuda.synchronize()
        assert ops.get_device_error() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert_close(outs[1].float().cpu().numpy(), ref, "early streaming, longer spans")


@pytest.mark.parametrize("decode_kernel", ["simt", "tensor"])
def test_early_streaming_with_either_decode_kernel(decode_kernel):
    # the CUDA-core decode ignores the ready word and waits for the planner's end; the
    # tensor-core one streams early: both give the rows of the plain call on the mixed batch
    bt = W.config(5)
    outs = []
    for opts in ({"decode_kernel": decode_kernel}, {"decode_kernel": decode_kernel, "stream_early": True}):
        d = Dev(bt)
        d.append()
        outs.append(ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.qsl, bt.scale,
                                        options=opts))
        torch.cuda.synchronize()
        assert ops.get_device_error() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_early_streaming_falls_back_when_the_plan_is_never_published():
    # the test-only fault keeps the planner from publishing its ready word: every decode CTA's
    # bounded poll runs out (2^24 SM clocks) and it waits for the planner's end instead, so the
    # call is slower but its rows are the plain call's, with no device error
    import time

    bt = W.config(3)
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache, bt.v_cache,
                                     bt.rope_theta)
    d = Dev(bt, q=q_rot, k_cache=kc, v_cache=vc)
    want = d.attend().clone()
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    ops.set_fault_injection("plan_no_ready")
    try:
        t0 = time.perf_counter()
        got = ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.qsl, bt.scale,
                                  options={"stream_early": True})
        torch.cuda.synchronize()
        waited = time.perf_counter() - t0
    finally:
        ops.set_fault_injection(None)
    assert ops.get_device_error() == 0
    assert waited > 2e-3  # the polls ran out (about 8 ms at 2 GHz)
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_early_streaming_step_in_a_cuda_graph():
    # the append + attention step captured with PKV_ATTN_STREAM_EARLY replays like eager
    bt = W.config(3)
    d = Dev(bt)
    opts = ops.attention_options({"stream_early": True})
    out = torch.empty_like(d.q)
    ws = ops.alloc_workspace(bt.num_tokens, bt.num_seqs, bt.num_q_heads, bt.num_kv_heads, bt.head_dim,
                             bt.block_tables.shape[1], device=d.q.device)
    q0 = d.q.clone()

    def step():
        d.q.copy_(q0)
        d.append()
        ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.qsl, bt.scale, out=out,
                            workspace=ws, options=opts)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    want = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert ops.get_device_error() == 0
        assert torch.equal(out.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("flags", [{}, {"plan_early": True}, {"stream_early": True}])
def test_more_sequences_than_planner_threads(flags):
    # 1500 one-row spans: the multi-pass planner (the early flags are ignored there)
    rng = np.random.default_rng(11)
    ctx = rng.integers(1, 200, size=1500)
    pages = int(sum(-(-int(c) // 16) for c in ctx))
    bt = W.make_batch(ctx, [1] * 1500, 4, 2, 64, pages + 4, seed=11)
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache, bt.v_cache,
                                     bt.rope_theta)
    ref = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc, bt.scale)
    d = Dev(bt, q=q_rot, k_cache=kc, v_cache=vc)
    got = ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.qsl, bt.scale,
                              options=flags)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    assert_close(got.float().cpu().numpy(), ref, "1500 sequences")


def test_caller_side_stream_gives_the_same_result():
    # the prefill beside the decode on the caller's own second stream and events
    bt, q_rot, kc, vc, ref = config_with_oracle(5)
    d = Dev(bt, q=q_rot, k_cache=kc, v_cache=vc)
    lib_side = d.attend()
    side = torch.cuda.Stream()
    opts = {"side_stream": side, "fork_event": torch.cuda.Event(), "join_event": torch.cuda.Event()}
    own_side = ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.qsl, bt.scale,
                                   options=opts)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    assert torch.equal(own_side.view(torch.int16), lib_side.view(torch.int16))
    assert_close(own_side.float().cpu().numpy(), ref, "caller side stream")


def test_eager_call_on_another_stream_while_a_capture_is_open():
    # a capture of stream A pulls the library's second stream into its graph until the capture
    # ends; an eager call on stream B meanwhile must not use it (it runs in the serial order)
    bt, q_rot, kc, vc, ref = config_with_oracle(5)
    d = Dev(bt, q=q_rot, k_cache=kc, v_cache=vc)
    d.attend()  # one-time per-device set-up outside the capture
    mk = lambda: ops.alloc_workspace(bt.num_tokens, bt.num_seqs, bt.num_q_heads, bt.num_kv_heads,  # noqa: E731
                                     bt.head_dim, bt.block_tables.shape[1])
    ws_a, ws_b = mk(), mk()
    out_a, out_b = torch.empty_like(d.q), torch.full_like(d.q, float("nan"))
    other = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.qsl, bt.scale,
                            out=out_a, workspace=ws_a)
        with torch.cuda.stream(other):
            ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.qsl, bt.scale,
                                out=out_b, workspace=ws_b)
    torch.cuda.synchronize()
    assert_close(out_b.float().cpu().numpy(), ref, "eager call during another stream's capture")
    g.replay()
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    assert_close(out_a.float().cpu().numpy(), ref, "captured call")
