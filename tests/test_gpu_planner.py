"""The work planner's counts on the GPU against the oracle's span classification.

The planner writes a small header at the start of the workspace: the number of decode
spans, the number of decode work units (page groups of 8 / Hkv pages, all kv heads), the
units per decode CTA, the number of prefill tiles and the number of split partials.  These
are fixed by the spans and context lengths alone ("09 -- Mini Inference Engine", "Week 3 --
Continuous batching": a step's batch mixes one-token decode spans with chunked-prefill
spans; "Week 4 -- Paged KV cache": a sequence of ctx tokens holds ceil(ctx / 16) blocks), so
they are compared exactly with counts taken from ``oracle.classify_spans``.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle.attention import SPAN_DECODE, SPAN_PREFILL
from paged_kv_gqa_14_gb300 import ops
from paged_kv_gqa_14_gb300 import workloads as W
from tests.gpu_util import Dev

pytestmark = pytest.mark.gpu

DECODE_WARPS = 8


def _expected(bt, decode_ctas, tile_q):
    kind, pages, spans = oracle.classify_spans(bt.query_start_loc, bt.context_lens)
    pps = DECODE_WARPS // bt.num_kv_heads
    dec = np.flatnonzero(kind == SPAN_DECODE)
    units = -(-pages[dec] // pps)
    U = int(units.sum())
    w = max(1, -(-U // decode_ctas))
    u0 = np.concatenate([[0], np.cumsum(units)[:-1]]).astype(np.int64)
    u1 = u0 + units
    slots = int(((u1 - 1) // w - u0 // w + 1).sum()) if len(dec) else 0
    tiles = int((-(-spans[kind == SPAN_PREFILL] // tile_q)).sum())
    return [len(dec), U, w, tiles, slots]


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("prefill", ["mma", "tcgen05"])
def test_planner_counts_match_oracle_classification(index, prefill):
    bt = W.config(index, poison=False)
    d = Dev(bt)
    T, hq, hd = bt.q.shape
    mb = bt.block_tables.shape[1]
    ctas = 100
    ops.set_decode_ctas(ctas)
    ops.set_prefill_kernel(prefill)
    try:
        ws = ops.alloc_workspace(T, bt.num_seqs, hq, bt.num_kv_heads, hd, mb, device=d.q.device)
        ws.fill_(0xFF)
        ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.qsl, bt.scale,
                            workspace=ws)
        torch.cuda.synchronize()
        assert ops.get_device_error() == 0
        header = ws[:20].cpu().numpy().view(np.int32)[:5].tolist()
    finally:
        ops.set_decode_ctas(0)
        ops.set_prefill_kernel("auto")
    # tcgen05 tiles stack the G q heads of a kv head: floor(128 / G) positions per tile
    tile_q = 128 // (bt.num_q_heads // bt.num_kv_heads) if prefill == "tcgen05" else 64
    assert header == _expected(bt, ctas, tile_q)


@pytest.mark.parametrize("case", ["mixed", "prefill-heavy"])
def test_split_gives_the_prefill_a_share_and_spreads_decode_units_over_the_rest(case):
    # header[5] = prefill CTAs that take items.  Beside the decode (default) the planner gives
    # the prefill P of the SMs and spreads the decode units over the other C - P; in the
    # serial order every launched prefill CTA takes items and the decode uses all C.
    if case == "mixed":
        bt = W.config(5, poison=False)
    else:  # three long chunks and three short decodes: most SMs belong to the prefill
        ctx, spans = [3000, 2500, 4096, 700, 33, 1500], [512, 1000, 700, 1, 1, 1]
        bt = W.make_batch(ctx, spans, 16, 8, 128, sum(-(-c // 16) for c in ctx) + 8, seed=11, poison=False)
    d = Dev(bt)
    T, hq, hd = bt.q.shape
    hkv = bt.num_kv_heads
    mb = bt.block_tables.shape[1]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tile_q = 128 // (hq // hkv)
    pf_grid = min((T // tile_q + bt.num_seqs + 1) * hkv, sms)
    ws = ops.alloc_workspace(T, bt.num_seqs, hq, hkv, hd, mb, device=d.q.device)
    try:
        for on in (True, False):
            ops.set_overlap(on)
            ws.fill_(0xFF)
            ops.paged_attention(d.q, d.k_cache, d.v_cache, d.block_tables, d.context_lens, d.qsl, bt.scale,
                                workspace=ws)
            torch.cuda.synchronize()
            assert ops.get_device_error() == 0
            h = ws[:24].cpu().numpy().view(np.int32)[:6].tolist()
            pn = h[5]
            if on:
                assert 1 <= pn < sms and pn <= h[3] * hkv
                assert h[:5] == _expected(bt, sms - pn, tile_q)
                if case == "prefill-heavy":
                    assert pn >= sms // 2
            else:
                assert pn == pf_grid
                assert h[:5] == _expected(bt, sms, tile_q)
    finally:
        ops.set_overlap(True)
