"""The no-allocation entry point, pkv_paged_attention_noalloc, on the GPU.

It exists for callers that must not call cudaMalloc (their device memory belongs to a host
framework, or their serving loop keeps allocation out of the step).  Its scratch is a fixed
16 MiB array inside the library instead of a caller workspace.  These tests call it through
the C ABI, on two calls in a row (the second one finds the first call's leftovers in the
shared array), and check that

* its output is bit-identical to the regular entry point's on the same inputs (same kernels,
  same sizes, same split of the work),
* it agrees with the fp64 oracle within the attention tolerance of the other tests,
* the largest batch whose scratch fits the array runs, and the next size up is refused.

The file sorts last so that a run stopping at the first failure has already run every other
test; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_14_gb300 import _lib
from paged_kv_gqa_14_gb300 import build as B
from paged_kv_gqa_14_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
SCRATCH_BYTES = 16 << 20  # PKV_NOALLOC_SCRATCH_BYTES


def _dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _upload(bt, q):
    return {"q": _dev_bf16(q), "kc": _dev_bf16(bt.k_cache), "vc": _dev_bf16(bt.v_cache),
            "bt": torch.from_numpy(bt.block_tables).cuda(), "ctx": torch.from_numpy(bt.context_lens).cuda(),
            "qsl": torch.from_numpy(bt.query_start_loc).cuda()}


def _args(bt, d, out):
    T, hq, hd = bt.q.shape
    return [d["q"].data_ptr(), d["q"].stride(0), d["q"].stride(1), d["kc"].data_ptr(), d["vc"].data_ptr(),
            bt.num_blocks, bt.block_size, d["bt"].data_ptr(), d["bt"].stride(0), bt.block_tables.shape[1],
            d["ctx"].data_ptr(), d["qsl"].data_ptr(), bt.num_seqs, out.data_ptr(), out.stride(0),
            out.stride(1), T, hq, bt.num_kv_heads, hd, ctypes.c_float(bt.scale)]


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ws_size(lib, bt):
    T, hq, hd = bt.q.shape
    return lib.pkv_paged_attention_workspace_size(T, bt.num_seqs, hq, bt.num_kv_heads, hd, bt.block_tables.shape[1])


def _clear_error(lib):
    bits = ctypes.c_uint32(0)
    assert lib.pkv_get_device_error(ctypes.byref(bits), 1, _stream()) == 0
    return bits.value


def _regular_and_noalloc(lib, bt, q):
    """Output of the regular entry point, then of two no-allocation calls in a row."""
    d = _upload(bt, q)
    ws_bytes = _ws_size(lib, bt)
    assert 0 < ws_bytes <= SCRATCH_BYTES
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ref = torch.full_like(d["q"], float("nan"))
    st = lib.pkv_paged_attention(*_args(bt, d, ref), ws.data_ptr(), ws_bytes, _stream())
    assert st == 0, _lib.STATUS.get(st)
    outs = []
    for _ in range(2):
        out = torch.full_like(d["q"], float("nan"))
        st = lib.pkv_paged_attention_noalloc(*_args(bt, d, out), _stream())
        assert st == 0, _lib.STATUS.get(st)
        outs.append(out)
    torch.cuda.synchronize()
    return ref, outs


@pytest.fixture(scope="module")
def lib():
    B.build()
    return _lib.load()


@pytest.mark.parametrize("index", [1, 5])
def test_noalloc_matches_regular_entry_point_and_oracle_twice(lib, index):
    bt = W.config(index)
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache, bt.v_cache,
                                     bt.rope_theta)
    want = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc, bt.scale)
    bt.k_cache, bt.v_cache = kc, vc
    _clear_error(lib)
    ref, outs = _regular_and_noalloc(lib, bt, q_rot)
    for call, out in enumerate(outs):
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"call {call}: differs from the regular entry point"
        got = out.float().cpu().numpy()
        assert np.all(np.isfinite(got)), f"call {call}: non-finite output"
        err = np.abs(got - want)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, f"call {call}: max {err.max()} mean {err.mean()}"
    assert _clear_error(lib) == 0


def _decode_batch(num_seqs, seed=3):
    # one-token spans over short contexts: 4 q heads on 1 kv head, head_dim 64
    rng = np.random.default_rng(seed)
    ctx = rng.integers(1, 33, size=num_seqs)
    pages = int(sum(-(-int(c) // 16) for c in ctx))
    return W.make_batch(ctx, [1] * num_seqs, 4, 1, 64, pages + 2, seed=seed, poison=False)


def test_noalloc_runs_at_its_limit_and_refuses_one_size_past_it(lib):
    # the split-state part of the scratch grows with the number of sequences: find the most
    # sequences whose scratch fits the 16 MiB array (for this shape, on this device)
    size = lambda n: lib.pkv_paged_attention_workspace_size(n, n, 4, 1, 64, 3)  # noqa: E731
    lo, hi = 1, 1
    while size(hi) <= SCRATCH_BYTES:
        lo, hi = hi, hi * 2
    while hi - lo > 1:
        mid = (lo + hi) // 2
        lo, hi = (mid, hi) if size(mid) <= SCRATCH_BYTES else (lo, mid)
    assert size(lo) <= SCRATCH_BYTES < size(lo + 1)
    # at the limit: runs, bit-identical to the regular entry point
    bt = _decode_batch(lo)
    assert _ws_size(lib, bt) == size(lo)
    _clear_error(lib)
    ref, outs = _regular_and_noalloc(lib, bt, bt.q)
    for out in outs:
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert np.all(np.isfinite(outs[0].float().cpu().numpy()))
    assert _clear_error(lib) == 0
    # one sequence more: refused before anything is launched, the output left as it was
    bt = _decode_batch(lo + 1)
    d = _upload(bt, bt.q)
    out = torch.full_like(d["q"], 7.0)
    assert lib.pkv_paged_attention_noalloc(*_args(bt, d, out), _stream()) == 6  # PKV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)


def test_noalloc_refuses_sizes_far_beyond_its_scratch(lib):
    # 10^6 sequences need far more than 16 MiB of split states: refused before any launch
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    st = lib.pkv_paged_attention_noalloc(x.data_ptr(), 1024, 128, x.data_ptr(), x.data_ptr(), 10, 16,
                                         x.data_ptr(), 8, 8, x.data_ptr(), x.data_ptr(), 1_000_000,
                                         x.data_ptr(), 1024, 128, 1_000_000, 8, 4, 128, ctypes.c_float(0.1),
                                         _stream())
    assert st == 6  # PKV_ERR_WORKSPACE
