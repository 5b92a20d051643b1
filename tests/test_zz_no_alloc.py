"""The no-allocation entry point, pkv_paged_attention_noalloc, on the GPU.

It exists for callers that must not call cudaMalloc (their device memory belongs to a host
framework, or their serving loop keeps allocation out of the step).  Its scratch is a fixed
16 MiB array inside the library instead of a caller workspace.  This test calls it through
the C ABI and checks, on two calls in a row (the second one finds the first call's leftovers
in the shared array), that its output matches the regular entry point's within the
attention tolerance used by the other tests.  It also checks that sizes needing more
scratch than the array holds are refused.  The file sorts last so that a run stopping at the
first failure has already run every other test; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

from paged_kv_gqa_14_gb300 import _lib
from paged_kv_gqa_14_gb300 import build as B
from paged_kv_gqa_14_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def _dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _args(bt, d, out):
    T, hq, hd = bt.q.shape
    return [d["q"].data_ptr(), d["q"].stride(0), d["q"].stride(1), d["kc"].data_ptr(), d["vc"].data_ptr(),
            bt.num_blocks, 16, d["bt"].data_ptr(), d["bt"].stride(0), bt.block_tables.shape[1],
            d["ctx"].data_ptr(), d["qsl"].data_ptr(), bt.num_seqs, out.data_ptr(), out.stride(0),
            out.stride(1), T, hq, bt.num_kv_heads, hd, ctypes.c_float(bt.scale)]


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.fixture(scope="module")
def lib():
    B.build()
    return _lib.load()


@pytest.mark.parametrize("index", [1, 5])
def test_noalloc_matches_regular_entry_point_twice(lib, index):
    bt = W.config(index, poison=False)
    bits = ctypes.c_uint32(0)
    assert lib.pkv_get_device_error(ctypes.byref(bits), 1, _stream()) == 0  # start from a clear word
    d = {"q": _dev_bf16(bt.q), "kc": _dev_bf16(bt.k_cache), "vc": _dev_bf16(bt.v_cache),
         "bt": torch.from_numpy(bt.block_tables).cuda(), "ctx": torch.from_numpy(bt.context_lens).cuda(),
         "qsl": torch.from_numpy(bt.query_start_loc).cuda()}
    T, hq, hd = bt.q.shape
    # the regular entry point with a caller-owned workspace
    ws_bytes = lib.pkv_paged_attention_workspace_size(T, bt.num_seqs, hq, bt.num_kv_heads, hd,
                                                      bt.block_tables.shape[1])
    assert 0 < ws_bytes <= 16 << 20
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ref = torch.empty_like(d["q"])
    st = lib.pkv_paged_attention(*_args(bt, d, ref), ws.data_ptr(), ws_bytes, _stream())
    assert st == 0, _lib.STATUS.get(st)
    torch.cuda.synchronize()
    ref_f = ref.float().cpu().numpy()
    assert np.all(np.isfinite(ref_f))
    # the no-allocation entry point, two calls in a row into fresh outputs
    for call in range(2):
        out = torch.full_like(d["q"], float("nan"))
        st = lib.pkv_paged_attention_noalloc(*_args(bt, d, out), _stream())
        assert st == 0, _lib.STATUS.get(st)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        err = np.abs(got - ref_f)
        assert np.all(np.isfinite(got)), f"call {call}: non-finite output"
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, f"call {call}: max {err.max()} mean {err.mean()}"
    bits = ctypes.c_uint32(0)
    assert lib.pkv_get_device_error(ctypes.byref(bits), 1, _stream()) == 0
    assert bits.value == 0


def test_noalloc_refuses_sizes_beyond_its_scratch(lib):
    # 10^6 sequences need far more than 16 MiB of split states: refused before any launch
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    st = lib.pkv_paged_attention_noalloc(x.data_ptr(), 1024, 128, x.data_ptr(), x.data_ptr(), 10, 16,
                                         x.data_ptr(), 8, 8, x.data_ptr(), x.data_ptr(), 1_000_000,
                                         x.data_ptr(), 1024, 128, 1_000_000, 8, 4, 128, ctypes.c_float(0.1),
                                         _stream())
    assert st == 6  # PKV_ERR_WORKSPACE
