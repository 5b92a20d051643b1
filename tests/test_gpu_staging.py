"""One-copy input staging (``paged_kv_gqa_14_gb300.staging``) on the GPU: a step run from
the staged device views is bit-identical to the same step run from separately uploaded
tensors, and one upload moves every field."""

import numpy as np
import pytest
import torch

from paged_kv_gqa_14_gb300 import ops
from paged_kv_gqa_14_gb300 import workloads as W
from paged_kv_gqa_14_gb300.staging import StepStaging
from tests.gpu_util import Dev, dev_to_bits

pytestmark = pytest.mark.gpu


def _bf(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("index", [1, 5])
def test_staged_step_matches_unstaged_step(index):
    bt = W.config(index)
    ref = Dev(bt)
    ref.append()
    ref_out = ref.attend()

    stg = StepStaging(bt.num_tokens, bt.num_seqs, bt.num_q_heads, bt.num_kv_heads, bt.head_dim,
                      bt.block_tables.shape[1])
    assert stg.nbytes % 256 == 0
    stg.host.q.copy_(_bf(bt.q))
    stg.host.k.copy_(_bf(bt.k))
    stg.host.v.copy_(_bf(bt.v))
    stg.host.positions.copy_(torch.from_numpy(bt.positions))
    stg.host.slot_mapping.copy_(torch.from_numpy(bt.slot_mapping))
    stg.host.block_tables.copy_(torch.from_numpy(bt.block_tables))
    stg.host.context_lens.copy_(torch.from_numpy(bt.context_lens))
    stg.host.query_start_loc.copy_(torch.from_numpy(bt.query_start_loc))
    stg.upload()
    d = Dev(bt)  # fresh pool
    s = stg.dev
    ops.kv_append(s.q, s.k, s.v, s.positions, s.slot_mapping, d.k_cache, d.v_cache, bt.rope_theta)
    out = ops.paged_attention(s.q, d.k_cache, d.v_cache, s.block_tables, s.context_lens, s.query_start_loc,
                              bt.scale)
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0
    assert np.array_equal(dev_to_bits(s.q), dev_to_bits(ref.q))
    assert np.array_equal(dev_to_bits(d.k_cache), dev_to_bits(ref.k_cache))
    assert np.array_equal(dev_to_bits(d.v_cache), dev_to_bits(ref.v_cache))
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    for name in ("positions", "slot_mapping", "block_tables", "context_lens", "query_start_loc"):
        assert torch.equal(getattr(s, name).cpu(), getattr(stg.host, name)), name


@pytest.mark.parametrize("nbytes", [16, 4096, 1 << 20, (3 << 20) + 48])
def test_kernel_copy_round_trip_through_pinned_host_memory(nbytes):
    g = torch.Generator().manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g).pin_memory()
    dev = torch.full((nbytes,), 7, dtype=torch.uint8, device="cuda")
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    ops.copy(dev, src)
    ops.copy(back, dev)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), src)
    assert torch.equal(back, src)


def test_staged_upload_by_kernel_equals_copy_engine():
    bt = W.config(1)
    a = StepStaging(bt.num_tokens, bt.num_seqs, bt.num_q_heads, bt.num_kv_heads, bt.head_dim,
                    bt.block_tables.shape[1])
    b = StepStaging(bt.num_tokens, bt.num_seqs, bt.num_q_heads, bt.num_kv_heads, bt.head_dim,
                    bt.block_tables.shape[1], kernel_copy=True)
    for st in (a, b):
        st._host.zero_()  # fields not set below hold whatever the allocation held
        st.host.q.copy_(_bf(bt.q))
        st.host.block_tables.copy_(torch.from_numpy(bt.block_tables))
        st.host.query_start_loc.copy_(torch.from_numpy(bt.query_start_loc))
        st.upload()
    torch.cuda.synchronize()
    assert torch.equal(a._dev.cpu(), b._dev.cpu())

