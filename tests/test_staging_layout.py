"""The one-copy step staging layout (``paged_kv_gqa_14_gb300.staging.layout``), on CPU:
every field starts on a 256-byte boundary, fields do not overlap, each holds exactly its
shape's bytes, and a field's offset is a multiple of its element size (so the typed views of
the byte buffer are legal)."""

import pytest
import torch

from paged_kv_gqa_14_gb300.staging import layout


@pytest.mark.parametrize("sizes", [(1, 1, 1, 1, 64, 1), (256, 256, 16, 8, 128, 128), (2248, 204, 16, 8, 128, 128),
                                   (7, 3, 28, 4, 64, 513), (0, 0, 8, 8, 128, 1)])
def test_fields_are_aligned_disjoint_and_sized(sizes):
    T, B, hq, hkv, d, mb = sizes
    fields, total = layout(T, B, hq, hkv, d, mb)
    assert [f[0] for f in fields] == ["q", "k", "v", "positions", "slot_mapping", "block_tables", "context_lens",
                                      "query_start_loc"]
    expect = {"q": (T, hq, d), "k": (T, hkv, d), "v": (T, hkv, d), "positions": (T,), "slot_mapping": (T,),
              "block_tables": (B, mb), "context_lens": (B,), "query_start_loc": (B + 1,)}
    end = 0
    for name, dtype, shape, off, nbytes in fields:
        assert shape == expect[name]
        esize = torch.empty((), dtype=dtype).element_size()
        n = 1
        for x in shape:
            n *= x
        assert nbytes == n * esize
        assert off % 256 == 0 and off >= end
        end = off + nbytes
    assert total % 256 == 0 and total >= end
