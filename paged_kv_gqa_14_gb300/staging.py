"""Per-step input staging: every host input of one step in one pinned buffer, one copy up.

A serving loop produces each step's inputs on the host: the new tokens' q, k and v, their
positions and slots, and the scheduler's block tables, context lengths and span offsets.
Sent as eight tensors that is eight host-to-device copies, each with its own launch
latency.  ``StepStaging`` lays all of them out in one pinned host buffer and a device
buffer of the same layout (each region 256-byte aligned), hands out typed views of both,
and moves the whole step with a single ``cudaMemcpyAsync``.  The device views are what
``ops.kv_append`` and ``ops.paged_attention`` take.  Layout only: no arithmetic here.
"""

from __future__ import annotations

import torch

_ALIGN = 256

# name -> (dtype, shape builder from the sizes)
_FIELDS = (
    ("q", torch.bfloat16, lambda s: (s["T"], s["hq"], s["d"])),
    ("k", torch.bfloat16, lambda s: (s["T"], s["hkv"], s["d"])),
    ("v", torch.bfloat16, lambda s: (s["T"], s["hkv"], s["d"])),
    ("positions", torch.int64, lambda s: (s["T"],)),
    ("slot_mapping", torch.int64, lambda s: (s["T"],)),
    ("block_tables", torch.int32, lambda s: (s["B"], s["max_blocks"])),
    ("context_lens", torch.int32, lambda s: (s["B"],)),
    ("query_start_loc", torch.int32, lambda s: (s["B"] + 1,)),
)


def layout(num_tokens, num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq):
    """[(name, dtype, shape, byte offset, bytes)] of one step's fields, and the total bytes.

    Fields are packed in ``_FIELDS`` order, each starting on a 256-byte boundary."""
    sizes = {"T": int(num_tokens), "B": int(num_seqs), "hq": int(num_q_heads), "hkv": int(num_kv_heads),
             "d": int(head_dim), "max_blocks": int(max_blocks_per_seq)}
    out = []
    off = 0
    for name, dtype, shape_of in _FIELDS:
        shape = shape_of(sizes)
        n = 1
        for x in shape:
            n *= x
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        out.append((name, dtype, shape, off, nbytes))
        off = (off + nbytes + _ALIGN - 1) // _ALIGN * _ALIGN
    return out, off


class StepStaging:
    """Pinned host and device buffers for one step's inputs, with views of each field.

    ``host.<name>`` and ``dev.<name>`` are tensors of the field's dtype and shape:
    q [T, Hq, d], k and v [T, Hkv, d] (bf16); positions and slot_mapping [T] (int64);
    block_tables [B, max_blocks], context_lens [B], query_start_loc [B + 1] (int32).
    """

    def __init__(self, num_tokens, num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                 device=None, kernel_copy=False):
        self.kernel_copy = bool(kernel_copy)
        fields, off = layout(num_tokens, num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq)
        self.nbytes = off
        self._host = torch.empty(off, dtype=torch.uint8).pin_memory()
        self._dev = torch.empty(off, dtype=torch.uint8, device=device or "cuda")
        self.host = _Views(self._host, fields)
        self.dev = _Views(self._dev, fields)

    def upload(self, stream=None):
        """Copy the whole staged step host -> device on ``stream`` (default: current): one
        copy-engine transfer, or with ``kernel_copy`` one copy kernel reading the pinned
        buffer directly (``ops.copy``)."""
        s = torch.cuda.current_stream() if stream is None else stream
        if self.kernel_copy:
            from . import ops

            ops.copy(self._dev, self._host, stream=s)
            return
        with torch.cuda.stream(s):
            self._dev.copy_(self._host, non_blocking=True)


class _Views:
    def __init__(self, buf, layout):
        for name, dtype, shape, off, nbytes in layout:
            setattr(self, name, buf[off : off + nbytes].view(dtype).view(shape))
