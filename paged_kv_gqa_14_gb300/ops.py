"""Python binding with the C-ABI's names: argument marshalling only.

Every function here checks dtypes/devices, turns torch tensors into pointers, sizes and
element strides, and calls the matching ``pkv_*`` entry point on the current torch CUDA
stream.  No arithmetic of the path runs in Python or torch: all of it is in the kernels.
PyTorch supplies device memory (the output and workspace buffers) and the stream.
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib

BLOCK_SIZE = 16  # the pool's default block size
SUPPORTED_BLOCK_SIZES = (8, 16, 32, 64, 128)


# The current stream's raw handle without building a torch.cuda.Stream object (about 0.1 us
# instead of 3 us per call on the Grace host); torch.cuda.current_stream() where torch lacks it.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream_ptr(stream):
    if stream is None and _raw_stream is not None and _cur_device is not None:
        return ctypes.c_void_p(_raw_stream(_cur_device()))
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, ndim):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def _rows(t, name):
    """(token stride, head stride) of a [T, H, d] tensor whose last dim is contiguous."""
    if t.stride(2) != 1:
        raise ValueError(f"{name}: head_dim must be contiguous")
    return t.stride(0), t.stride(1)


def _contig1(t, name):
    if t.dim() != 1 or (t.numel() > 1 and t.stride(0) != 1):
        raise ValueError(f"{name} must be a contiguous 1-D tensor")


def kv_append(q, k, v, positions, slot_mapping, k_cache, v_cache, rope_theta, stream=None):
    """Fused RoPE + KV append (``pkv_kv_append``).  q is rotated in place."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(positions, "positions", torch.int64, 1)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _contig1(positions, "positions")
    _contig1(slot_mapping, "slot_mapping")
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("k_cache / v_cache must be contiguous [num_blocks, block_size, Hkv, d]")
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache differ in shape")
    T, hq, d = q.shape
    nb, bs, hkv, dc = k_cache.shape
    if k.shape != (T, hkv, d) or v.shape != (T, hkv, d) or dc != d:
        raise ValueError("k / v / cache shapes disagree with q")
    if positions.shape[0] != T or slot_mapping.shape[0] != T:
        raise ValueError("positions / slot_mapping must have num_tokens entries")
    qs, qh = _rows(q, "q")
    ks, kh = _rows(k, "k")
    vs, vh = _rows(v, "v")
    st = _lib.load().pkv_kv_append(
        q.data_ptr(), qs, qh, k.data_ptr(), ks, kh, v.data_ptr(), vs, vh,
        positions.data_ptr(), slot_mapping.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        T, hq, hkv, d, nb, bs, float(rope_theta), _stream_ptr(stream))
    _lib.check("pkv_kv_append", st)


def kv_append_paged(q, k, v, block_tables, context_lens, query_start_loc, k_cache, v_cache, rope_theta,
                    positions_out=None, slot_mapping_out=None, max_blocks_per_seq=None, stream=None):
    """kv_append with positions and slots derived on the GPU from the scheduler's tables
    (``pkv_kv_append_paged``).  q is rotated in place."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(query_start_loc, "query_start_loc", torch.int32, 1)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _contig1(context_lens, "context_lens")
    _contig1(query_start_loc, "query_start_loc")
    if block_tables.stride(1) != 1:
        raise ValueError("block_tables rows must be contiguous")
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("k_cache / v_cache must be contiguous [num_blocks, block_size, Hkv, d]")
    T, hq, d = q.shape
    nb, bs, hkv, dc = k_cache.shape
    if k.shape != (T, hkv, d) or v.shape != (T, hkv, d) or dc != d or v_cache.shape != k_cache.shape:
        raise ValueError("k / v / cache shapes disagree with q")
    B = context_lens.shape[0]
    if query_start_loc.shape[0] != B + 1 or block_tables.shape[0] != B:
        raise ValueError("query_start_loc must have num_seqs + 1 entries, block_tables num_seqs rows")
    for name, t in (("positions_out", positions_out), ("slot_mapping_out", slot_mapping_out)):
        if t is not None:
            _need(t, name, torch.int64, 1)
            _contig1(t, name)
            if t.shape[0] != T:
                raise ValueError(f"{name} must have num_tokens entries")
    mb = block_tables.shape[1] if max_blocks_per_seq is None else int(max_blocks_per_seq)
    qs, qh = _rows(q, "q")
    ks, kh = _rows(k, "k")
    vs, vh = _rows(v, "v")
    st = _lib.load().pkv_kv_append_paged(
        q.data_ptr(), qs, qh, k.data_ptr(), ks, kh, v.data_ptr(), vs, vh, block_tables.data_ptr(),
        block_tables.stride(0), mb, context_lens.data_ptr(), query_start_loc.data_ptr(), B, k_cache.data_ptr(),
        v_cache.data_ptr(), T, hq, hkv, d, nb, bs, float(rope_theta),
        None if positions_out is None else positions_out.data_ptr(),
        None if slot_mapping_out is None else slot_mapping_out.data_ptr(), _stream_ptr(stream))
    _lib.check("pkv_kv_append_paged", st)


def rope_turn_table(rope_theta, head_dim):
    """The rotation frequencies kv_append uses, as uint64 0.64 fixed-point turn fractions
    (``pkv_rope_turn_table``; host only, no GPU)."""
    import numpy as np

    out = (ctypes.c_uint64 * (int(head_dim) // 2 or 1))()
    _lib.check("pkv_rope_turn_table", _lib.load().pkv_rope_turn_table(float(rope_theta), int(head_dim), out))
    return np.frombuffer(out, dtype=np.uint64)[: int(head_dim) // 2].copy()


def workspace_size(num_tokens, num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, decode_ctas=0):
    """Bytes of workspace ``paged_attention`` needs (``pkv_paged_attention_workspace_size_ex``;
    ``decode_ctas`` as the per-call option, 0 for the process default)."""
    n = _lib.load().pkv_paged_attention_workspace_size_ex(num_tokens, num_seqs, num_q_heads, num_kv_heads,
                                                          head_dim, max_blocks_per_seq, int(decode_ctas))
    if n == 0:
        raise ValueError("invalid sizes for paged_attention")
    return int(n)


def alloc_workspace(num_tokens, num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                    device=None, decode_ctas=0):
    """A caller-owned workspace tensor (uint8) of the required size on `device` (default: the
    current CUDA device); torch's caching allocator returns 512-byte aligned blocks."""
    n = workspace_size(num_tokens, num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, decode_ctas)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


_OVERLAP = {None: 0, True: 1, False: 2}
PLAN_EARLY = 1  # PKV_ATTN_PLAN_EARLY
STREAM_EARLY = 2  # PKV_ATTN_STREAM_EARLY


STREAM_EARLY_MIN_KEYS = 1 << 17


def stream_early_pays(num_seqs, max_blocks_per_seq, block_size):
    """Whether PKV_ATTN_STREAM_EARLY is worth setting for a batch of this size: the decode then
    reads the plan through a published word, one round trip to L2 later than through the
    planner's end, which costs about 1 us on a batch that is latency-bound anyway and is repaid
    once the pages a decode CTA can copy during the append dominate (append + attention step on
    one GB300: 32 sequences of up to 1152 keys, L2 flushed, 20.1 -> 21.2 us; 256 of up to 2048,
    156.2 -> 154.0 us; 50 of 8192, 133.9 -> 132.5 us).  The rule: at least STREAM_EARLY_MIN_KEYS
    key slots in the block tables."""
    return num_seqs * max_blocks_per_seq * block_size >= STREAM_EARLY_MIN_KEYS


def attention_options(options):
    """A pkv_attention_options from a dict (build it once and pass it to every call):
    decode_kernel ('auto' | 'simt' | 'tensor'), prefill_kernel ('auto' | 'mma' | 'tcgen05'),
    overlap (None | True | False), decode_ctas (int), plan_early (bool: PKV_ATTN_PLAN_EARLY),
    stream_early (bool: PKV_ATTN_STREAM_EARLY; both flags are defined in include/pkv.h),
    side_stream (torch.cuda.Stream) with fork_event and join_event (torch.cuda.Event)."""
    if options is None or isinstance(options, _lib.AttentionOptions):
        return options  # (a struct built earlier is passed through: no per-call marshalling)
    unknown = set(options) - {"decode_kernel", "prefill_kernel", "overlap", "decode_ctas", "plan_early",
                              "stream_early", "side_stream", "fork_event", "join_event"}
    if unknown:
        raise ValueError(f"unknown options {sorted(unknown)}")
    opt = _lib.AttentionOptions()
    opt.struct_size = ctypes.sizeof(_lib.AttentionOptions)
    opt.decode_kernel = DECODE_KERNELS[options.get("decode_kernel", "auto")]
    opt.prefill_kernel = PREFILL_KERNELS[options.get("prefill_kernel", "auto")]
    opt.overlap = _OVERLAP[options.get("overlap", None)]
    opt.decode_ctas = int(options.get("decode_ctas", 0))
    opt.flags = (PLAN_EARLY if options.get("plan_early", False) else 0) | (
        STREAM_EARLY if options.get("stream_early", False) else 0)
    side = options.get("side_stream")
    if side is not None:
        fork, join = options.get("fork_event"), options.get("join_event")
        for ev in (fork, join):  # torch creates an event's CUDA handle at its first record
            if ev is not None and not ev.cuda_event:
                ev.record(side)
        opt.side_stream = ctypes.c_void_p(side.cuda_stream)
        opt.fork_event = ctypes.c_void_p(fork.cuda_event) if fork is not None else None
        opt.join_event = ctypes.c_void_p(join.cuda_event) if join is not None else None
    return opt


def paged_attention(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, scale, out=None,
                    workspace=None, max_blocks_per_seq=None, stream=None, options=None):
    """Paged GQA over a ragged prefill/decode batch (``pkv_paged_attention``, or with per-call
    ``options`` -- a dict or a struct from ``attention_options`` -- ``pkv_paged_attention_ex``).
    Returns out."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(query_start_loc, "query_start_loc", torch.int32, 1)
    _contig1(context_lens, "context_lens")
    _contig1(query_start_loc, "query_start_loc")
    if block_tables.stride(1) != 1:
        raise ValueError("block_tables rows must be contiguous")
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("k_cache / v_cache must be contiguous [num_blocks, block_size, Hkv, d]")
    T, hq, d = q.shape
    nb, bs, hkv, dc = k_cache.shape
    if dc != d or v_cache.shape != k_cache.shape:
        raise ValueError("cache shapes disagree with q")
    B = context_lens.shape[0]
    if query_start_loc.shape[0] != B + 1 or block_tables.shape[0] != B:
        raise ValueError("query_start_loc must have num_seqs + 1 entries, block_tables num_seqs rows")
    mb = block_tables.shape[1] if max_blocks_per_seq is None else int(max_blocks_per_seq)
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    _need(out, "out", torch.bfloat16, 3)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    opt = attention_options(options)
    if workspace is None:
        workspace = alloc_workspace(T, B, hq, hkv, d, mb, device=q.device,
                                    decode_ctas=opt.decode_ctas if opt is not None else 0)
    qs, qh = _rows(q, "q")
    os_, oh = _rows(out, "out")
    args = (q.data_ptr(), qs, qh, k_cache.data_ptr(), v_cache.data_ptr(), nb, bs,
            block_tables.data_ptr(), block_tables.stride(0), mb, context_lens.data_ptr(),
            query_start_loc.data_ptr(), B, out.data_ptr(), os_, oh, T, hq, hkv, d, float(scale),
            workspace.data_ptr(), workspace.numel(), _stream_ptr(stream))
    if opt is None:
        _lib.check("pkv_paged_attention", _lib.load().pkv_paged_attention(*args))
    else:
        _lib.check("pkv_paged_attention_ex", _lib.load().pkv_paged_attention_ex(*args, ctypes.byref(opt)))
    return out


def set_decode_ctas(n):
    """Override the decode split-K grid (0 = one CTA per SM).  Process-wide."""
    _lib.check("pkv_set_decode_ctas", _lib.load().pkv_set_decode_ctas(int(n)))


def set_overlap(on):
    """Run a mixed batch's prefill tiles beside the decode on a second stream (True, the
    default) or before it on the caller's stream (False).  Process-wide."""
    _lib.check("pkv_set_overlap", _lib.load().pkv_set_overlap(1 if on else 0))


DECODE_KERNELS = {"auto": 0, "simt": 1, "tensor": 2}


def set_decode_kernel(kind):
    """Decode arithmetic for later calls: "auto", "simt" (CUDA cores) or "tensor" (mma.sync)."""
    _lib.check("pkv_set_decode_kernel", _lib.load().pkv_set_decode_kernel(DECODE_KERNELS[kind]))


PREFILL_KERNELS = {"auto": 0, "mma": 1, "tcgen05": 2}


def set_prefill_kernel(kind):
    """Prefill-tile arithmetic for later calls: "auto", "mma" (mma.sync) or "tcgen05"."""
    _lib.check("pkv_set_prefill_kernel", _lib.load().pkv_set_prefill_kernel(PREFILL_KERNELS[kind]))


def set_fault_injection(kind):
    """Test only (``pkv_set_fault_injection``): ``"decode_no_copies"`` makes the decode producer
    issue nothing, so its consumers' bounded waits run out; ``"plan_no_ready"`` keeps the
    planner from publishing its ready word under ``stream_early``, so the decode's bounded polls
    run out and it falls back to the planner's end; ``None`` turns it off."""
    code = {None: 0, "decode_no_copies": 1, "plan_no_ready": 2}[kind]
    _lib.check("pkv_set_fault_injection", _lib.load().pkv_set_fault_injection(code))


def get_device_error(clear=True, stream=None):
    """Synchronise the stream and return the or-ed PKV_DEVERR_* bits of the current device."""
    bits = ctypes.c_uint32(0)
    st = _lib.load().pkv_get_device_error(ctypes.byref(bits), 1 if clear else 0, _stream_ptr(stream))
    _lib.check("pkv_get_device_error", st)
    return int(bits.value)


def set_kernel_events(kernel, start=None, stop=None):
    """Record torch.cuda.Event ``start``/``stop`` around every launch of ``kernel``
    ("kv_append", "plan", "prefill", "decode"); None switches it off."""
    which = _lib.KERNELS[kernel]
    for e in (start, stop):
        if e is not None and e.cuda_event == 0:
            e.record()  # torch creates the CUDA event lazily, on its first record
    sp = ctypes.c_void_p(start.cuda_event) if start is not None else None
    ep = ctypes.c_void_p(stop.cuda_event) if stop is not None else None
    _lib.check("pkv_set_kernel_events", _lib.load().pkv_set_kernel_events(which, sp, ep))


def copy(dst, src, stream=None):
    """Byte copy src -> dst by a kernel (``pkv_copy``); either tensor may be on the device or in
    pinned host memory.  Both must be contiguous, of equal byte size, 16-byte aligned."""
    for name, t in (("dst", dst), ("src", src)):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError("dst and src differ in byte size")
    _lib.check("pkv_copy", _lib.load().pkv_copy(dst.data_ptr(), src.data_ptr(), nbytes, _stream_ptr(stream)))
    return dst

