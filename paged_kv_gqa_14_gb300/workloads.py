"""Seeded synthetic batches shaped like the serving workloads of the paged-KV engines.

This module only draws inputs: random values, context lengths, block assignments and the
slot/position bookkeeping a scheduler would hand to the kernels.  It holds none of the
attention or RoPE arithmetic, imports nothing from the kernels' package or from the
oracle, and is the one module both sides' callers share.

All bf16 tensors are numpy ``uint16`` bit patterns (numpy has no bf16).  Values are
standard normal, drawn in fp32 with ``numpy.random.default_rng(seed)`` and rounded to
bf16 nearest-even.  ``poison=True`` (correctness runs) fills every pool slot that no
sequence's context covers -- unreferenced blocks, the tail of each sequence's last block and
the slots the step's new tokens will be appended to -- with NaN, so that any stray read
shows up as NaN in the output.  ``poison=False`` (timing runs) leaves unreferenced blocks
zero and fills the new tokens' slots with ordinary values.

Workload shapes (page title, section):

1. tiny decode -- 4 sequences, contexts {1, 17, 33, 100}, 4 q / 2 kv heads, d 64, a
   64-block pool, block tables a seeded permutation of the physical ids.
2. Qwen2.5-0.5B decode layer -- 32 sequences, 14 q / 2 kv heads, d 64, contexts uniform in
   [129, 1152], a 4096-block pool ("mini-vllm" README, "Benchmark" runs Qwen2.5-0.5B).
3. Qwen3-0.6B decode layer -- 256 sequences, 16 q / 8 kv heads, d 128, contexts uniform in
   [100, 2048], a 40000-block pool; a quarter of the sequences share their first (up to 32)
   physical blocks, the effect of the prefix cache ("mini_engine" README, "Results": 256
   concurrent sequences, max_model_len 2048; "09 -- Mini Inference Engine (The Capstone)",
   "Week 5 -- Prefix caching").
4. Qwen2.5-7B long-context decode layer -- 50 sequences x 8192 context, 28 q / 4 kv heads,
   d 128, a 26000-block pool ("09 -- Mini Inference Engine (The Capstone)", "Acceptance
   criteria": at least 50 concurrent sequences at 8k context on Qwen 2.5 7B).
5. mixed chunked prefill + decode under an 8192-token budget, Qwen3-0.6B heads: 4 prefill
   chunks of 512 tokens over prior contexts {0, 512, 1024, 1536} plus 200 decode sequences
   with contexts uniform in [64, 2048], a 20000-block pool ("mini_engine" README, "What it
   does": chunked prefill under max_num_batched_tokens; "09 -- Mini Inference Engine (The
   Capstone)", "Week 3": mixed prefill and decode batches).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16
NAN_BF16 = np.uint16(0x7FC0)
_CHUNK = 1 << 22  # values drawn per call; fixed so the stream never depends on the sizes


@dataclass
class Batch:
    """One step's inputs: new tokens, the paged KV pool and the scheduler's tables."""

    name: str
    q: np.ndarray  # uint16 [T, Hq, d]
    k: np.ndarray  # uint16 [T, Hkv, d]
    v: np.ndarray  # uint16 [T, Hkv, d]
    positions: np.ndarray  # int64 [T]
    slot_mapping: np.ndarray  # int64 [T]
    k_cache: np.ndarray  # uint16 [num_blocks, block_size, Hkv, d]
    v_cache: np.ndarray  # uint16 [num_blocks, block_size, Hkv, d]
    block_tables: np.ndarray  # int32 [B, max_blocks], -1 padded
    context_lens: np.ndarray  # int32 [B], including the step's new tokens
    query_start_loc: np.ndarray  # int32 [B + 1]
    scale: float
    rope_theta: float
    info: dict = field(default_factory=dict)

    @property
    def num_tokens(self):
        return self.q.shape[0]

    @property
    def num_seqs(self):
        return self.context_lens.shape[0]

    @property
    def num_q_heads(self):
        return self.q.shape[1]

    @property
    def num_kv_heads(self):
        return self.k_cache.shape[2]

    @property
    def head_dim(self):
        return self.q.shape[2]

    @property
    def num_blocks(self):
        return self.k_cache.shape[0]

    @property
    def block_size(self):
        return self.k_cache.shape[1]


def _to_bf16_bits(x32):
    u = x32.view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def normal_bf16(rng, shape):
    """Standard-normal bf16 bit patterns, drawn in fixed-size chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        out[s:e] = _to_bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


def make_batch(
    context_lens,
    spans,
    num_q_heads,
    num_kv_heads,
    head_dim,
    num_blocks,
    seed,
    *,
    poison=True,
    scale=None,
    rope_theta=1.0e6,
    max_blocks_per_seq=None,
    shared_seqs=(),
    shared_prefix_blocks=0,
    name="custom",
    block_size=BLOCK_SIZE,
):
    """Build a batch: sequence b holds ``context_lens[b]`` keys after the step, of which the
    last ``spans[b]`` are the step's new tokens (1 = decode, >1 = prefill chunk, 0 = idle).

    Physical blocks come from a seeded permutation of the pool.  Sequences listed in
    ``shared_seqs`` point their first ``min(shared_prefix_blocks, (ctx - 1) // block_size)``
    logical blocks at one common run of physical blocks (prefix-cache reuse); the block
    receiving their new token is always private.  ``block_size`` is the tokens per pool block
    (16 unless a block-size variant is being measured).
    """
    bs = int(block_size)
    rng = np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int64)
    spans = np.asarray(spans, dtype=np.int64)
    B = ctx.shape[0]
    if spans.shape[0] != B:
        raise ValueError("context_lens and spans differ in length")
    if np.any(spans > ctx) or np.any(spans < 0):
        raise ValueError("every span must satisfy 0 <= span <= context")
    hq, hkv, d = int(num_q_heads), int(num_kv_heads), int(head_dim)
    pages = -(-ctx // bs)
    width = int(max_blocks_per_seq) if max_blocks_per_seq else max(1, int(pages.max()) if B else 1)
    if np.any(pages > width):
        raise ValueError("a context is longer than max_blocks_per_seq * block_size")

    perm = rng.permutation(num_blocks).astype(np.int64)
    cursor = 0
    shared_set = set(int(s) for s in shared_seqs)
    shared_run = None
    if shared_set and shared_prefix_blocks > 0:
        shared_run = perm[cursor : cursor + shared_prefix_blocks]
        cursor += shared_prefix_blocks
    bt = np.full((B, width), -1, dtype=np.int32)
    for b in range(B):
        n_sh = 0
        if b in shared_set and shared_run is not None:
            n_sh = min(shared_prefix_blocks, max(0, (int(ctx[b]) - 1) // bs))
            bt[b, :n_sh] = shared_run[:n_sh]
        need = int(pages[b]) - n_sh
        if cursor + need > num_blocks:
            raise ValueError("pool too small for the requested contexts")
        bt[b, n_sh : n_sh + need] = perm[cursor : cursor + need]
        cursor += need

    T = int(spans.sum())
    qsl = np.zeros(B + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(spans)
    positions = np.empty(T, dtype=np.int64)
    slots = np.empty(T, dtype=np.int64)
    for b in range(B):
        n = int(spans[b])
        p = np.arange(int(ctx[b]) - n, int(ctx[b]), dtype=np.int64)
        positions[qsl[b] : qsl[b + 1]] = p
        slots[qsl[b] : qsl[b + 1]] = bt[b, p // bs].astype(np.int64) * bs + p % bs

    q = normal_bf16(rng, (T, hq, d))
    k = normal_bf16(rng, (T, hkv, d))
    v = normal_bf16(rng, (T, hkv, d))

    # the pool: which (block, row) slots hold context before the step
    used_blocks = np.unique(bt[bt >= 0]).astype(np.int64)
    row_valid = np.zeros((num_blocks, bs), dtype=bool)
    for b in range(B):
        c = int(ctx[b])
        old = c - int(spans[b])  # keys that already exist before the step
        full, rem = divmod(old, bs)
        row_valid[bt[b, :full]] = True
        if rem:
            row_valid[bt[b, full], :rem] = True
    caches = []
    for _ in range(2):
        cache = np.zeros((num_blocks, bs, hkv, d), dtype=np.uint16)
        if used_blocks.size:
            cache[used_blocks] = normal_bf16(rng, (used_blocks.size, bs, hkv, d))
        if poison:
            cache[~row_valid] = NAN_BF16
        caches.append(cache)

    return Batch(
        name=name,
        q=q,
        k=k,
        v=v,
        positions=positions,
        slot_mapping=slots,
        k_cache=caches[0],
        v_cache=caches[1],
        block_tables=bt,
        context_lens=ctx.astype(np.int32),
        query_start_loc=qsl,
        scale=float(scale) if scale is not None else float(1.0 / np.sqrt(d)),
        rope_theta=float(rope_theta),
        info={"seed": seed, "poison": poison, "shared_seqs": sorted(shared_set)},
    )


CONFIG_NAMES = {
    1: "tiny-decode",
    2: "qwen2.5-0.5b-decode",
    3: "qwen3-0.6b-decode-256",
    4: "qwen2.5-7b-decode-50x8192",
    5: "mixed-prefill-decode",
}


def config(index, *, poison=True, seed=None, block_size=BLOCK_SIZE):
    """The five workloads listed in this module's docstring; seed defaults to index - 1.

    ``block_size`` other than 16 builds the same workload over blocks of that many tokens:
    the pool keeps its capacity in tokens, the table width and the shared prefix their
    lengths in tokens.  Lengths and sharing do not change; the block permutation does.
    """
    s = index - 1 if seed is None else seed
    name = CONFIG_NAMES[index] + ("" if block_size == BLOCK_SIZE else f"-bs{block_size}")
    rng = np.random.default_rng(1000 + s)  # lengths and sharing; values use ``s``
    bs = int(block_size)

    def blocks(tokens):
        return -(-tokens // bs)

    kw = dict(poison=poison, name=name, block_size=bs)
    if index == 1:
        return make_batch([1, 17, 33, 100], [1, 1, 1, 1], 4, 2, 64, blocks(64 * 16), s, **kw)
    if index == 2:
        ctx = rng.integers(129, 1152, size=32, endpoint=True)
        return make_batch(ctx, np.ones(32, np.int64), 14, 2, 64, blocks(4096 * 16), s, scale=1.0 / 8.0, **kw)
    if index == 3:
        ctx = rng.integers(100, 2048, size=256, endpoint=True)
        shared = rng.permutation(256)[:64]
        return make_batch(ctx, np.ones(256, np.int64), 16, 8, 128, blocks(40000 * 16), s,
                          max_blocks_per_seq=blocks(2048), shared_seqs=shared,
                          shared_prefix_blocks=blocks(512), **kw)
    if index == 4:
        return make_batch(np.full(50, 8192), np.ones(50, np.int64), 28, 4, 128, blocks(26000 * 16), s, **kw)
    if index == 5:
        dec = rng.integers(64, 2048, size=200, endpoint=True)
        prior = np.array([0, 512, 1024, 1536])
        ctx = np.concatenate([dec, prior + 512])
        spans = np.concatenate([np.ones(200, np.int64), np.full(4, 512)])
        return make_batch(ctx, spans, 16, 8, 128, blocks(20000 * 16), s, max_blocks_per_seq=blocks(2048), **kw)
    raise KeyError(index)


def random_case(seed, *, max_seqs=3, max_ctx=40, head_dims=(8, 64), groups=(1, 2, 3),
                kv_heads=(1, 2), allow_prefill=True, poison=True, block_size=BLOCK_SIZE):
    """A small random mixed batch for brute-force and micro parity checks."""
    rng = np.random.default_rng(50_000 + seed)
    B = int(rng.integers(1, max_seqs, endpoint=True))
    d = int(rng.choice(head_dims))
    hkv = int(rng.choice(kv_heads))
    hq = hkv * int(rng.choice(groups))
    ctx = rng.integers(1, max_ctx, size=B, endpoint=True)
    spans = np.ones(B, np.int64)
    if allow_prefill:
        for b in range(B):
            if rng.random() < 0.5:
                spans[b] = int(rng.integers(1, ctx[b], endpoint=True))
    pages = int((-(-ctx // block_size)).sum())
    nb = pages + int(rng.integers(0, 8))
    return make_batch(ctx, spans, hq, hkv, d, nb, seed, poison=poison,
                      rope_theta=float(rng.choice([1.0e4, 1.0e6])), name=f"random-{seed}",
                      block_size=block_size)
