#!/usr/bin/env python
"""Benchmark of the hot path: one step = fused RoPE-and-append + paged GQA attention over a
seeded synthetic batch shaped like a Qwen3-0.6B decode layer at 256 concurrent sequences
(16 q / 8 kv heads, head_dim 128, contexts uniform in [100, 2048], a quarter of the
sequences sharing up to 32 prefix blocks, 40000-block pool).

Prints ONE JSON line (rank 0).  ``value`` is the unique KV bytes the step must read divided
by the device time of the whole step (kv_append + paged_attention), in GB/s.  The roofline
object is for the dominant kernel (decode split-K), timed live with CUDA events recorded by
the library around that kernel on the launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference] [--workload I]

``--impl reference`` times the fp64 CPU oracle (the only reference this path has) on the
host cores, on a bounded sample of the same workload.  With N > 1 (torchrun) every rank runs
an independent replica (the path has no exchange step); rank 0 prints.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_gqa_14_gb300 import replicas  # noqa: E402
from paged_kv_gqa_14_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention achieved KV GB/s"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 10**6     # GB300 L2
FLUSH_BYTES = 256 << 20    # scratch written between timed steps in flush mode (> 2 x L2)


# ------------------------------------------------------------------------ workload facts
def kv_unique_bytes(bt, spans=None):
    """K+V bytes of every distinct (physical slot, kv head) the step's attention reads; with
    ``spans`` given, only over the sequences whose span length is in it."""
    bs = bt.block_size
    rows = set()
    for b in range(bt.num_seqs):
        n = int(bt.query_start_loc[b + 1] - bt.query_start_loc[b])
        if n == 0 or (spans is not None and n not in spans):
            continue
        ctx = int(bt.context_lens[b])
        for j in range(-(-ctx // bs)):
            blk = int(bt.block_tables[b, j])
            last = min(bs, ctx - bs * j)
            rows.update((blk, r) for r in range(last))
    return len(rows) * bt.num_kv_heads * bt.head_dim * 2 * 2


def kv_logical_bytes(bt):
    spans = np.diff(bt.query_start_loc)
    return int(bt.context_lens[spans > 0].astype(np.int64).sum()) * bt.num_kv_heads * bt.head_dim * 2 * 2


def decode_algorithmic_bytes(bt):
    """Algorithmic bytes of one decode-kernel launch: the unique KV of the decode sequences
    (span 1), their q rows read and out rows written, and their block-table entries and
    per-sequence metadata.  Prefill spans are the prefill kernel's."""
    spans = np.diff(bt.query_start_loc)
    dec = spans == 1
    kv = kv_unique_bytes(bt, spans=(1,))
    qo = 2 * int(dec.sum()) * bt.num_q_heads * bt.head_dim * 2
    tables = int((-(-bt.context_lens[dec].astype(np.int64) // bt.block_size)).sum()) * 4 + int(dec.sum()) * 8
    return kv + qo + tables


def sub_batch(bt, seqs):
    """A batch of the chosen sequences with a compact pool (for host-side oracle timing)."""
    seqs = list(seqs)
    blocks = sorted({int(x) for b in seqs for x in bt.block_tables[b] if x >= 0})
    remap = {b: i for i, b in enumerate(blocks)}
    idx = np.array(blocks, dtype=np.int64)
    rows = []
    qsl = [0]
    for b in seqs:
        s, e = int(bt.query_start_loc[b]), int(bt.query_start_loc[b + 1])
        rows.extend(range(s, e))
        qsl.append(qsl[-1] + e - s)
    rows = np.array(rows, dtype=np.int64)
    tables = np.array([[remap[int(x)] if x >= 0 else -1 for x in bt.block_tables[b]] for b in seqs], dtype=np.int32)
    slots = bt.slot_mapping[rows]
    bs = bt.block_size
    new_slots = np.array([remap[int(s) // bs] * bs + int(s) % bs if s >= 0 else -1 for s in slots], dtype=np.int64)
    return W.Batch(name=bt.name + f"-sample{len(seqs)}", q=bt.q[rows], k=bt.k[rows], v=bt.v[rows],
                   positions=bt.positions[rows], slot_mapping=new_slots, k_cache=bt.k_cache[idx],
                   v_cache=bt.v_cache[idx], block_tables=tables, context_lens=bt.context_lens[seqs],
                   query_start_loc=np.array(qsl, dtype=np.int32), scale=bt.scale, rope_theta=bt.rope_theta)


def prefill_flops(bt):
    """Algorithmic FLOPs of the prefill spans (n > 1 rows): 4 d per unmasked (query, key) pair
    per q head (QK^T and P.V, two flops per multiply-add).  Row r of an n-row span over ctx keys
    sees ctx - n + r + 1 keys."""
    pairs = 0
    for b in range(bt.num_seqs):
        n = int(bt.query_start_loc[b + 1] - bt.query_start_loc[b])
        if n > 1:
            ctx = int(bt.context_lens[b])
            pairs += n * (ctx - n + 1) + n * (n - 1) // 2
    return 4 * bt.head_dim * bt.num_q_heads * pairs


def oracle_step(sb):
    import oracle

    q_rot, kc, vc = oracle.kv_append(sb.q, sb.k, sb.v, sb.positions, sb.slot_mapping, sb.k_cache,
                                     sb.v_cache, sb.rope_theta)
    return oracle.paged_attention(q_rot, kc, vc, sb.block_tables, sb.context_lens, sb.query_start_loc,
                                  sb.scale)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def threads_used(cpu_s, wall_s):
    """Threads a run kept busy on average: its process CPU time over its wall time."""
    return max(1, int(round(cpu_s / max(wall_s, 1e-9))))


def time_oracle(bt, budget_s=12.0, min_seqs=2):
    """Time the oracle on the first n sequences, n grown until a step costs ~budget/4.
    Returns (sub-batch, wall seconds, n, threads used)."""
    n = min_seqs
    while True:
        sb = sub_batch(bt, range(n))
        c0, t0 = time.process_time(), time.perf_counter()
        oracle_step(sb)
        dt = time.perf_counter() - t0
        cpu = time.process_time() - c0
        if dt > budget_s / 4 or n >= bt.num_seqs:
            return sb, dt, n, threads_used(cpu, dt)
        n = min(bt.num_seqs, max(n + 1, int(n * min(8.0, (budget_s / 4) / max(dt, 1e-3)))))


# ------------------------------------------------------------- the oracle on all host cores
def _oracle_worker(conn):
    """A worker process: receives its sub-batch once, then runs the oracle on it per request
    and answers (wall seconds, CPU seconds)."""
    sb = conn.recv()
    while conn.recv() is not None:
        c0, t0 = time.process_time(), time.perf_counter()
        oracle_step(sb)
        conn.send((time.perf_counter() - t0, time.process_time() - c0))


class OracleWorkers:
    """The oracle over the first `n` sequences, split by sequence (they are independent) into
    one sub-batch per worker process.  Processes start with `spawn`: the parent may already
    hold a CUDA context, which a forked child must not inherit.  A step sends every worker
    its run request and waits for all answers, so its wall time is the parallel pass."""

    def __init__(self, bt, n, procs):
        import multiprocessing as mp

        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ.setdefault(var, "1")  # one thread per worker; the children inherit it
        ctx = mp.get_context("spawn")
        chunks = [c for c in np.array_split(np.arange(n), max(1, procs)) if len(c)]
        self.conns, self.procs = [], []
        for c in chunks:
            mine, theirs = ctx.Pipe()
            p = ctx.Process(target=_oracle_worker, args=(theirs,), daemon=True)
            p.start()
            mine.send(sub_batch(bt, [int(x) for x in c]))
            self.conns.append(mine)
            self.procs.append(p)

    def step(self):
        """(wall seconds, CPU seconds summed over the workers) of one parallel pass."""
        t0 = time.perf_counter()
        for c in self.conns:
            c.send(1)
        answers = [c.recv() for c in self.conns]
        return time.perf_counter() - t0, sum(a[1] for a in answers)

    def close(self):
        for c in self.conns:
            c.send(None)
        for p in self.procs:
            p.join(timeout=30)


def parallel_oracle(bt, budget_s, procs):
    """Workers over a sample sized so that a parallel pass costs about budget/4 (estimated from
    a short serial pass).  Returns (workers, sample size, unique KV bytes of the sample)."""
    _, dt, n0, _ = time_oracle(bt, budget_s=min(budget_s, 4.0) / 4)
    per_seq = dt / n0
    n = int(min(bt.num_seqs, max(n0, procs * (budget_s / 4) / max(per_seq, 1e-6))))
    workers = OracleWorkers(bt, n, procs)
    return workers, n, kv_unique_bytes(sub_batch(bt, range(n)))


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="pkv_clocks_", suffix=".csv")
            f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------ peaks
def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def hbm_peak():
    try:
        return float(_peaks()["hbm_gbs"]), "measured"
    except (KeyError, TypeError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    """Dense bf16 tensor peak in TFLOP/s: the measured burst figure (a kernel timed on its own
    inside a short step), else the fallback."""
    try:
        return float(_peaks()["bf16_tflops"]), "measured (burst)"
    except (KeyError, TypeError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback"


# ---------------------------------------------------------- DRAM traffic from ncu captures
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "kernel_traffic.json")
KERNEL_PATTERNS = {"decode": "decode_tc_kernel", "prefill": "prefill_tc_kernel"}


def source_sha256():
    """SHA-256 over the library's sources (header and every file of csrc/): a recorded
    traffic figure stands only for the code it was measured on."""
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_gqa_14_gb300", "csrc")
    for path in [os.path.join(ROOT, "include", "pkv.h")] + [os.path.join(csrc, f) for f in sorted(os.listdir(csrc))]:
        h.update(os.path.basename(path).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def kernel_traffic(kernel, workload):
    """Recorded DRAM bytes per launch of `kernel` on `workload`, or None when there is no record
    or it was taken on other sources."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)["records"][f"{kernel}/{workload}"]
    except (OSError, ValueError, KeyError):
        return None
    return float(rec["dram_bytes_per_launch"]) if rec.get("source_sha256") == source_sha256() else None


_UNIT = {"byte": 1, "b": 1, "kbyte": 1e3, "kb": 1e3, "mbyte": 1e6, "mb": 1e6, "gbyte": 1e9, "gb": 1e9}


def parse_ncu_dram(csv_path, pattern):
    """Per-launch (read, write) DRAM bytes of the kernels whose name contains `pattern`, from an
    ``ncu --csv --metrics dram__bytes_read.sum,dram__bytes_write.sum`` log."""
    import csv

    with open(csv_path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    launches = {}
    for row in csv.DictReader(lines):
        if pattern not in row.get("Kernel Name", ""):
            continue
        name = row.get("Metric Name", "")
        if name not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        val = float(row["Metric Value"].replace(",", "")) * _UNIT.get(row.get("Metric Unit", "byte").lower(), 1)
        launches.setdefault(row["ID"], {})[name] = val
    return [(v["dram__bytes_read.sum"], v["dram__bytes_write.sum"]) for v in launches.values()
            if len(v) == 2]


def record_traffic(csv_path, kernel, workload, command):
    """Store the mean DRAM bytes per launch of an ncu capture for (kernel, workload), stamped
    with the current sources' hash (run right after the capture, on the same sources)."""
    got = parse_ncu_dram(csv_path, KERNEL_PATTERNS[kernel])
    if not got:
        raise SystemExit(f"no {kernel} launches with DRAM metrics in {csv_path}")
    try:
        with open(TRAFFIC_FILE) as f:
            data = json.load(f)
    except (OSError, ValueError):
        data = {}
    data.setdefault("about", "DRAM traffic per kernel launch (dram__bytes_read.sum + dram__bytes_write.sum) "
                              "from ncu captures; written by `bench.py --record-traffic`; valid while "
                              "source_sha256 equals the hash of include/pkv.h and csrc/")
    rd = sum(r for r, _ in got) / len(got)
    wr = sum(w for _, w in got) / len(got)
    data.setdefault("records", {})[f"{kernel}/{workload}"] = {
        "kernel": KERNEL_PATTERNS[kernel], "workload": workload, "launches": len(got),
        "dram_read_bytes": round(rd), "dram_write_bytes": round(wr), "dram_bytes_per_launch": round(rd + wr),
        "source_sha256": source_sha256(), "command": command}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
        f.write("\n")
    return data["records"][f"{kernel}/{workload}"]


def percentiles(xs):
    """[p10, p50, p90] of a list of per-launch times (nearest rank), rounded."""
    v = sorted(xs)
    if not v:
        return None
    pick = lambda q: v[min(len(v) - 1, max(0, int(round(q * (len(v) - 1)))))]  # noqa: E731
    return [round(pick(0.1), 5), round(pick(0.5), 5), round(pick(0.9), 5)]


# ----------------------------------------------------------------------------- GPU arm
def run_gpu(args, rank, world, local_rank):
    import torch

    from paged_kv_gqa_14_gb300 import build as B
    from paged_kv_gqa_14_gb300 import ops

    B.build()
    torch.cuda.set_device(local_rank)
    if args.decode_kernel != "auto":
        ops.set_decode_kernel(args.decode_kernel)
    if args.prefill_kernel != "auto":
        ops.set_prefill_kernel(args.prefill_kernel)
    ops.set_overlap(not args.no_overlap)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    bt = W.config(args.workload, poison=False, block_size=args.block_size)
    if args.seqs:
        bt = sub_batch(bt, range(min(args.seqs, bt.num_seqs)))
    kv_u = kv_unique_bytes(bt)
    kv_l = kv_logical_bytes(bt)
    algo = decode_algorithmic_bytes(bt)
    n_decode = int((np.diff(bt.query_start_loc) == 1).sum())

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    q0 = up(bt.q)
    q = q0.clone()
    k, v = up(bt.k), up(bt.v)
    kc, vc = up(bt.k_cache), up(bt.v_cache)
    pos = torch.from_numpy(bt.positions).to(dev)
    slots = torch.from_numpy(bt.slot_mapping).to(dev)
    tables = torch.from_numpy(bt.block_tables).to(dev)
    ctx = torch.from_numpy(bt.context_lens).to(dev)
    qsl = torch.from_numpy(bt.query_start_loc).to(dev)
    out = torch.empty_like(q)
    ws = ops.alloc_workspace(bt.num_tokens, bt.num_seqs, bt.num_q_heads, bt.num_kv_heads, bt.head_dim,
                             bt.block_tables.shape[1], device=dev)
    stream = torch.cuda.current_stream()

    # the step's kv_append sits between the index tables' upload and the attention call, so the
    # planner may do its arithmetic while the append runs (PKV_ATTN_PLAN_EARLY) and, for a batch
    # large enough that it pays, the decode may copy the pages that hold no new key meanwhile
    # (PKV_ATTN_STREAM_EARLY)
    stream_early = not (args.no_plan_early or args.no_stream_early) and ops.stream_early_pays(
        bt.num_seqs, bt.block_tables.shape[1], bt.block_size)
    attn_opts = ops.attention_options({"plan_early": not args.no_plan_early, "stream_early": stream_early})

    def step():
        ops.kv_append(q, k, v, pos, slots, kc, vc, bt.rope_theta)
        ops.paged_attention(q, kc, vc, tables, ctx, qsl, bt.scale, out=out, workspace=ws, options=attn_opts)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert ops.get_device_error() == 0, "device error during warm-up"

    K = args.steps
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    # A step whose KV is not well above the L2 size would be timed partly from L2: then each
    # timed step runs alone, after a 256 MiB scratch write (twice the 129 MB L2) has evicted
    # what the previous step left there, and only the step sits between its two events.
    flush = kv_u < 2 * L2_BYTES
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None

    def timed(fn, n):
        """Mean ms of fn() over n calls on `stream`: back to back between two events, or in
        flush mode each call between its own events after an L2 flush."""
        if not flush:
            a, b = ev(), ev()
            a.record(stream)
            for _ in range(n):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / n
        pairs = [(ev(), ev()) for _ in range(n)]
        for i, (a, b) in enumerate(pairs):
            flush_buf.fill_(i & 0xFF)
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in pairs) / n

    dec = [(ev(), ev()) for _ in range(K)]
    pre = [(ev(), ev()) for _ in range(K)]
    app = [(ev(), ev()) for _ in range(K)]
    att0 = [ev() for _ in range(K)]
    scratch = [ev() for _ in range(K)]
    clocks = ClockSampler(local_rank)
    clocks.start()
    # (A) the timed region behind `value`: K steps back to back, nothing else on the stream
    # (or, in flush mode, each step alone after an L2 flush)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    total_ms = timed(step, K) * K
    if dist:
        dist.barrier()
    # (B) the same K steps again with the library recording events around each kernel
    for i in range(K):
        if flush:
            flush_buf.fill_(i & 0xFF)
        ops.set_kernel_events("decode", *dec[i])
        ops.set_kernel_events("prefill", *pre[i])
        ops.set_kernel_events("kv_append", *app[i])
        ops.set_kernel_events("plan", att0[i], scratch[i])
        step()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ops.set_kernel_events("decode")
    ops.set_kernel_events("prefill")
    ops.set_kernel_events("kv_append")
    ops.set_kernel_events("plan")
    dec_ms = [a.elapsed_time(b) for a, b in dec]
    app_ms = [a.elapsed_time(b) for a, b in app]
    # the prefill kernel runs only when some span can hold two or more tokens (more tokens
    # than sequences); otherwise its events are never recorded
    has_prefill_kernel = bt.num_tokens > bt.num_seqs
    pre_ms = [a.elapsed_time(b) for a, b in pre] if has_prefill_kernel else []
    att_ms = [a.elapsed_time(d[1]) for a, d in zip(att0, dec)]  # planner start .. decode end
    total_ms = replicas.max_over_ranks(total_ms, dist, device=dev)
    ms_step = total_ms / K
    dec_avg = sum(dec_ms) / K
    peak, peak_kind = hbm_peak()
    achieved = algo / (dec_avg * 1e-3) / 1e9
    traffic = kernel_traffic("decode", bt.name)
    # the prefill tiles' tensor-core roofline (batches with prefill spans): unmasked-pair FLOPs
    # over the prefill kernel's mean event time, against the bf16 peak; beside the decode also
    # per SM over the share of the SMs the planner gave it (workspace header word 5)
    pf_flops = prefill_flops(bt)
    roofline_prefill = None
    if pf_flops and pre_ms:
        pre_avg = sum(pre_ms) / K
        tpeak, tpeak_kind = bf16_peak()
        pf_tf = pf_flops / (pre_avg * 1e-3) / 1e12
        pf_ctas = int(ws[:64].view(torch.int32)[5].item())
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        roofline_prefill = {
            "kernel": "prefill_tiles",
            "bound": "tensor",
            "achieved": round(pf_tf, 1),
            "peak": tpeak,
            "peak_source": tpeak_kind,
            "unit": "TFLOP/s",
            "frac": round(pf_tf / tpeak, 4),
            "traffic": kernel_traffic("prefill", bt.name),
            "algorithmic_flops": pf_flops,
            "ms": round(pre_avg, 5),
            "prefill_ctas": pf_ctas,
            "sms": sms,
            "frac_of_its_sms": round(pf_tf / (tpeak * max(1, min(pf_ctas, sms)) / sms), 4),
        }

    # the same step captured once in a CUDA graph and replayed (host launch cost removed)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    graph_ms = timed(graph.replay, K)
    del graph

    # end to end through the public API with host buffers, every step: the step's inputs,
    # staged in one pinned host buffer, go up in one copy; the result comes back to pinned host
    from paged_kv_gqa_14_gb300.staging import StepStaging

    # auto: steps timed back to back overlap the copies with the steps, where the copy engines
    # win (no SMs taken from the step); a step timed alone waits for its copies, where the copy
    # kernel's lower start-up wins (measured on GB300)
    e2e_copy = args.e2e_copy if args.e2e_copy != "auto" else ("kernel" if flush else "engine")
    kernel_copy = e2e_copy == "kernel"
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)  # noqa: E731

    def staged():
        st = StepStaging(bt.num_tokens, bt.num_seqs, bt.num_q_heads, bt.num_kv_heads, bt.head_dim,
                         bt.block_tables.shape[1], device=dev, kernel_copy=kernel_copy)
        st.host.q.copy_(bf(bt.q))
        st.host.k.copy_(bf(bt.k))
        st.host.v.copy_(bf(bt.v))
        st.host.positions.copy_(torch.from_numpy(bt.positions))
        st.host.slot_mapping.copy_(torch.from_numpy(bt.slot_mapping))
        st.host.block_tables.copy_(torch.from_numpy(bt.block_tables))
        st.host.context_lens.copy_(torch.from_numpy(bt.context_lens))
        st.host.query_start_loc.copy_(torch.from_numpy(bt.query_start_loc))
        return st

    stg = staged()
    sd = stg.dev
    # (back to back) the next step's inputs go up on their own stream into a second staging
    # buffer while this step runs: every step's inputs still cross the link inside the timed
    # region, one step ahead, as its result crosses back one step behind
    stgs = [stg, staged()] if not flush else [stg]
    h2d_stream = torch.cuda.Stream(device=dev) if not flush else stream
    in_ready = [torch.cuda.Event(), torch.cuda.Event()]  # the step's inputs are on the device
    in_free = [torch.cuda.Event(), torch.cuda.Event()]   # the step that read them has finished
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = stg.nbytes
    d2h = host_out.numel() * host_out.element_size()
    # The result of step i goes back on a second stream while step i + 1 uploads and runs:
    # `out` is double-buffered, and step i + 2 writes its buffer only after that buffer's
    # copy back has finished (the two copies use the two directions of the host link).  In
    # flush mode every step is timed alone, nothing overlaps, and the copy back stays on the
    # step's own stream.
    d2h_stream = stream if flush else torch.cuda.Stream(device=dev)
    outs = [out, torch.empty_like(out)]
    out_ready = [torch.cuda.Event(), torch.cuda.Event()]  # attention wrote outs[j]
    out_free = [torch.cuda.Event(), torch.cuda.Event()]   # outs[j] is back on the host
    for j in range(2):
        out_free[j].record(stream)
        in_free[j].record(stream)
    e2e_no = [0]
    if not flush:  # the first step's inputs
        stgs[0].upload(h2d_stream)
        in_ready[0].record(h2d_stream)

    def e2e_step():
        if flush:  # one step alone: upload, step, copy back, all on the step's stream
            stg.upload(stream)
            ops.kv_append(sd.q, sd.k, sd.v, sd.positions, sd.slot_mapping, kc, vc, bt.rope_theta)
            ops.paged_attention(sd.q, kc, vc, sd.block_tables, sd.context_lens, sd.query_start_loc, bt.scale,
                                out=out, workspace=ws, options=attn_opts)
            if kernel_copy:
                ops.copy(host_out, out)
            else:
                host_out.copy_(out, non_blocking=True)
            return
        j = e2e_no[0] & 1
        e2e_no[0] += 1
        nj = 1 - j
        h2d_stream.wait_event(in_free[nj])  # the next step's staging buffer, once free
        stgs[nj].upload(h2d_stream)
        in_ready[nj].record(h2d_stream)
        # both waits before the append, so that nothing sits between the append and the
        # attention call (the planner overlaps the append only when they are adjacent)
        stream.wait_event(out_free[j])
        stream.wait_event(in_ready[j])
        sdj = stgs[j].dev
        ops.kv_append(sdj.q, sdj.k, sdj.v, sdj.positions, sdj.slot_mapping, kc, vc, bt.rope_theta)
        ops.paged_attention(sdj.q, kc, vc, sdj.block_tables, sdj.context_lens, sdj.query_start_loc, bt.scale,
                            out=outs[j], workspace=ws, options=attn_opts)
        in_free[j].record(stream)
        out_ready[j].record(stream)
        d2h_stream.wait_event(out_ready[j])
        if kernel_copy:
            ops.copy(host_out, outs[j], stream=d2h_stream)
        else:
            with torch.cuda.stream(d2h_stream):
                host_out.copy_(outs[j], non_blocking=True)
        out_free[j].record(d2h_stream)

    def e2e_steps_joined(n):
        """n end-to-end steps; the timed region ends when the last result is on the host."""
        def run():
            for _ in range(n):
                e2e_step()
            if d2h_stream is not stream:
                stream.wait_stream(d2h_stream)
        return run

    for _ in range(args.warmup):
        e2e_step()
    if d2h_stream is not stream:
        stream.wait_stream(d2h_stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e2e_ms = timed(e2e_steps_joined(K), 1) / K if not flush else timed(e2e_steps_joined(1), K)
    e2e_ms = replicas.max_over_ranks(e2e_ms, dist, device=dev)
    assert ops.get_device_error() == 0, "device error during timing"

    line = {
        "metric": METRIC,
        "value": round(replicas.job_throughput(kv_u, world, ms_step * 1e-3) / 1e9, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": bt.name,
            "num_seqs": bt.num_seqs,
            "num_q_heads": bt.num_q_heads,
            "num_kv_heads": bt.num_kv_heads,
            "head_dim": bt.head_dim,
            "block_size": bt.block_size,
            "context_lens": [int(bt.context_lens.min()), int(bt.context_lens.max())],
            "num_blocks": bt.num_blocks,
            "new_tokens": bt.num_tokens,
            "parallelism": f"replicas x{world}",
            "decode_kernel": args.decode_kernel,
            "prefill_kernel": args.prefill_kernel,
            "prefill_beside_decode": not args.no_overlap,
            "plan_early": not args.no_plan_early,
            "stream_early": stream_early,
            "l2": ("L2 flushed between timed steps (unique KV per step %.1f MB < 2 x 129 MB): a %d MiB "
                   "scratch write before each step, each step timed alone with CUDA events"
                   % (kv_u / 1e6, FLUSH_BYTES >> 20)) if flush else
                  ("inputs larger than L2 (unique KV per step %.0f MB > 2 x 129 MB); no flush" % (kv_u / 1e6)),
        },
        "tokens_per_s_per_layer": round(world * bt.num_tokens / (ms_step * 1e-3), 1),
        "kv_unique_bytes": kv_u,
        "kv_logical_bytes": kv_l,
        "kv_logical_gbs": round(world * kv_l / (ms_step * 1e-3) / 1e9, 2),
        "hbm_frac_step": round(kv_u / (ms_step * 1e-3) / 1e9 / peak, 4),
        "kernels_ms": {
            "kv_append": round(sum(app_ms) / K, 5),
            "paged_attention_call": round(sum(att_ms) / K, 5),
            "decode_splitk": round(dec_avg, 5),
            "prefill_tiles": round(sum(pre_ms) / K, 5) if pre_ms else None,
        },
        "kernels_ms_p10_p50_p90": {
            "kv_append": percentiles(app_ms),
            "paged_attention_call": percentiles(att_ms),
            "decode_splitk": percentiles(dec_ms),
            "prefill_tiles": percentiles(pre_ms),
        },
        "roofline": {
            "kernel": "decode_splitk",
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_source": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes": algo,
        },
        "roofline_prefill": roofline_prefill,
        "graph": {
            "ms_per_step": round(graph_ms, 5),
            "value": round(world * kv_u / (graph_ms * 1e-3) / 1e9, 2),
            "tokens_per_s_per_layer": round(world * bt.num_tokens / (graph_ms * 1e-3), 1),
        },
        "e2e": {
            "value": round(world * kv_u / (e2e_ms * 1e-3) / 1e9, 2),
            "unit": UNIT,
            "ms_per_step": round(e2e_ms, 5),
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "copy": e2e_copy,
            "pipeline": ("each step alone: upload, step, result copied back, on one stream" if flush else
                         "each step's inputs uploaded on a third stream one step ahead, into the other of two "
                         "staging buffers, while the step before runs; its result copied back on a second "
                         "stream while the next step runs (double-buffered out); every step's inputs and "
                         "result cross the link inside the timed region, which ends with the last result on "
                         "the host"),
        },
        # kv_append, planner, decode split-K (+ merge), and the prefill tiles when a span can
        # hold two or more tokens
        "gpu_launches": (4 if has_prefill_kernel else 3) * K,
        "clocks": clk,
        "decode_seqs": n_decode,
    }
    if rank == 0 and not args.no_cpu_baseline:
        procs = host_cores()
        workers, n, kv_s = parallel_oracle(bt, args.cpu_budget, procs)
        try:
            workers.step()  # warm-up: imports and first touch in every worker
            dt, cpu = workers.step()
        finally:
            workers.close()
        line["cpu_baseline"] = {
            "value": round(kv_s / dt / 1e9, 4),
            "unit": UNIT,
            "cores": threads_used(cpu, dt),
            "cores_available": procs,
            "workers": len(workers.procs),
            "kind": "oracle",
            "sample": f"first {n} of {bt.num_seqs} sequences of {bt.name} ({kv_s / 1e6:.1f} MB unique KV), "
                      f"oracle kv_append + paged_attention split by sequence over {len(workers.procs)} "
                      f"worker processes, one parallel pass {dt:.3f} s",
        }
    if dist:
        dist.destroy_process_group()
    return line


# ----------------------------------------------------------------------- reference arm
def run_reference(args):
    bt = W.config(args.workload, poison=False, block_size=args.block_size)
    procs = host_cores()
    workers, n, kv_s = parallel_oracle(bt, min(args.cpu_budget, 8.0), procs)
    times, cpus = [], []
    try:
        for _ in range(args.warmup):
            workers.step()
        for _ in range(args.steps):
            dt, cpu = workers.step()
            times.append(dt)
            cpus.append(cpu)
    finally:
        workers.close()
    used = threads_used(sum(cpus), sum(times))
    ms = 1e3 * sum(times) / len(times)
    value = round(kv_s / (ms * 1e-3) / 1e9, 4)
    return {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "impl": "reference",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": bt.name, "sample_seqs": n, "num_seqs": bt.num_seqs},
        "cpu_baseline": {
            "value": value,
            "unit": UNIT,
            "cores": used,
            "cores_available": host_cores(),
            "kind": "oracle",
            "workers": len(workers.procs),
            "sample": f"first {n} of {bt.num_seqs} sequences of {bt.name} per step ({kv_s / 1e6:.1f} MB unique KV), "
                      f"split by sequence over {len(workers.procs)} worker processes",
        },
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", type=int, default=3, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--e2e-copy", choices=["auto", "engine", "kernel"], default="auto",
                    help="end-to-end leg: move the staged inputs and the output with the copy engines "
                         "(cudaMemcpyAsync) or with a copy kernel reading/writing pinned host memory "
                         "(auto: engines when steps run back to back, the kernel when each runs alone)")
    ap.add_argument("--block-size", type=int, default=16, choices=[8, 16, 32, 64, 128],
                    help="tokens per pool block (the workload keeps its pool size in tokens)")
    ap.add_argument("--seqs", type=int, default=0, help="only the first N sequences (small profiling case)")
    ap.add_argument("--decode-kernel", choices=["auto", "simt", "tensor"], default="auto")
    ap.add_argument("--prefill-kernel", choices=["auto", "mma", "tcgen05"], default="auto")
    ap.add_argument("--no-plan-early", action="store_true",
                    help="plan after the append has finished (default: the planner computes while it runs)")
    ap.add_argument("--no-stream-early", action="store_true",
                    help="the decode reads the plan after the append has finished (default: it copies "
                         "the pages without new keys while the append runs)")
    ap.add_argument("--no-overlap", action="store_true",
                    help="prefill tiles before the decode on one stream (default: beside it, SMs split)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--record-traffic", metavar="CSV",
                    help="no benchmark: store the DRAM bytes per launch of an ncu capture "
                         "(--csv --print-units base --metrics dram__bytes_read.sum,dram__bytes_write.sum) of "
                         "--kernel on --workload in profiles/kernel_traffic.json, stamped with the sources' hash")
    ap.add_argument("--kernel", choices=sorted(KERNEL_PATTERNS), default="decode")
    ap.add_argument("--command", default="", help="the capture command, stored with --record-traffic")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.record_traffic:
        name = W.CONFIG_NAMES[args.workload] + ("" if args.block_size == W.BLOCK_SIZE else f"-bs{args.block_size}")
        if args.seqs:
            name += f"-sample{args.seqs}"
        rec = record_traffic(args.record_traffic, args.kernel, name, args.command)
        print(json.dumps(rec))
        return
    rank, world, local_rank = replicas.rank_info()
    if args.gpus != world:
        ap.error(f"--gpus {args.gpus} but {world} process(es) (WORLD_SIZE): start N > 1 replicas with "
                 f"`python -m torch.distributed.run --nproc-per-node {args.gpus} bench.py --gpus {args.gpus} ...`")
    if args.impl == "reference":
        if rank != 0:
            return
        line = run_reference(args)
    else:
        line = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
