"""Helpers for the GPU tests: upload seeded batches, run the CUDA path, compare with the oracle."""

import functools

import numpy as np
import torch

import oracle
from paged_kv_gqa_14_gb300 import ops
from paged_kv_gqa_14_gb300 import workloads as W

MAX_ABS = 2e-2  # attention tolerance vs the fp64 oracle (bf16 in, fp32 accumulate)
MEAN_ABS = 2e-3


def dev():
    return torch.device("cuda:0")


def bf16_to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev())


def dev_to_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def idx_to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


class Dev:
    """A batch resident on the GPU."""

    def __init__(self, bt, q=None, k_cache=None, v_cache=None):
        self.bt = bt
        self.q = bf16_to_dev(bt.q if q is None else q)
        self.k = bf16_to_dev(bt.k)
        self.v = bf16_to_dev(bt.v)
        self.k_cache = bf16_to_dev(bt.k_cache if k_cache is None else k_cache)
        self.v_cache = bf16_to_dev(bt.v_cache if v_cache is None else v_cache)
        self.positions = idx_to_dev(bt.positions)
        self.slots = idx_to_dev(bt.slot_mapping)
        self.block_tables = idx_to_dev(bt.block_tables)
        self.context_lens = idx_to_dev(bt.context_lens)
        self.qsl = idx_to_dev(bt.query_start_loc)

    def append(self):
        ops.kv_append(self.q, self.k, self.v, self.positions, self.slots, self.k_cache, self.v_cache,
                      self.bt.rope_theta)

    def attend(self, out=None):
        return ops.paged_attention(self.q, self.k_cache, self.v_cache, self.block_tables, self.context_lens,
                                   self.qsl, self.bt.scale, out=out)


@functools.lru_cache(maxsize=2)
def config_with_oracle(index):
    """(batch, q_rot, k_cache, v_cache, oracle out) for a workload, computed once per process."""
    bt = W.config(index)
    q_rot, kc, vc = oracle.kv_append(bt.q, bt.k, bt.v, bt.positions, bt.slot_mapping, bt.k_cache,
                                     bt.v_cache, bt.rope_theta)
    ref = oracle.paged_attention(q_rot, kc, vc, bt.block_tables, bt.context_lens, bt.query_start_loc,
                                 bt.scale)
    return bt, q_rot, kc, vc, ref


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (
        f"{what}: max abs {err.max():.3e} (<= {MAX_ABS}), mean abs {err.mean():.3e} (<= {MEAN_ABS})")
    return err.max(), err.mean()


def ulp_bf16(x):
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.maximum(x, 2.0**-126))
    return np.ldexp(1.0, e - 8)


def rope_tol(x_bits, ref):
    """Allowed |gpu - oracle| for a rotated bf16 value.

    Error budget of the kernel's fp32 value before its bf16 rounding, for a pair (x, y) at a
    position p < 2^31 (both sides start from the same bf16 inputs and the same fp64 f_i):
      * angle: the 0.64 fixed-point turn p F_i mod 2^64 is exact up to F_i's rounding
        (p 2 pi / 2^64 rad); the quarter turn is exact; the remainder r in [-pi/4, pi/4]
        reaches fp32 with one rounding, <= 2^-25 rad;
      * sincosf: <= 2 ulp, i.e. <= 2^-23 absolute on values in [-1, 1];
      * x c - y s: one product rounding and one sum rounding, <= 2^-23 (|x| + |y|);
    so |fp32 - exact| <= (2^-23 + 2^-25 + 2^-23) (|x| + |y|) < 2.7e-7 (|x| + |y|) for the
    positions tested (p 2 pi 2^-64 < 1e-11 for p <= 2^24).  The oracle's own fp64 angle p f_i
    carries p f_i 2^-53 rad (below 2^-28 here).  Rounding both to bf16 then differs by at most
    that error plus one bf16 ulp, so the bound is one ulp of the reference plus
    2^-21 (|x_i| + |x_{i+d/2}|), which holds the derived 2.7e-7 with a margin of 1.7.
    """
    x = np.abs(np.asarray(x_bits_to_f64(x_bits)))
    half = x.shape[-1] // 2
    m = x[..., :half] + x[..., half:]
    pair = np.concatenate([m, m], axis=-1)
    return ulp_bf16(ref) + 2.0**-21 * pair


def x_bits_to_f64(bits):
    return oracle.bf16_bits_to_f64(bits)
