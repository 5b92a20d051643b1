"""The rotation frequencies of kv_append (``pkv_rope_turn_table``, host code of the library, no
GPU) against their definition: F_i = round(frac(f_i / (2 pi)) * 2^64) with f_i = theta^(-2i/d)
("mini_engine" README, "What it does": RoPE; rotate-half pairs, f_i as the oracle reads it).
Checked exactly with 200-bit arithmetic, for bases above and below one (below one a pair turns
by more than a full turn per position), and through the oracle's fp64 rotation."""

import math

import numpy as np
import pytest

import oracle
from paged_kv_gqa_14_gb300 import build as B
from paged_kv_gqa_14_gb300 import ops

mp = pytest.importorskip("mpmath")

THETAS = [1.0e6, 1.0e4, 500.0, 10.0, 1.0, 0.5, 0.1, 1.0e-3]


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()


def exact_table(theta, d):
    with mp.workprec(200):
        two_pi = 2 * mp.pi
        out = []
        for i in range(d // 2):
            f = math.pow(theta, -2.0 * i / d)  # the fp64 frequency both sides start from
            frac = mp.mpf(f) / two_pi
            frac -= mp.floor(frac)
            out.append(int(mp.nint(frac * mp.mpf(2) ** 64)) % 2**64)
        return out


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("theta", THETAS)
def test_turn_table_matches_definition_to_one_unit(theta, d):
    got = [int(x) for x in ops.rope_turn_table(theta, d)]
    ref = exact_table(theta, d)
    for i, (g, r) in enumerate(zip(got, ref)):
        diff = (g - r) % 2**64
        assert min(diff, 2**64 - diff) <= 1, (theta, d, i, g, r)


@pytest.mark.parametrize("theta", [0.5, 0.1, 1.0e-3, 1.0e6])
def test_turn_table_rotation_equals_oracle_rope(theta):
    # rotating the unit vector e_i gives (cos a_i, sin a_i) in the oracle; the table's angle is
    # 2 pi (p F_i mod 2^64) / 2^64.  The oracle's fp64 angle p f_i is exact to p f_i 2^-53.
    d = 64
    F = [int(x) for x in ops.rope_turn_table(theta, d)]
    pos = np.array([0, 1, 2, 3, 17, 1000, 65537, 1_000_003], dtype=np.int64)
    x = np.zeros((len(pos), d))
    x[:, :] = 0.0
    x[:, : d // 2] = 1.0  # every pair (1, 0)
    rot = oracle.rope64(x, pos, theta)
    f = oracle.rope_inv_freq(d, theta)
    for r, p in enumerate(pos):
        for i in range(d // 2):
            with mp.workprec(120):
                a = 2 * mp.pi * mp.mpf((int(p) * F[i]) % 2**64) / mp.mpf(2) ** 64
                c, s = float(mp.cos(a)), float(mp.sin(a))
            tol = 4 * (float(p) * f[i] * 2.0**-53 + 1e-15) + int(p) * 2 * math.pi * 2.0**-64
            assert abs(rot[r, i] - c) <= tol and abs(rot[r, i + d // 2] - s) <= tol, (theta, p, i)


@pytest.mark.parametrize("theta", [0.0, -1.0, float("inf"), float("nan"), 1e-300])
def test_refused_bases(theta):
    with pytest.raises(RuntimeError, match="PKV_ERR_SHAPE"):
        ops.rope_turn_table(theta, 64)


def test_refused_head_dim():
    with pytest.raises(RuntimeError, match="PKV_ERR_UNSUPPORTED"):
        ops.rope_turn_table(1e6, 96)
