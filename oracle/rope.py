"""Rotary position embedding in fp64 (test infrastructure only).

Follows "mini_engine" README, "What it does" (the Qwen3 decoder uses RoPE) and
"Next: fused kernels" (RoPE fused into the KV write).  The pages name RoPE without a
formula; the reading taken is the rotate-half form the Qwen model family uses:

* the d coordinates of one head form d/2 pairs (x_i, x_{i + d/2}), i in [0, d/2);
* pair i turns by the angle a_i = pos * f_i with f_i = theta ** (-2 i / d);
* (x_i, x_{i+d/2}) -> (x_i cos a_i - x_{i+d/2} sin a_i,  x_{i+d/2} cos a_i + x_i sin a_i).

No frequency scaling (no NTK / YaRN).  V is never rotated.
"""

import numpy as np


def rope_inv_freq(head_dim, theta):
    """f_i = theta ** (-2 i / d) for i in [0, d/2), in fp64."""
    if head_dim % 2:
        raise ValueError("RoPE needs an even head_dim")
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.float64(theta) ** (-2.0 * i / head_dim)


def rope64(x, positions, theta):
    """Rotate the last axis of ``x`` (float64, [..., d]).

    ``positions`` broadcasts against ``x[..., 0]``; it is converted to float64 exactly
    (integer positions below 2**53).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    pos = np.asarray(positions, dtype=np.float64)
    ang = pos[..., None] * rope_inv_freq(d, theta)
    c = np.cos(ang)
    s = np.sin(ang)
    x1 = x[..., :half]
    x2 = x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)
