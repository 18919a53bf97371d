"""Rotary position embedding in fp64 (oracle; test infrastructure only).

Source: MiniPIC: Position-Independent Caching ..., section 2.1 ("Position-free KV"): the cache
stores unrotated keys k~_j and the score of query t against cached key j is
(R_t q_t)^T (R_pi(j) k~_j) / sqrt(d), with R the rotation matrix and pi(j) the key's logical
position in the current request.

The pages do not fix the pairing of dimensions or the frequencies.  Reading used here: the
"rotate-half" convention -- dimension i is paired with i + d/2 for i < d/2, and
the pair turns by the angle p * theta^(-2i/d).  No frequency scaling.
"""
from __future__ import annotations

import numpy as np


def inv_freq(d: int, theta: float) -> np.ndarray:
    """theta^(-2i/d) for i = 0 .. d/2-1, fp64."""
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * i / d)


def angles(pos: np.ndarray, d: int, theta: float) -> np.ndarray:
    """[n, d/2] angles p * theta^(-2i/d) in fp64."""
    return np.asarray(pos, dtype=np.float64)[:, None] * inv_freq(d, theta)[None, :]


def rotate(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """R_pos x for x of shape [n, ..., d] and positions pos of shape [n] (one position per leading
    index).  Pair (x_i, x_{i+d/2}) -> (x_i cos a - x_{i+d/2} sin a, x_{i+d/2} cos a + x_i sin a)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    h = d // 2
    a = angles(pos, d, theta)                       # [n, h]
    a = a.reshape((a.shape[0],) + (1,) * (x.ndim - 2) + (h,))
    c, s = np.cos(a), np.sin(a)
    x1, x2 = x[..., :h], x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)
