"""Seeded synthetic inputs for the five row-op workloads.

This module only draws random numbers (numpy PCG64, one spawned stream per
tensor) and arranges them into the shapes, distributions and structure of the
workloads; it contains none of the row ops' arithmetic.  The same arrays feed
the CUDA path and the CPU oracle, so both sides always see identical fp32 bytes.

Workloads (sizes are the defaults; every generator also takes smaller sizes
with the same distributions for parity cases):

* ``softmax_pair``  - softmax_rows forward + backward, rows=256, cols=128,
  x ~ N(0, 2^2), dy ~ N(0, 1).
* ``layernorm``     - rows=4096 (8 x 512 tokens), cols=768, eps=1e-5; row i is
  N(0,1)*s_i + c_i with s_i ~ U(0.1, 10), c_i ~ U(-5, 5); gamma = 1 + N(0, 0.1^2),
  beta ~ N(0, 0.1^2), upstream gradient ~ N(0, 1).
* ``attention``     - scores of shape (8, 12, 1024, 1024) ~ N(0, 8^2), scale 1/8,
  upstream gradient ~ N(0, 1).
* ``cross_entropy`` - logits (8192 x 50304) ~ N(0, 2^2) with exactly
  round(1e-4 * rows * cols) distinct entries set to +-30 (fair sign), targets
  uniform int32 in [0, cols).
* ``router``        - logits (262144 x 64) uniform on the 65 multiples of 1/8 in
  [-4, 4] (forces ties); uint8 mask allowing each entry with probability 0.9,
  then exactly round(0.01 * rows) whole rows blocked; k = 2.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "streams",
    "softmax_pair",
    "layernorm",
    "attention",
    "cross_entropy",
    "router",
    "WORKLOADS",
]


def streams(seed: int, n: int) -> list[np.random.Generator]:
    """n independent PCG64 generators spawned from one seed."""
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def _normal32(rng: np.random.Generator, shape, sigma: float) -> np.ndarray:
    # float32 draws scaled by a power of two (sigma in {1, 2, 8}) stay exact.
    out = rng.standard_normal(shape, dtype=np.float32)
    if sigma != 1.0:
        out *= np.float32(sigma)
    return out


def softmax_pair(seed: int = 0, rows: int = 256, cols: int = 128) -> dict:
    r_x, r_dy = streams(seed, 2)
    return {
        "x": _normal32(r_x, (rows, cols), 2.0),
        "dy": _normal32(r_dy, (rows, cols), 1.0),
    }


def layernorm(seed: int = 0, rows: int = 4096, cols: int = 768, eps: float = 1e-5) -> dict:
    r_z, r_s, r_c, r_g, r_b, r_dy = streams(seed, 6)
    z = r_z.standard_normal((rows, cols))
    s = r_s.uniform(0.1, 10.0, size=(rows, 1))
    c = r_c.uniform(-5.0, 5.0, size=(rows, 1))
    return {
        "x": (z * s + c).astype(np.float32),
        "gamma": (1.0 + 0.1 * r_g.standard_normal(cols)).astype(np.float32),
        "beta": (0.1 * r_b.standard_normal(cols)).astype(np.float32),
        "dy": r_dy.standard_normal((rows, cols)).astype(np.float32),
        "eps": eps,
    }


def attention(seed: int = 0, batch: int = 8, heads: int = 12, seq: int = 1024,
              head_dim: int = 64) -> dict:
    r_s, r_dp = streams(seed, 2)
    rows = batch * heads * seq
    return {
        "scores": _normal32(r_s, (rows, seq), 8.0),
        "dp": _normal32(r_dp, (rows, seq), 1.0),
        "seq_len": seq,
        "scale": 1.0 / float(np.sqrt(head_dim)),
    }


def cross_entropy(seed: int = 0, rows: int = 8192, cols: int = 50304,
                  outlier_frac: float = 1e-4, outlier: float = 30.0) -> dict:
    r_x, r_pos, r_sign, r_t = streams(seed, 4)
    logits = _normal32(r_x, (rows, cols), 2.0)
    n_out = int(round(outlier_frac * rows * cols))
    if n_out:
        pos = r_pos.choice(rows * cols, size=n_out, replace=False)
        sign = r_sign.integers(0, 2, size=n_out).astype(np.float32) * 2.0 - 1.0
        logits.reshape(-1)[pos] = np.float32(outlier) * sign
    return {
        "logits": logits,
        "targets": r_t.integers(0, cols, size=rows, dtype=np.int32),
        "grad_scale": 1.0 / rows,
    }


def router(seed: int = 0, rows: int = 262144, cols: int = 64, k: int = 2,
           p_allow: float = 0.9, blocked_row_frac: float = 0.01) -> dict:
    r_x, r_m, r_rows = streams(seed, 3)
    x = (r_x.integers(-32, 33, size=(rows, cols), dtype=np.int32).astype(np.float32)
         / np.float32(8.0))
    mask = (r_m.random((rows, cols), dtype=np.float32) < np.float32(p_allow)).astype(np.uint8)
    n_blocked = int(round(blocked_row_frac * rows))
    blocked_rows = np.sort(r_rows.choice(rows, size=n_blocked, replace=False)) if n_blocked else \
        np.zeros(0, dtype=np.int64)
    mask[blocked_rows] = 0
    return {"x": x, "mask": mask, "k": k, "blocked_rows": blocked_rows}


WORKLOADS = {
    "softmax_pair": softmax_pair,
    "layernorm": layernorm,
    "attention": attention,
    "cross_entropy": cross_entropy,
    "router": router,
}
