"""Seeded synthetic inputs for the Four Over Six NVFP4 workloads.

This module holds only random-number generation and bf16 packing; it contains
none of the quantization arithmetic.  Both the CPU oracle's tests and the CUDA
path's tests and benchmark draw their inputs from here, so the two sides read
identical bytes.

Workloads (the pages publish no benchmark suite; these synthetic tensors stand
in for the weight, activation and gradient tensors they describe):

* ``outlier_matrix``  256 x 256, N(0,1), every 512th element (row-major) x20
  (the outlier pattern of the worked MAE example on the "FP4" glossary page).
* ``qwen3_8b_weights``  the q/k/v/o/gate/up/down projection shapes of one
  Qwen3-8B decoder layer (the model named on the "Four Over Six" page);
  Student-t (nu = 4) scaled to std 0.02.  Shapes only; no trained weights.
* ``activations``  N(0,1) with a few seeded channels (columns) scaled x50.
* ``gradients``  Laplace(0, 1e-3) with 0.1% of entries from Laplace(0, 0.1).

Every generator takes an explicit seed; chunking is fixed so the stream does
not depend on memory limits.
"""
from __future__ import annotations

import numpy as np

_CHUNK = 1 << 22

# name -> (rows, cols) = (out_features, in_features) of one Qwen3-8B layer
QWEN3_8B_LAYER = {
    "q_proj": (4096, 4096),
    "k_proj": (1024, 4096),
    "v_proj": (1024, 4096),
    "o_proj": (4096, 4096),
    "gate_proj": (12288, 4096),
    "up_proj": (12288, 4096),
    "down_proj": (4096, 12288),
}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even (finite x)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _chunked(n: int, seed: int, draw) -> np.ndarray:
    out = np.empty(n, np.float32)
    ss = np.random.SeedSequence(seed)
    for i, child in enumerate(ss.spawn((n + _CHUNK - 1) // _CHUNK)):
        lo = i * _CHUNK
        hi = min(n, lo + _CHUNK)
        out[lo:hi] = draw(np.random.default_rng(child), hi - lo)
    return out


def normal(rows: int, cols: int, seed: int) -> np.ndarray:
    return _chunked(rows * cols, seed, lambda g, m: g.standard_normal(m, dtype=np.float32)).reshape(rows, cols)


def outlier_matrix(seed: int = 1001, rows: int = 256, cols: int = 256) -> np.ndarray:
    """bf16 bits: N(0,1) with every 512th element (row-major) multiplied by 20."""
    x = normal(rows, cols, seed).reshape(-1)
    x[::512] *= 20.0
    return bf16_bits(x.reshape(rows, cols))


def student_t(rows: int, cols: int, seed: int, std: float = 0.02, nu: float = 4.0) -> np.ndarray:
    """bf16 bits: Student-t(nu) scaled so the std is `std` (t_4 has variance 2)."""
    scale = std / np.sqrt(nu / (nu - 2.0))
    x = _chunked(rows * cols, seed, lambda g, m: (g.standard_t(nu, m) * scale).astype(np.float32))
    return bf16_bits(x.reshape(rows, cols))


def qwen3_8b_weights(seed_base: int = 2000) -> dict[str, np.ndarray]:
    return {name: student_t(r, c, seed_base + j) for j, (name, (r, c)) in enumerate(QWEN3_8B_LAYER.items())}


def activations(rows: int, cols: int, seed: int, n_hot: int = 8, hot_scale: float = 50.0) -> np.ndarray:
    """bf16 bits: N(0,1) with `n_hot` seeded channels (columns) scaled by `hot_scale`."""
    x = normal(rows, cols, seed)
    hot = np.random.default_rng(seed + 7919).choice(cols, size=min(n_hot, cols), replace=False)
    x[:, hot] *= hot_scale
    return bf16_bits(x)


def gradients(rows: int, cols: int, seed: int, b: float = 1e-3, b_out: float = 0.1, frac: float = 1e-3) -> np.ndarray:
    """bf16 bits: Laplace(0, b), with a fraction `frac` of entries from Laplace(0, b_out)."""

    def draw(g, m):
        v = g.laplace(0.0, b, m)
        sel = g.random(m) < frac
        v[sel] = g.laplace(0.0, b_out, int(sel.sum()))
        return v.astype(np.float32)

    return bf16_bits(_chunked(rows * cols, seed, draw).reshape(rows, cols))


def uniform_bits(rows: int, cols: int, seed: int, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    x = _chunked(rows * cols, seed, lambda g, m: g.uniform(lo, hi, m).astype(np.float32))
    return bf16_bits(x.reshape(rows, cols))
