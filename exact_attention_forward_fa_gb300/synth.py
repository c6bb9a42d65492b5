"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no attention arithmetic: it only draws random numbers and
rounds them to the storage dtype.  Both the CUDA path and the CPU oracle
consume exactly the tensors it returns.

Recipe (the workloads of "FlashAttention-3" as reviewed on diycv.top,
"experimental setup" and "numerical error" sections):

* Q, K, V entries iid N(0, 1), drawn with numpy's PCG64 ``default_rng`` as
  float32, then rounded to bf16 (or fp16) round-to-nearest-even by torch.
  Q uses ``seed``, K ``seed + 1``, V ``seed + 2``.
* FP8 outlier inputs: each entry is N(0, 1) plus, with probability 1e-3,
  an added N(0, 100) term (standard deviation 10).
* Hadamard signs for incoherent processing: d entries of +-1 from
  ``default_rng(seed)``.
* Sink logits (one per query head): N(2, 2) from ``default_rng(seed)`` as
  float32, so that e^sigma ranges from negligible to larger than the row
  sum of a narrow window.

Layout: [B][N][H][d] (batch, sequence, head, head dim), contiguous.
"""
from __future__ import annotations

import numpy as np
import torch

BASE_SEED = 20261202

_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


def normal(shape, seed: int, outliers: bool = False) -> np.ndarray:
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape, dtype=np.float32)
    if outliers:
        hit = rng.random(shape, dtype=np.float32) < np.float32(1e-3)
        extra = np.float32(10.0) * rng.standard_normal(shape, dtype=np.float32)
        x = x + np.where(hit, extra, np.float32(0.0))
    return x


def qkv(B: int, H: int, N: int, d: int, seed: int = BASE_SEED,
        dtype: str = "bf16", outliers: bool = False):
    """Q, K, V as CPU torch tensors [B, N, H, d] in ``dtype``."""
    tdt = _DTYPES[dtype]
    shape = (B, N, H, d)
    return tuple(torch.from_numpy(normal(shape, seed + i, outliers)).to(tdt)
                 for i in range(3))


def hadamard_signs(d: int, seed: int = BASE_SEED) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return np.where(rng.random(d) < 0.5, -1.0, 1.0).astype(np.float32)


def default_alpha(d: int) -> float:
    """1/sqrt(d) rounded to float32 (the value handed to the kernel)."""
    return float(np.float32(1.0 / np.sqrt(np.float64(d))))


def sinks(H: int, seed: int = BASE_SEED) -> np.ndarray:
    """float32 [H] sink logits, N(2, 2)."""
    rng = np.random.default_rng(seed)
    return (np.float32(2.0) + np.float32(2.0) * rng.standard_normal(H, dtype=np.float32))
