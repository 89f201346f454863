"""fp64 CPU oracle for the flat GEMM of the decode phase.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or run
this module. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it. It shares no code with the CUDA path.

Source: "【FlashAttention-V4，非官方】FlashDecoding++". Sections 1 and 2 state the
problem: in the decode phase the GEMMs either side of attention are flat, because
only a few tokens (the batch) go through them at a time; with one token the GEMM is
a GEMV. Section 4 (Flat GEMM Optimization with Double Buffering) writes them as
the product of an M x K matrix and a K x N matrix, where M is the small token
count, and says that libraries pad M with zeros up to 64 while the page pads it
to 8 only, and that two shared-memory buffers overlap the loads of the next tile
with the products of the current one. Neither the padding nor the buffering
changes what is computed, so the oracle is the matrix product itself, in fp64.

Readings where the page is silent:

* The K x N operand (the weights) is passed as its transpose ``w[N, K]``: each of
  its N columns is contiguous, the layout projection weights are kept in. Then
  ``y[m, n] = sum_k x[m, k] * w[n, k]``, i.e. ``Y = X W^T``.
* The inputs are the exact values the GPU sees (bf16-rounded, widened to fp64);
  the GPU accumulates in fp32 and rounds ``Y`` to bf16 (nearest even).
"""
from __future__ import annotations

import numpy as np

__all__ = ["flat_gemm", "pad_rows"]


def flat_gemm(x, w):
    """``Y[M, N] = X[M, K] @ W[N, K]^T`` in float64 (the definition; a library matmul)."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    if x.ndim != 2 or w.ndim != 2 or x.shape[1] != w.shape[1]:
        raise ValueError(f"flat_gemm: x {x.shape} and w {w.shape} do not share K")
    return x @ w.T


def pad_rows(x, multiple):
    """``x`` with zero rows appended until its row count is a multiple of ``multiple``
    (the page's padding of the token dimension M to 8, or the libraries' to 64)."""
    x = np.asarray(x, dtype=np.float64)
    m = x.shape[0]
    target = -(-m // multiple) * multiple
    out = np.zeros((target, x.shape[1]), dtype=np.float64)
    out[:m] = x
    return out
