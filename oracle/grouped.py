"""Grouped-layout GEMM oracle ([Chord] "그룹 SM90 커널 기법").

The grouped kernels take activation rows already grouped by expert, in one
of two layouts:
  * contiguous (prefill): the experts' row groups follow one another in
    expert order, each padded to a 128-row boundary;
  * masked (decode): a fixed budget of max_m rows per expert, A shaped
    [E, max_m, K]; expert e uses its first group_rows[e] rows.
Each used row r of expert e gives C[r] = A[r] . W_e^T (W_e exactly
dequantised, FP64), optionally followed by SiLU(gate) * up (layer.py's
silu_mul).  Readings where the page is silent: the groups are described by
per-expert row counts (the layout's offsets follow from them), and rows past
an expert's count are not outputs.
"""
from __future__ import annotations

import numpy as np

from .layer import expert_rows_gemm, silu_mul
from .quant import dequant_expert

PAD_CONTIGUOUS = 128


def group_starts(group_rows, layout: str, max_m: int = 0) -> np.ndarray:
    """First row of each expert's group: [E] int64."""
    c = np.asarray(group_rows, dtype=np.int64)
    if layout == "masked":
        return np.arange(c.size, dtype=np.int64) * max_m
    padded = (c + PAD_CONTIGUOUS - 1) // PAD_CONTIGUOUS * PAD_CONTIGUOUS
    return np.concatenate([[0], np.cumsum(padded)[:-1]]).astype(np.int64)


def grouped_gemm(a_rows, group_rows, w_q, w_s, layout: str, max_m: int = 0, silu: bool = False):
    """a_rows float64 [rows, K] (masked: [E * max_m, K]); returns (row indices, outputs)."""
    a_rows = np.asarray(a_rows, np.float64)
    starts = group_starts(group_rows, layout, max_m)
    idx, out = [], []
    for e, (r0, n) in enumerate(zip(starts, np.asarray(group_rows, np.int64))):
        if n == 0:
            continue
        rows = np.arange(r0, r0 + n)
        y = expert_rows_gemm(a_rows[rows], dequant_expert(w_q[e], w_s[e]))
        idx.append(rows)
        out.append(silu_mul(y) if silu else y)
    if not idx:
        width = w_q.shape[1] // (2 if silu else 1)
        return np.zeros(0, np.int64), np.zeros((0, width))
    return np.concatenate(idx), np.concatenate(out)
