"""MoE layer oracle: gate/up GEMM, SiLU*mul, down GEMM, top-k weighted sum.

For each kept assignment (t, j) with local expert e (see align.py):
  g = W13[e, 0:I] . x_t,  u = W13[e, I:2I] . x_t       (gate rows first)
  h = silu(g) * u,  silu(z) = z / (1 + e^-z)
  y = W2[e] . h
  out_t += w[t, j] * y
All in FP64 with exactly dequantised weights (quant.py); x is BF16.  The
indexed GEMMs are [Chord] "핵심 기여" / "인덱스 커널 기법" (gate/up and down
reported separately in "성능 요약"); the weighted sum is `moe_fused_mul_sum`
([HumPR] "왜 이게 좋은가", item 3).  The gate-first row order of W13 and the
SiLU gate are readings of the Kimi-K2 expert MLP; the pages do not print it.
Assignments whose expert is not local contribute nothing to this shard's out.
"""
from __future__ import annotations

import numpy as np

from .quant import bf16_to_f64, dequant_expert, f64_to_bf16_f64
from .routing import route


def silu(z) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_rows_gemm(a_rows, W) -> np.ndarray:
    """rows [R, K] (float64) times one expert's weights W [N, K] -> [R, N]."""
    return np.asarray(a_rows, np.float64) @ np.asarray(W, np.float64).T


def silu_mul(gu) -> np.ndarray:
    """[R, 2I] gate|up -> [R, I]."""
    gu = np.asarray(gu, np.float64)
    I = gu.shape[1] // 2
    return silu(gu[:, :I]) * gu[:, I:]


def moe_sum(y_rows, topk_weights, sorted_positions, M: int, topk: int) -> np.ndarray:
    """out[t] = sum_j w[t, j] * y[pos(t, j)] over kept assignments (j ascending)."""
    y_rows = np.asarray(y_rows, np.float64)
    out = np.zeros((M, y_rows.shape[1]), dtype=np.float64)
    w = np.asarray(topk_weights, np.float64).reshape(M, topk)
    pos = np.asarray(sorted_positions).reshape(M, topk)
    for j in range(topk):
        keep = pos[:, j] >= 0
        out[keep] += w[keep, j, None] * y_rows[pos[keep, j]]
    return out


def _expert_mlp(X, e, w13_q, w13_s, w2_q, w2_s, round_bf16):
    W13 = dequant_expert(w13_q[e], w13_s[e])
    W2 = dequant_expert(w2_q[e], w2_s[e])
    if round_bf16:
        W13, W2 = f64_to_bf16_f64(W13), f64_to_bf16_f64(W2)
    h = silu_mul(expert_rows_gemm(X, W13))
    if round_bf16:
        h = f64_to_bf16_f64(h)
    return expert_rows_gemm(h, W2)


def moe_layer_tokens(tokens, x, logits, bias, w13_q, w13_s, w2_q, w2_s, topk: int,
                     expert_begin: int = 0, round_bf16: bool = False):
    """Layer output FP64 [len(tokens), H] for a subset of tokens only.

    Routing is per token, so the subset's outputs equal those rows of the
    full layer.  With round_bf16=True the dequantised weights and h are
    rounded to BF16 (an emulation of a BF16 tensor-core path, used only to
    estimate the error such a path can reach; not the reference result).
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    E_local = w13_q.shape[0]
    w, ids, _ = route(np.asarray(logits)[tokens], bias, topk)
    X = bf16_to_f64(np.asarray(x)[tokens])
    out = np.zeros((tokens.size, w2_q.shape[1]), dtype=np.float64)
    local = ids.astype(np.int64) - expert_begin
    for e in np.unique(local[(local >= 0) & (local < E_local)]):
        rows, slots = np.nonzero(local == e)
        y = _expert_mlp(X[rows], int(e), w13_q, w13_s, w2_q, w2_s, round_bf16)
        np.add.at(out, rows, w[rows, slots, None].astype(np.float64) * y)
    return out


def moe_layer(x, logits, bias, w13_q, w13_s, w2_q, w2_s, topk: int,
              expert_begin: int = 0, round_bf16: bool = False):
    """Full layer: returns (out FP64 [M, H], topk_weights, topk_ids)."""
    M = np.asarray(x).shape[0]
    out = moe_layer_tokens(np.arange(M), x, logits, bias, w13_q, w13_s, w2_q, w2_s,
                           topk, expert_begin, round_bf16)
    w, ids, _ = route(logits, bias, topk)
    return out, w, ids
