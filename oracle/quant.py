"""W4A16 weight format oracle: INT4 group-32 symmetric weights, BF16 scales.

Format ([Chord] "TL;DR": INT4 weights with BF16 activations; "런타임 고려사항":
the group-32 quantisation key; [Humming] "통합 양자화 표현": per-group INT4
weights paired with BF16 activations, weight format / scale granularity /
scale dtype / zero point as separate parameters).  Readings where the pages
are silent:

  * qweight uint8 [E, N, K/2]; byte k//2 of a row holds k even in its low
    nibble and k odd in its high nibble; a nibble is a two's-complement
    integer in -8..7;
  * scales BF16 [E, N, K/32]; symmetric (no zero point):
    W[e, n, k] = q[e, n, k] * s[e, n, k // 32], exact in FP64.
"""
from __future__ import annotations

import numpy as np

GROUP = 32


def bf16_to_f64(u16) -> np.ndarray:
    """BF16 bit patterns (uint16) -> exact float64 values."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def f64_to_bf16_f64(a) -> np.ndarray:
    """Round float64 to the nearest BF16 value (ties to even), returned as float64.
    Used only by the BF16-emulating reference that estimates achievable error."""
    a = np.asarray(a, dtype=np.float64)
    m, e = np.frexp(a)                      # a = m * 2^e, 0.5 <= |m| < 1
    q = np.round(m * 256.0) / 256.0         # 8 significant bits, ties to even
    return np.ldexp(q, e)


def unpack_int4(q) -> np.ndarray:
    """uint8 [..., K/2] -> int8 [..., K] with the nibble order above."""
    q = np.asarray(q, dtype=np.uint8)
    lo = (q & 0x0F).astype(np.int16)
    hi = (q >> 4).astype(np.int16)
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), dtype=np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def dequant_expert(q, s, group: int = GROUP) -> np.ndarray:
    """One expert: uint8 [N, K/2], BF16 [N, K/group] -> float64 [N, K]."""
    w = unpack_int4(q).astype(np.float64)
    sc = bf16_to_f64(s)
    N, K = w.shape
    return (w.reshape(N, K // group, group) * sc[:, :, None]).reshape(N, K)


def dequant(q, s, group: int = GROUP) -> np.ndarray:
    """All experts: [E, N, K/2], [E, N, K/group] -> float64 [E, N, K]."""
    return np.stack([dequant_expert(q[e], s[e], group) for e in range(q.shape[0])])
