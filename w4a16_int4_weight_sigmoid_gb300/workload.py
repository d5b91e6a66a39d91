"""Seeded synthetic inputs for the W4A16 MoE layer, and the named workloads.

This module only draws numbers.  It holds none of the layer's arithmetic
(no sigmoid, no routing, no dequantisation, no GEMM), so both the CUDA path
and the CPU oracle can be fed from it without sharing any method code.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used as a counter-based hash.  Value ``i`` of
stream ``s`` under seed ``seed`` is ``mix(key + (i + 1) * GAMMA)`` with
``key = mix(seed * GAMMA ^ s * C_STREAM)``.  Everything is 64-bit integer
arithmetic, so the raw words are identical on every machine.

Distributions (the Kimi-K2-shaped layer workloads):
  * activations x ~ N(0, 1), rounded to BF16 (round to nearest even);
  * router logits ~ N(0, 1) in FP32 (Box-Muller on two 53-bit uniforms);
  * expert score bias ~ U(-0.1, 0.1) in FP32;
  * INT4 weights ~ U{-8..7}: the packed bytes ARE the raw generator bytes,
    so every nibble is an exactly uniform two's-complement 4-bit value;
  * per-group-32 scales ~ U(0.005, 0.02), rounded to BF16.
The TP8 decode workload draws Zipf(1.1)-skewed expert popularity: a seeded
permutation ranks the experts, p_e is proportional to rank^-1.1, and the
logits are log p_e + Gumbel(0, 1), so the top-k before bias is a sample
without replacement proportional to p.

BF16 tensors are returned as ``uint16`` bit patterns.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
C_STREAM = np.uint64(0xD1B54A32D192ED03)
M1 = np.uint64(0xBF58476D1CE4E5B9)
M2 = np.uint64(0x94D049BB133111EB)

# stream ids, one per tensor
S_X, S_LOGITS, S_BIAS, S_Q13, S_S13, S_Q2, S_S2, S_PERM, S_GUMBEL = range(1, 10)


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= M1
    z ^= z >> np.uint64(27)
    z *= M2
    z ^= z >> np.uint64(31)
    return z


def words(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """Raw 64-bit words ``start .. start+n-1`` of (seed, stream)."""
    with np.errstate(over="ignore"):
        key = _mix(np.array([np.uint64(seed) * GAMMA ^ np.uint64(stream) * C_STREAM],
                            dtype=np.uint64))[0]
        ctr = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix(key + ctr * GAMMA)


def uniform01(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """float64 in [0, 1) from the top 53 bits of each word."""
    return (words(seed, stream, n, start) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """float64 N(0,1) by Box-Muller (cosine branch) on consecutive word pairs."""
    u = uniform01(seed, stream, 2 * n)
    u1 = 1.0 - u[0::2]          # (0, 1]
    u2 = u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to BF16 (nearest, ties to even); return uint16 bits."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))
    return (b >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(u) -> np.ndarray:
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def random_bytes(seed: int, stream: int, nbytes: int) -> np.ndarray:
    nw = (nbytes + 7) // 8
    return words(seed, stream, nw).view(np.uint8)[:nbytes]


# --------------------------------------------------------------------------
# named workloads
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class LayerShape:
    name: str
    M: int                 # tokens
    H: int                 # hidden size (K of gate/up, N of down)
    I: int                 # expert intermediate size on this GPU
    E_total: int           # experts the router scores
    E_local: int           # experts whose weights live on this GPU
    expert_begin: int      # first local expert id
    topk: int
    seed: int
    zipf: float = 0.0      # > 0: Zipf-skewed popularity (TP8 decode workload)
    block_m: int = 0       # 0: chosen by the library's tokens-per-expert policy


TINY = LayerShape("tiny_m16_h256_i128_e8_top2", 16, 256, 128, 8, 8, 0, 2, 0, block_m=16)
EP8_DECODE = LayerShape("kimi_k2_ep8_decode_m64_e48of384", 64, 7168, 2048, 384, 48, 0, 8, 1)
TP8_DECODE = LayerShape("kimi_k2_tp8_decode_m128_e384_i256_zipf1.1", 128, 7168, 256, 384, 384,
                        0, 8, 2, zipf=1.1)
EP8_PREFILL = LayerShape("kimi_k2_ep8_prefill_m8192_e48of384", 8192, 7168, 2048, 384, 48, 0, 8, 3)
WORKLOADS = {s.name: s for s in (TINY, EP8_DECODE, TP8_DECODE, EP8_PREFILL)}
# the Kimi-K2 layer shards the throughput metric is quoted on
LAYER_WORKLOADS = (EP8_DECODE, TP8_DECODE, EP8_PREFILL)

ROUTER_ALIGN_M = (1, 8, 128, 4096)
ROUTER_ALIGN_BM = (16, 64, 128)
ROUTER_ALIGN_E = 384
ROUTER_ALIGN_TOPK = 8
ROUTER_ALIGN_SEED = 4


def router_inputs(M: int, E_total: int, seed: int, zipf: float = 0.0):
    """logits FP32 [M, E_total], bias FP32 [E_total]."""
    if zipf > 0.0:
        perm = np.argsort(words(seed, S_PERM, E_total), kind="stable")
        rank = np.empty(E_total, dtype=np.int64)
        rank[perm] = np.arange(E_total)
        logp = -zipf * np.log(rank + 1.0)
        logp -= np.log(np.exp(logp).sum())
        u = uniform01(seed, S_GUMBEL, M * E_total).reshape(M, E_total)
        u = np.clip(u, 2.0 ** -53, 1.0 - 2.0 ** -53)
        logits = (logp[None, :] - np.log(-np.log(u))).astype(np.float32)
    else:
        logits = normal(seed, S_LOGITS, M * E_total).reshape(M, E_total).astype(np.float32)
    bias = (-0.1 + 0.2 * uniform01(seed, S_BIAS, E_total)).astype(np.float32)
    return logits, bias


def activations(M: int, H: int, seed: int) -> np.ndarray:
    """x BF16 bits [M, H], N(0, 1)."""
    return f32_to_bf16_bits(normal(seed, S_X, M * H).astype(np.float32)).reshape(M, H)


def int4_weights(E: int, N: int, K: int, seed: int, stream: int) -> np.ndarray:
    """Packed INT4 uint8 [E, N, K/2]: low nibble = even k, two's complement."""
    return random_bytes(seed, stream, E * N * K // 2).reshape(E, N, K // 2)


def group_scales(E: int, N: int, K: int, seed: int, stream: int, group: int = 32) -> np.ndarray:
    """BF16 bits [E, N, K/group], U(0.005, 0.02)."""
    n = E * N * (K // group)
    s = (0.005 + 0.015 * uniform01(seed, stream, n)).astype(np.float32)
    return f32_to_bf16_bits(s).reshape(E, N, K // group)


def layer_inputs(shape: LayerShape, seed: int | None = None, weights: bool = True):
    """All inputs of one MoE layer as numpy arrays (BF16 as uint16 bits).

    w13 rows 0..I-1 are the gate projection, rows I..2I-1 the up projection.
    """
    seed = shape.seed if seed is None else seed
    logits, bias = router_inputs(shape.M, shape.E_total, seed, shape.zipf)
    d = dict(x=activations(shape.M, shape.H, seed), logits=logits, bias=bias)
    if weights:
        E, H, I = shape.E_local, shape.H, shape.I
        d["w13_q"] = int4_weights(E, 2 * I, H, seed, S_Q13)
        d["w13_s"] = group_scales(E, 2 * I, H, seed, S_S13)
        d["w2_q"] = int4_weights(E, H, I, seed, S_Q2)
        d["w2_s"] = group_scales(E, H, I, seed, S_S2)
    return d
