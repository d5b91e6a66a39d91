"""Pins of the grouped-layout GEMM oracle against a brute-force scalar
computation written from the format's definition (nibbles and BF16 scales
decoded bit by bit here, not through oracle.quant), layout invariants, and
the one-expert case reducing to the plain expert GEMM."""
import math
import struct

import numpy as np
import pytest

import oracle
from w4a16_int4_weight_sigmoid_gb300 import workload as wl


def _bf16(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def _w(q, s, e, n, k):
    byte = int(q[e, n, k // 2])
    nib = byte & 0x0F if k % 2 == 0 else byte >> 4
    return (nib - 16 if nib >= 8 else nib) * _bf16(s[e, n, k // 32])


def _brute(a, q, s, layout, counts, max_m, silu):
    E, N, K = q.shape[0], q.shape[1], q.shape[2] * 2
    out = {}
    start = 0
    for e in range(E):
        r0 = e * max_m if layout == "masked" else start
        for r in range(r0, r0 + counts[e]):
            y = [sum(a[r, k] * _w(q, s, e, n, k) for k in range(K)) for n in range(N)]
            if silu:
                I = N // 2
                y = [y[i] / (1.0 + math.exp(-y[i])) * y[I + i] for i in range(I)]
            out[r] = y
        start += -(-counts[e] // 128) * 128
    return out


@pytest.mark.parametrize("layout,max_m", [("contiguous", 0), ("masked", 16)])
@pytest.mark.parametrize("silu", [False, True])
def test_grouped_gemm_brute_force(layout, max_m, silu):
    E, N, K = 3, 4, 64
    counts = [2, 0, 3]
    rows = 3 * max_m if layout == "masked" else 128 * 2 + 3
    rng = np.random.default_rng(5)
    a = rng.standard_normal((rows, K))
    q = wl.int4_weights(E, N, K, 61, wl.S_Q13)
    s = wl.group_scales(E, N, K, 62, wl.S_S13)
    idx, got = oracle.grouped_gemm(a, counts, q, s, layout, max_m, silu)
    ref = _brute(a, q, s, layout, counts, max_m, silu)
    assert sorted(idx.tolist()) == sorted(ref)
    for i, r in enumerate(idx):
        np.testing.assert_allclose(got[i], ref[int(r)], rtol=1e-12, atol=1e-12)


def test_group_starts_layout_invariants():
    c = np.array([0, 5, 128, 129, 0, 1])
    st = oracle.group_starts(c, "contiguous")
    assert np.all(st % 128 == 0)
    assert st[0] == 0 and np.all(np.diff(st) >= c[:-1]) and np.all(np.diff(st) - c[:-1] < 128)
    assert np.array_equal(oracle.group_starts(c, "masked", 160), np.arange(6) * 160)


def test_one_expert_contiguous_is_the_expert_gemm():
    M, N, K = 37, 32, 128
    a = np.random.default_rng(6).standard_normal((M, K))
    q = wl.int4_weights(1, N, K, 63, wl.S_Q13)
    s = wl.group_scales(1, N, K, 64, wl.S_S13)
    idx, got = oracle.grouped_gemm(a, [M], q, s, "contiguous")
    assert np.array_equal(idx, np.arange(M))
    np.testing.assert_array_equal(got, oracle.expert_rows_gemm(a, oracle.dequant_expert(q[0], s[0])))
