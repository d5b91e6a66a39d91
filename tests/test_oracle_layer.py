"""Pins for the weight-format and layer oracle (CPU only).

Closed forms (identity layer, hand-worked single-expert case), a pure-Python
brute force on tiny inputs that decodes nibbles with its own bit arithmetic,
exact invariances (power-of-two scales, expert and token permutations), and
the tolerance pin: a BF16 emulation meets the parity bar while planted
mistakes miss it.
"""
import math
import struct

import numpy as np
import pytest

import oracle
from oracle.quant import f64_to_bf16_f64
from w4a16_int4_weight_sigmoid_gb300 import workload as wl

REL_FROB_BAR = 5e-3
MAXABS_BAR = 1e-2


def _bf16_bits(v: float) -> int:
    return struct.unpack("<I", struct.pack("<f", v))[0] >> 16   # exact for BF16 values


def _pack(qint):
    """int array [..., K] in -8..7 -> uint8 [..., K/2] (low nibble = even k)."""
    q = (np.asarray(qint, np.int64) & 0xF).astype(np.uint8)
    return (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)


def test_unpack_int4_hand_case():
    q = np.array([0x8F, 0x70, 0x01], np.uint8)
    assert oracle.unpack_int4(q).tolist() == [-1, -8, 0, 7, 1, 0]


def test_unpack_int4_all_bytes_by_sign_extension():
    b = np.arange(256, dtype=np.uint8)
    out = oracle.unpack_int4(b[:, None])
    # sign-extend each nibble through an int8 arithmetic shift
    lo = ((b << 4).astype(np.uint8).view(np.int8) >> 4).astype(np.int64)
    hi = (b.view(np.int8) >> 4).astype(np.int64)
    assert np.array_equal(out[:, 0], lo) and np.array_equal(out[:, 1], hi)


def test_bf16_decode_and_round():
    assert oracle.bf16_to_f64(np.array([0x3F80, 0xC000, 0x0000, 0x4300], np.uint16)).tolist() == \
        [1.0, -2.0, 0.0, 128.0]
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -9, -(1 + 2 ** -8 + 2 ** -12), 0.1])
    r = f64_to_bf16_f64(x)
    assert r[0] == 1.0                          # tie -> even
    assert r[1] == 1 + 2 ** -7                  # tie -> even (odd neighbour below)
    assert r[2] == -(1 + 2 ** -7)
    assert abs(r[3] - 0.1) <= 2 ** -4 * 2 ** -8 and _bf16_bits(r[3]) == 0x3DCD


def test_dequant_group_scaling_hand_case():
    K = 64
    q = np.zeros((1, K), np.int64)
    q[0, 0], q[0, 31], q[0, 32], q[0, 63] = 3, -8, 7, -1
    s = np.array([[_bf16_bits(0.5), _bf16_bits(-2.0)]], np.uint16)
    W = oracle.dequant_expert(_pack(q), s)
    exp = np.zeros((1, K))
    exp[0, 0], exp[0, 31], exp[0, 32], exp[0, 63] = 1.5, -4.0, -14.0, 2.0
    assert np.array_equal(W, exp)


def _identity_weights(E, D, up_mult=1):
    q13 = np.zeros((E, 2 * D, D), np.int64)
    q2 = np.zeros((E, D, D), np.int64)
    for e in range(E):
        q13[e, np.arange(D), np.arange(D)] = 1
        q13[e, D + np.arange(D), np.arange(D)] = up_mult
        q2[e, np.arange(D), np.arange(D)] = 1
    one = _bf16_bits(1.0)
    s13 = np.full((E, 2 * D, D // 32), one, np.uint16)
    s2 = np.full((E, D, D // 32), one, np.uint16)
    return _pack(q13), s13, _pack(q2), s2


def test_identity_layer_closed_form():
    """W_gate = W_up = W_down = identity: out = silu(x) * x * sum(w) = silu(x) * x."""
    M, D, E, k = 7, 32, 4, 2
    x = wl.activations(M, D, 3)
    logits, bias = wl.router_inputs(M, E, 3)
    q13, s13, q2, s2 = _identity_weights(E, D)
    out, w, _ = oracle.moe_layer(x, logits, bias, q13, s13, q2, s2, k)
    xf = oracle.bf16_to_f64(x)
    exp = xf / (1 + np.exp(-xf)) * xf
    assert np.allclose(out, exp * w.astype(np.float64).sum(1, keepdims=True), rtol=1e-13, atol=0)
    assert np.allclose(out, exp, rtol=4 * k * 2.0 ** -24, atol=1e-300)


def test_single_expert_hand_case():
    """M=1, E=2, k=1, H=I=32, x = 1: expert 1 (the larger logit) has gate = I,
    up = 2I, down = I, so every output is 2 * silu(1) = 2 / (1 + e^-1);
    expert 0 is all zeros and must not be used."""
    D = 32
    x = np.full((1, D), _bf16_bits(1.0), np.uint16)
    logits = np.array([[0.0, 1.0]], np.float32)
    bias = np.zeros(2, np.float32)
    q13, s13, q2, s2 = _identity_weights(2, D, up_mult=2)
    q13[0] = 0
    q2[0] = 0
    out, w, ids = oracle.moe_layer(x, logits, bias, q13, s13, q2, s2, 1)
    assert ids.tolist() == [[1]] and w.tolist() == [[1.0]]
    assert np.all(out == 2.0 / (1.0 + math.exp(-1.0)))


def _brute_force_layer(x, logits, bias, q13, s13, q2, s2, k, begin):
    """Pure-Python loops: own nibble decode, own BF16 decode, explicit sums."""
    def bf(u):
        return struct.unpack("<f", struct.pack("<I", int(u) << 16))[0]

    def w_at(qb, sb, n, kk):
        byte = int(qb[n][kk // 2])
        nib = (byte >> (4 * (kk % 2))) & 15
        val = nib - 16 if nib & 8 else nib
        return val * bf(sb[n][kk // 32])

    M, H = x.shape
    E_local = q13.shape[0]
    I = q13.shape[1] // 2
    w, ids, _ = oracle.route(logits, bias, k)     # routing pinned separately
    out = [[0.0] * H for _ in range(M)]
    for t in range(M):
        xt = [bf(v) for v in x[t]]
        for j in range(k):
            e = int(ids[t][j]) - begin
            if not 0 <= e < E_local:
                continue
            g = [sum(w_at(q13[e], s13[e], i, kk) * xt[kk] for kk in range(H)) for i in range(I)]
            u = [sum(w_at(q13[e], s13[e], I + i, kk) * xt[kk] for kk in range(H)) for i in range(I)]
            h = [g[i] / (1.0 + math.exp(-g[i])) * u[i] for i in range(I)]
            for n in range(H):
                y = sum(w_at(q2[e], s2[e], n, i) * h[i] for i in range(I))
                out[t][n] += float(w[t][j]) * y
    return np.array(out)


@pytest.mark.parametrize("begin,E_local", [(0, 3), (1, 2)])
def test_layer_matches_pure_python_brute_force(begin, E_local):
    M, H, I, E, k = 3, 64, 32, 3, 2
    x = wl.activations(M, H, 5)
    logits, bias = wl.router_inputs(M, E, 5)
    q13 = wl.int4_weights(E_local, 2 * I, H, 5, wl.S_Q13)
    s13 = wl.group_scales(E_local, 2 * I, H, 5, wl.S_S13)
    q2 = wl.int4_weights(E_local, H, I, 5, wl.S_Q2)
    s2 = wl.group_scales(E_local, H, I, 5, wl.S_S2)
    out, _, _ = oracle.moe_layer(x, logits, bias, q13, s13, q2, s2, k, begin)
    bf = _brute_force_layer(x, logits, bias, q13, s13, q2, s2, k, begin)
    assert np.allclose(out, bf, rtol=1e-12, atol=1e-12 * np.abs(bf).max())


@pytest.fixture(scope="module")
def tiny():
    return wl.layer_inputs(wl.TINY)


def _layer(d, **kw):
    return oracle.moe_layer(d["x"], d["logits"], d["bias"], d["w13_q"], d["w13_s"], d["w2_q"],
                            d["w2_s"], wl.TINY.topk, **kw)[0]


def test_power_of_two_scale_invariance(tiny):
    out = _layer(tiny)
    d = dict(tiny)
    d["w2_s"] = (tiny["w2_s"].astype(np.uint32) + 0x80).astype(np.uint16)   # exponent + 1
    assert np.array_equal(_layer(d), 2.0 * out)


def test_expert_permutation_invariance(tiny):
    out = _layer(tiny)
    perm = np.array([3, 0, 7, 5, 1, 6, 2, 4])      # new expert p holds old expert perm[p]
    d = dict(tiny)
    for key in ("w13_q", "w13_s", "w2_q", "w2_s"):
        d[key] = tiny[key][perm]
    d["logits"] = tiny["logits"][:, perm]
    d["bias"] = tiny["bias"][perm]
    assert np.allclose(_layer(d), out, rtol=1e-13, atol=1e-13 * np.abs(out).max())


def test_token_permutation_equivariance(tiny):
    out = _layer(tiny)
    perm = np.random.default_rng(0).permutation(wl.TINY.M)
    d = dict(tiny)
    d["x"], d["logits"] = tiny["x"][perm], tiny["logits"][perm]
    assert np.allclose(_layer(d), out[perm], rtol=1e-13, atol=1e-13 * np.abs(out).max())


def test_moe_sum_hand_case():
    y = np.array([[1.0, 2.0], [10.0, 20.0], [100.0, 200.0], [0.0, 0.0]])
    w = np.array([[0.25, 0.75], [0.5, 0.5]])
    pos = np.array([[2, 0], [-1, 1]])
    out = oracle.moe_sum(y, w, pos, 2, 2)
    assert out.tolist() == [[25.75, 51.5], [5.0, 10.0]]


def _errs(a, ref):
    return (np.linalg.norm(a - ref) / np.linalg.norm(ref), np.abs(a - ref).max() / np.abs(ref).max())


def test_tolerance_bar_separates_bf16_path_from_mistakes(tiny):
    """A BF16 tensor-core path (weights and h rounded to BF16, output to BF16)
    meets the bar; plausible kernel mistakes (gate/up swapped, a dropped
    scale group, a wrong expert, a transposed nibble order) miss it."""
    ref = _layer(tiny)
    emu = f64_to_bf16_f64(_layer(tiny, round_bf16=True))
    fro, mx = _errs(emu, ref)
    assert 1e-4 < fro < REL_FROB_BAR and mx < MAXABS_BAR
    I = wl.TINY.I
    bad = []
    d = dict(tiny); d["w13_q"] = np.concatenate([tiny["w13_q"][:, I:], tiny["w13_q"][:, :I]], 1)
    d["w13_s"] = np.concatenate([tiny["w13_s"][:, I:], tiny["w13_s"][:, :I]], 1); bad.append(d)
    d = dict(tiny); s = tiny["w2_s"].copy(); s[:, :, 1] = s[:, :, 0]; d["w2_s"] = s; bad.append(d)
    d = dict(tiny); d["w2_q"] = np.roll(tiny["w2_q"], 1, axis=0); d["w2_s"] = np.roll(tiny["w2_s"], 1, 0)
    bad.append(d)
    d = dict(tiny); q = tiny["w13_q"]; d["w13_q"] = ((q >> 4) | (q << 4)).astype(np.uint8); bad.append(d)
    for d in bad:
        fro, mx = _errs(_layer(d), ref)
        assert fro > 10 * REL_FROB_BAR
