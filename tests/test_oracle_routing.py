"""Pins for the router oracle (CPU only).

The sigmoid is pinned to the FP64 definition within a stated ulp bound; the
top-k selection to a brute-force Python sort; the weights to closed forms
and hand-worked cases (tests/golden/route_hand.json); and the outputs to the
invariants every routing must satisfy.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle.routing import exp_binary32, sigmoid_binary32
from w4a16_int4_weight_sigmoid_gb300 import workload as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ulps(a32, ref64):
    a32 = np.asarray(a32, np.float32)
    sp = np.spacing(np.abs(ref64).astype(np.float32)).astype(np.float64)
    return np.abs(a32.astype(np.float64) - ref64) / sp


def test_exp_binary32_within_two_ulp_of_fp64():
    y = np.linspace(-87.0, 87.0, 400_001, dtype=np.float64).astype(np.float32)
    ref = np.exp(y.astype(np.float64))
    assert _ulps(exp_binary32(y), ref).max() <= 2.0
    assert exp_binary32(np.float32(0.0)) == np.float32(1.0)
    # exact powers of two where the reduction leaves r = 0
    for n in (-20, -1, 1, 7, 30):
        y = np.float32(n * math.log(2.0))
        assert _ulps(exp_binary32(y), math.exp(float(y))) <= 2.0


def test_sigmoid_binary32_accuracy_and_shape():
    x = np.concatenate([np.linspace(-87, 87, 1_000_001), np.linspace(-2, 2, 100_001)]).astype(np.float32)
    ref = 1.0 / (1.0 + np.exp(-x.astype(np.float64)))
    assert _ulps(sigmoid_binary32(x), ref).max() <= 4.0
    xs = np.sort(x)
    assert np.all(np.diff(sigmoid_binary32(xs)) >= 0), "sigmoid must be monotone"
    assert sigmoid_binary32(np.float32(0.0)) == np.float32(0.5)
    assert np.all(sigmoid_binary32(np.float32([17.5, 50, 1e4, np.inf])) == 1.0)
    s = sigmoid_binary32(x)
    t = sigmoid_binary32(-x)
    assert np.max(np.abs(s.astype(np.float64) + t - 1.0)) <= 2.0 ** -23
    # the clamp: below -87 the score is the score at -87 (tiny, positive)
    assert sigmoid_binary32(np.float32(-500.0)) == sigmoid_binary32(np.float32(-87.0))
    assert 0.0 < float(sigmoid_binary32(np.float32(-87.0))) < 2e-38


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "route_hand.json")))["cases"],
                         ids=lambda c: c["name"])
def test_route_hand_cases(case):
    logits = np.array([case["logits"]], dtype=np.float32)
    bias = np.array(case["bias"], dtype=np.float32)
    w, ids, _ = oracle.route(logits, bias, case["k"])
    assert ids[0].tolist() == case["ids"]
    exp = np.array(case["weights"], dtype=np.float64)
    if case["ulp"] == 0:
        assert w[0].astype(np.float64).tolist() == exp.tolist()
    else:
        assert _ulps(w[0], exp).max() <= case["ulp"]


def _brute_force_route(logits, bias, k):
    """Independent restatement: a Python sort of (-key, id) per token and a
    left-to-right binary32 sum with numpy scalars."""
    s = sigmoid_binary32(logits)
    M, E = logits.shape
    ids = np.zeros((M, k), np.int32)
    w = np.zeros((M, k), np.float32)
    for t in range(M):
        keys = [(-(float(np.float32(s[t, e]) + np.float32(bias[e]))), e) for e in range(E)]
        top = [e for _, e in sorted(keys)[:k]]
        ids[t] = top
        S = np.float32(0.0)
        for e in top:
            S = np.float32(S + s[t, e])
        w[t] = [np.float32(s[t, e]) / S for e in top]
    return w, ids


@pytest.mark.parametrize("M,E,k,seed,zipf", [(16, 8, 2, 0, 0.0), (8, 384, 8, 4, 0.0),
                                            (128, 384, 8, 4, 0.0), (64, 384, 8, 2, 1.1),
                                            (5, 33, 32, 9, 0.0), (3, 1, 1, 5, 0.0)])
def test_route_matches_brute_force(M, E, k, seed, zipf):
    logits, bias = wl.router_inputs(M, E, seed, zipf)
    w, ids, _ = oracle.route(logits, bias, k)
    bw, bids = _brute_force_route(logits, bias, k)
    assert np.array_equal(ids, bids)
    assert np.array_equal(w.view(np.uint32), bw.view(np.uint32))


def test_route_ties_among_equal_keys_pick_lower_ids():
    logits = np.zeros((4, 384), np.float32)
    bias = np.zeros(384, np.float32)
    bias[[300, 7, 100]] = 0.05
    _, ids, _ = oracle.route(logits, bias, 8)
    for t in range(4):
        assert ids[t].tolist() == [7, 100, 300, 0, 1, 2, 3, 4]


@pytest.mark.parametrize("M", wl.ROUTER_ALIGN_M)
def test_route_invariants(M):
    k, E = wl.ROUTER_ALIGN_TOPK, wl.ROUTER_ALIGN_E
    logits, bias = wl.router_inputs(M, E, wl.ROUTER_ALIGN_SEED)
    w, ids, s = oracle.route(logits, bias, k)
    assert ids.shape == (M, k) and w.shape == (M, k)
    assert ids.min() >= 0 and ids.max() < E
    assert all(len(set(r)) == k for r in ids.tolist())
    assert np.all(w > 0)
    assert np.max(np.abs(w.astype(np.float64).sum(1) - 1.0)) <= 2 * k * 2.0 ** -24
    key = s + bias[None, :]
    ksel = np.take_along_axis(key, ids, 1)
    assert np.all(np.diff(ksel, axis=1) <= 0), "ids are emitted in rank order"
    # no unselected expert beats the k-th selected key
    mask = np.ones_like(key, bool)
    np.put_along_axis(mask, ids, False, 1)
    assert np.all(np.where(mask, key, -np.inf).max(1) <= ksel[:, -1])


def test_route_selection_stable_against_fp64_scores():
    """Report-style check: binary32 scores give the same selections as FP64
    scores on the router workload (differences would only be near-ties)."""
    k, E = wl.ROUTER_ALIGN_TOPK, wl.ROUTER_ALIGN_E
    logits, bias = wl.router_inputs(4096, E, wl.ROUTER_ALIGN_SEED)
    _, ids, _ = oracle.route(logits, bias, k)
    key64 = 1.0 / (1.0 + np.exp(-logits.astype(np.float64))) + bias.astype(np.float64)
    ids64 = np.argsort(-key64, axis=1, kind="stable")[:, :k]
    differ = np.sum(np.any(np.sort(ids, 1) != np.sort(ids64, 1), axis=1))
    assert differ <= 2
