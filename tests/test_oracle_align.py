"""Pins for the align oracle (CPU only): hand-worked cases
(tests/golden/align_hand.json), a brute-force Python construction, and the
invariants of moe_align_block_size."""
import json
import os

import numpy as np
import pytest

import oracle
from w4a16_int4_weight_sigmoid_gb300 import workload as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "align_hand.json")))["cases"],
                         ids=lambda c: c["name"])
def test_align_hand_cases(case):
    r = oracle.moe_align(np.array(case["topk_ids"]), case["expert_begin"], case["E_local"],
                         case["block_m"])
    assert r["expert_counts"].tolist() == case["counts"]
    assert r["expert_offsets"].tolist() == case["offsets"]
    assert r["num_tokens_post_padded"] == case["ntpp"]
    assert r["sorted_token_ids"].tolist() == case["sorted_token_ids"]
    assert r["expert_ids"].tolist() == case["expert_ids"]
    assert r["sorted_positions"].tolist() == case["sorted_positions"]


def _brute_force_align(topk_ids, begin, E_local, bm):
    M, k = len(topk_ids), len(topk_ids[0])
    rows, eids = [], []
    for e in range(E_local):
        mine = [t * k + j for t in range(M) for j in range(k) if topk_ids[t][j] == begin + e]
        if not mine:
            continue
        nblk = -(-len(mine) // bm)
        rows += mine + [M * k] * (nblk * bm - len(mine))
        eids += [e] * nblk
    return rows, eids


@pytest.mark.parametrize("M,E,k,begin,E_local,bm", [(16, 8, 2, 0, 8, 16), (8, 384, 8, 0, 384, 16),
                                                    (37, 384, 8, 48, 48, 64), (128, 384, 8, 0, 384, 128),
                                                    (5, 16, 4, 3, 5, 8), (1, 384, 8, 0, 384, 16)])
def test_align_matches_brute_force(M, E, k, begin, E_local, bm):
    logits, bias = wl.router_inputs(M, E, 11)
    _, ids, _ = oracle.route(logits, bias, k)
    r = oracle.moe_align(ids, begin, E_local, bm)
    rows, eids = _brute_force_align(ids.tolist(), begin, E_local, bm)
    assert r["sorted_token_ids"].tolist() == rows
    assert r["expert_ids"].tolist() == eids
    assert r["num_tokens_post_padded"] == len(rows)


@pytest.mark.parametrize("M", wl.ROUTER_ALIGN_M)
@pytest.mark.parametrize("bm", wl.ROUTER_ALIGN_BM)
def test_align_invariants(M, bm):
    k, E = wl.ROUTER_ALIGN_TOPK, wl.ROUTER_ALIGN_E
    logits, bias = wl.router_inputs(M, E, wl.ROUTER_ALIGN_SEED)
    _, ids, _ = oracle.route(logits, bias, k)
    r = oracle.moe_align(ids, 0, E, bm)
    st, off, cnt = r["sorted_token_ids"], r["expert_offsets"], r["expert_counts"]
    ntpp = r["num_tokens_post_padded"]
    assert ntpp == off[-1] <= oracle.align_capacity(M, k, E, bm)
    assert np.all((off[1:] - off[:-1]) % bm == 0)
    assert cnt.sum() == M * k
    real = st[st != M * k]
    assert np.array_equal(np.sort(real), np.arange(M * k)), "every assignment exactly once"
    for e in range(E):
        seg = st[off[e]:off[e] + cnt[e]]
        assert np.all(np.diff(seg) > 0), "stable: ascending flat index within an expert"
        assert np.all(ids.reshape(-1)[seg] == e)
        assert np.all(st[off[e] + cnt[e]:off[e + 1]] == M * k)
    eid = r["expert_ids"]
    assert eid.size == ntpp // bm and np.all(np.diff(eid) >= 0)
    for b, e in enumerate(eid):
        assert off[e] <= b * bm < off[e + 1]
    pos = r["sorted_positions"]
    assert np.array_equal(st[pos], np.arange(M * k))


def test_align_capacity_bound_is_tight():
    # every assignment on its own expert: each needs a full block
    M, k, E, bm = 4, 2, 8, 16
    ids = np.arange(M * k).reshape(M, k)
    r = oracle.moe_align(ids, 0, E, bm)
    assert r["num_tokens_post_padded"] == oracle.align_capacity(M, k, E, bm) == M * k * bm


def test_align_empty_shard():
    ids = np.array([[0, 1], [1, 2]])
    r = oracle.moe_align(ids, 10, 4, 16)
    assert r["num_tokens_post_padded"] == 0
    assert r["sorted_token_ids"].size == 0 and r["expert_ids"].size == 0
    assert np.all(r["sorted_positions"] == -1)
