"""GPU parity: router and align kernels against the oracle, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from w4a16_int4_weight_sigmoid_gb300 import chord
from w4a16_int4_weight_sigmoid_gb300 import workload as wl

from gpu_util import ensure_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def gpu_route(logits, bias, k):
    lg = torch.from_numpy(logits).cuda()
    bs = torch.from_numpy(bias).cuda()
    M = logits.shape[0]
    w = torch.full((M, k), -1.0, dtype=torch.float32, device="cuda")
    ids = torch.full((M, k), -1, dtype=torch.int32, device="cuda")
    chord.chord_moe_route(lg, bs, k, w, ids)
    torch.cuda.synchronize()
    return w.cpu().numpy(), ids.cpu().numpy()


def check_route(logits, bias, k):
    w, ids, _ = oracle.route(logits, bias, k)
    for _ in range(2):   # twice: catches nondeterminism
        gw, gids = gpu_route(logits, bias, k)
        assert np.array_equal(gids, ids)
        assert np.array_equal(gw.view(np.uint32), w.view(np.uint32))


@pytest.mark.parametrize("M", wl.ROUTER_ALIGN_M)
def test_route_router_workload(M):
    logits, bias = wl.router_inputs(M, wl.ROUTER_ALIGN_E, wl.ROUTER_ALIGN_SEED)
    check_route(logits, bias, wl.ROUTER_ALIGN_TOPK)


@pytest.mark.parametrize("shape", [wl.TINY, wl.EP8_DECODE, wl.TP8_DECODE, wl.EP8_PREFILL],
                         ids=lambda s: s.name)
def test_route_layer_workloads(shape):
    logits, bias = wl.router_inputs(shape.M, shape.E_total, shape.seed, shape.zipf)
    check_route(logits, bias, shape.topk)


@pytest.mark.parametrize("M,E,k", [(7, 1, 1), (5, 33, 32), (9, 64, 6), (3, 1000, 17), (33, 256, 8)])
def test_route_odd_shapes(M, E, k):
    logits, bias = wl.router_inputs(M, E, 21)
    check_route(logits, bias, k)


def test_route_special_values():
    vals = np.float32([0.0, -0.0, 87.0, -87.0, 88.0, -88.0, 100.0, -100.0, 1e-30, -1e-30, 17.0,
                       -17.0, 0.5, -0.5, 3e38, -3e38])
    logits = np.tile(vals, (4, 24)).astype(np.float32)            # 384 columns, many ties
    bias = np.zeros(384, np.float32)
    bias[::7] = 0.1
    bias[::11] = -0.05
    check_route(logits, bias, 8)
    # sweep the sigmoid through the weights of a top-32 route over 32 experts
    x = np.linspace(-90, 90, 64 * 32, dtype=np.float32).reshape(64, 32)
    check_route(x, np.zeros(32, np.float32), 32)


def test_route_empty():
    gw, gids = gpu_route(np.zeros((0, 384), np.float32), np.zeros(384, np.float32), 8)
    assert gw.shape == (0, 8)


def gpu_align(ids_np, begin, E_local, bm, M=None):
    M = ids_np.shape[0] if M is None else M
    k = ids_np.shape[1]
    cap = chord.chord_moe_align_capacity(M, k, E_local, bm)
    dev = "cuda"
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, np.int32)).to(dev)
    st = torch.full((max(cap, 1),), -7, dtype=torch.int32, device=dev)
    eid = torch.full((max(cap // bm, 1),), -7, dtype=torch.int32, device=dev)
    ntpp = torch.full((1,), -7, dtype=torch.int32, device=dev)
    cnt = torch.full((E_local,), -7, dtype=torch.int32, device=dev)
    off = torch.full((E_local + 1,), -7, dtype=torch.int32, device=dev)
    pos = torch.full((max(M * k, 1),), -7, dtype=torch.int32, device=dev)
    wsb = chord.chord_moe_align_workspace_bytes(M, k, E_local)
    ws = torch.full((max(wsb, 16),), 0x5A, dtype=torch.uint8, device=dev) if wsb else None
    chord.chord_moe_align(ids, begin, E_local, bm, st[:cap] if cap else st, eid, ntpp, cnt, off,
                          pos, ws)
    torch.cuda.synchronize()
    n = int(ntpp.item())
    return dict(sorted_token_ids=st.cpu().numpy()[:n], expert_ids=eid.cpu().numpy()[:n // bm],
                num_tokens_post_padded=n, expert_counts=cnt.cpu().numpy(),
                expert_offsets=off.cpu().numpy(), sorted_positions=pos.cpu().numpy()[:M * k])


def check_align(ids_np, begin, E_local, bm):
    ref = oracle.moe_align(ids_np, begin, E_local, bm)
    for _ in range(2):
        got = gpu_align(ids_np, begin, E_local, bm)
        assert got["num_tokens_post_padded"] == ref["num_tokens_post_padded"]
        for key in ("expert_counts", "expert_offsets", "sorted_token_ids", "expert_ids",
                    "sorted_positions"):
            assert np.array_equal(got[key], ref[key]), key


@pytest.mark.parametrize("M", wl.ROUTER_ALIGN_M)
@pytest.mark.parametrize("bm", wl.ROUTER_ALIGN_BM)
def test_align_router_workload(M, bm):
    logits, bias = wl.router_inputs(M, wl.ROUTER_ALIGN_E, wl.ROUTER_ALIGN_SEED)
    _, ids, _ = oracle.route(logits, bias, wl.ROUTER_ALIGN_TOPK)
    check_align(ids, 0, wl.ROUTER_ALIGN_E, bm)


@pytest.mark.parametrize("shape", [wl.TINY, wl.EP8_DECODE, wl.TP8_DECODE, wl.EP8_PREFILL],
                         ids=lambda s: s.name)
def test_align_layer_workloads(shape):
    logits, bias = wl.router_inputs(shape.M, shape.E_total, shape.seed, shape.zipf)
    _, ids, _ = oracle.route(logits, bias, shape.topk)
    check_align(ids, shape.expert_begin, shape.E_local, 16)


@pytest.mark.parametrize("M,k,E,begin,E_local,bm", [
    (1000, 8, 384, 96, 48, 8),      # 8000 assignments: 8 chunks of 1024, ragged, EP shard
    (513, 8, 384, 0, 384, 32),      # 4104: just over one CTA's 4096, 5 chunks
    (3, 2, 4, 0, 4, 128),
    (40, 4, 1024, 0, 1024, 16),     # widest shard
    (6000, 6, 16, 0, 16, 64),       # heavy per-expert counts over 36 chunks
    # one chunk, by assignments per thread (512 threads): 1 (n <= 512), 2
    # (n <= 1024), 8; and by the cross-warp prefix: lane scans (E_local <= 64)
    # or a loop per expert
    (64, 8, 384, 0, 48, 8),         # n = 512, 1 per thread, lane scans
    (65, 8, 384, 0, 48, 8),         # n = 520, 2 per thread
    (128, 8, 384, 0, 64, 16),       # n = 1024, 2 per thread, E_local = 64
    (129, 8, 384, 0, 65, 16),       # n = 1032, 8 per thread, loop prefix
    (250, 8, 384, 16, 48, 16),      # n = 2000, 8 per thread, lane scans
])
def test_align_edge_shapes(M, k, E, begin, E_local, bm):
    logits, bias = wl.router_inputs(M, E, 31)
    _, ids, _ = oracle.route(logits, bias, k)
    check_align(ids, begin, E_local, bm)


def test_align_all_dropped_and_empty():
    ids = np.array([[0, 1], [1, 2]], np.int32)
    check_align(ids, 10, 4, 16)
    got = gpu_align(np.zeros((0, 8), np.int32), 0, 384, 16)
    assert got["num_tokens_post_padded"] == 0 and np.all(got["expert_counts"] == 0)
    assert np.all(got["expert_offsets"] == 0)


# ------------------------------------------------------- fused route + align
def gpu_route_align(logits, bias, k, begin, E_local, bm):
    M, E = logits.shape
    dev = "cuda"
    cap = chord.chord_moe_align_capacity(M, k, E_local, bm)
    lg, bs = torch.from_numpy(logits).to(dev), torch.from_numpy(bias).to(dev)
    w = torch.full((M, k), -1.0, dtype=torch.float32, device=dev)
    ids = torch.full((M, k), -1, dtype=torch.int32, device=dev)
    st = torch.full((max(cap, 1),), -7, dtype=torch.int32, device=dev)
    eid = torch.full((max(cap // bm, 1),), -7, dtype=torch.int32, device=dev)
    ntpp = torch.full((1,), -7, dtype=torch.int32, device=dev)
    cnt = torch.full((E_local,), -7, dtype=torch.int32, device=dev)
    off = torch.full((E_local + 1,), -7, dtype=torch.int32, device=dev)
    pos = torch.full((max(M * k, 1),), -7, dtype=torch.int32, device=dev)
    wsb = chord.chord_moe_align_workspace_bytes(M, k, E_local)
    ws = torch.full((max(wsb, 16),), 0x5A, dtype=torch.uint8, device=dev) if wsb else None
    chord.chord_moe_route_align(lg, bs, k, begin, E_local, bm, w, ids, st[:cap] if cap else st, eid, ntpp,
                                cnt, off, pos, ws)
    torch.cuda.synchronize()
    n = int(ntpp.item())
    return w.cpu().numpy(), ids.cpu().numpy(), dict(
        sorted_token_ids=st.cpu().numpy()[:n], expert_ids=eid.cpu().numpy()[:n // bm],
        num_tokens_post_padded=n, expert_counts=cnt.cpu().numpy(), expert_offsets=off.cpu().numpy(),
        sorted_positions=pos.cpu().numpy()[:M * k])


def check_route_align(logits, bias, k, begin, E_local, bm):
    rw, rids, _ = oracle.route(logits, bias, k)
    ref = oracle.moe_align(rids, begin, E_local, bm)
    for _ in range(2):
        w, ids, got = gpu_route_align(logits, bias, k, begin, E_local, bm)
        assert np.array_equal(ids, rids)
        assert np.array_equal(w.view(np.uint32), rw.view(np.uint32))
        assert got["num_tokens_post_padded"] == ref["num_tokens_post_padded"]
        for key in ("expert_counts", "expert_offsets", "sorted_token_ids", "expert_ids", "sorted_positions"):
            assert np.array_equal(got[key], ref[key]), key


@pytest.mark.parametrize("M", wl.ROUTER_ALIGN_M)
@pytest.mark.parametrize("bm", wl.ROUTER_ALIGN_BM)
def test_route_align_fused_router_workload(M, bm):
    """At top-8, one launch up to 4 tokens (M = 1: four warps route the
    token); M = 8 and larger take the two-launch path."""
    logits, bias = wl.router_inputs(M, wl.ROUTER_ALIGN_E, wl.ROUTER_ALIGN_SEED)
    check_route_align(logits, bias, wl.ROUTER_ALIGN_TOPK, 0, wl.ROUTER_ALIGN_E, bm)


@pytest.mark.parametrize("M,E,k,begin,E_local,bm", [
    (16, 384, 8, 96, 48, 16),        # two launches at top-8 (one CTA per token), shard in the middle
    (17, 384, 8, 0, 48, 8),          # one token more: two launches
    (16, 1024, 32, 0, 1024, 128),    # widest router and shard in one launch
    (7, 1, 1, 0, 1, 128),
    (9, 1000, 17, 500, 500, 64),
    (0, 384, 8, 0, 48, 16),
    # up to 32 assignments: one CTA routes and aligns (four warps a token at top-k <= 8, up to 4 tokens)
    (32, 384, 1, 0, 384, 16),       # 32 tokens at top-1: two launches
    (1, 1024, 8, 0, 1024, 128),     # widest router, expert ids up to 1023 in the ballot ranking
    (4, 1024, 8, 512, 512, 8),      # shard in the middle of 1024 experts
    (3, 384, 1, 0, 384, 64),        # top-1, three tokens
    (4, 384, 8, 100, 48, 128),      # 32 assignments, shard in the middle, long padding
    (3, 64, 8, 0, 64, 8),
    (2, 1024, 16, 0, 1024, 16),     # widest router
    (1, 384, 8, 376, 8, 16),        # shard at the end
    (2, 384, 8, 300, 3, 32),        # few local experts, most assignments dropped
])
def test_route_align_fused_edges(M, E, k, begin, E_local, bm):
    logits, bias = wl.router_inputs(M, E, 41)
    check_route_align(logits, bias, k, begin, E_local, bm)
