"""GPU parity: prepack + indexed W4A16 GEMM (both epilogues, gather and
direct A) and the top-k weighted sum, against the FP64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from w4a16_int4_weight_sigmoid_gb300 import chord
from w4a16_int4_weight_sigmoid_gb300 import workload as wl
from w4a16_int4_weight_sigmoid_gb300.layer import prepack

from gpu_util import assert_close_to_oracle, bf16_to_np, ensure_lib, to_device

pytestmark = pytest.mark.gpu

# GEMM alone.  Register-MMA path: FP32 accumulation of exact products, one
# BF16 rounding of C.  Tensor-core path: the dequantised weight q*s is also
# rounded once to BF16 (up to 2^-9 relative for |q| in 3, 5, 6, 7), which
# roughly doubles the RMS error, so it is held to the layer's parity bar.
GEMM_TOL = {chord.CHORD_PATH_SMALL_M: (8e-3, 3e-3), chord.CHORD_PATH_LARGE_M: (1e-2, 5e-3)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _problem(M, K, N, E_total, E_local, begin, topk, seed, bm=16, zipf=0.0):
    logits, bias = wl.router_inputs(M, E_total, seed, zipf)
    _, ids, _ = oracle.route(logits, bias, topk)
    al = oracle.moe_align(ids, begin, E_local, bm)
    x = wl.activations(M, K, seed)
    q = wl.int4_weights(E_local, N, K, seed, wl.S_Q13)
    s = wl.group_scales(E_local, N, K, seed, wl.S_S13)
    return ids, al, x, q, s


def _upload_align(al, M, topk, E_local, bm):
    cap = max(oracle.align_capacity(M, topk, E_local, bm), bm)
    n = al["num_tokens_post_padded"]
    st = np.full(cap, M * topk, np.int32)
    st[:n] = al["sorted_token_ids"]
    eids = np.full(cap // bm, -1, np.int32)
    eids[:n // bm] = al["expert_ids"]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    return (cap, t(st), t(eids), t(np.array([n])), t(al["expert_counts"]),
            t(al["expert_offsets"]))


def _run_gemm(A, gather, packed, E_local, N, K, M, topk, up, bm, epi, C, path, status):
    cap, st, eids, ntpp, cnt, off = up
    ws = torch.zeros(chord.chord_w4a16_moe_gemm_workspace_bytes(cap, K, gather), dtype=torch.uint8,
                     device="cuda")
    tun = chord.chord_tuning(path, 0, 0, 0)
    chord.chord_w4a16_moe_gemm(A, gather, packed, E_local, N, K, M, topk, st, eids, ntpp, cnt, off, bm,
                               epi, C, ws, tuning=tun, dev_status=status)
    torch.cuda.synchronize()
    assert int(ws[:8].view(torch.int32).abs().sum().item()) == 0, "work counters must be left at zero"


def _oracle_rows(A_rows_bf16, q, s, al, topk, epi, gather):
    """Expected C rows (FP64) for every valid sorted row."""
    st, off, cnt = al["sorted_token_ids"], al["expert_offsets"], al["expert_counts"]
    out = {}
    for e in range(q.shape[0]):
        if cnt[e] == 0:
            continue
        rows = np.arange(off[e], off[e] + cnt[e])
        src = st[rows] // topk if gather else rows
        W = oracle.dequant_expert(q[e], s[e])
        acc = oracle.expert_rows_gemm(oracle.bf16_to_f64(A_rows_bf16[src]), W)
        out[e] = (rows, oracle.silu_mul(acc) if epi == chord.CHORD_EPI_SILU_MUL else acc)
    return out


SMALL, LARGE = chord.CHORD_PATH_SMALL_M, chord.CHORD_PATH_LARGE_M
STORE, SILU = chord.CHORD_EPI_STORE, chord.CHORD_EPI_SILU_MUL
CASES = [
    # M, K, N, E_total, E_local, begin, topk, epilogue, block_m, paths
    (40, 320, 384, 8, 8, 0, 2, STORE, 16, (SMALL, LARGE)),       # 3 tiles, ragged K stage
    (40, 320, 384, 8, 8, 0, 2, SILU, 8, (SMALL, LARGE)),
    (64, 7168, 256, 384, 48, 0, 8, SILU, 8, (SMALL, LARGE)),      # Kimi K, decode rows
    (300, 256, 144, 6, 3, 2, 2, STORE, 32, (SMALL,)),             # N padded to a tile, many blocks
    (300, 512, 256, 6, 6, 0, 3, SILU, 16, (SMALL, LARGE)),        # ~150 rows per expert
    (1200, 256, 256, 4, 4, 0, 2, STORE, 16, (SMALL, LARGE)),      # ~600 rows: 3 tcgen05 passes
    (2, 128, 128, 4, 4, 0, 1, STORE, 8, (SMALL, LARGE)),
    (96, 1024, 128, 32, 32, 0, 6, SILU, 8, (SMALL, LARGE)),       # Zipf skew: one heavy expert
    # short K, 8 rows per pass: items of two weight tiles (K = 256: the
    # straight-line stage) or four (K = 128), and a last item with fewer tiles
    (8, 256, 320, 16, 16, 0, 2, STORE, 8, (SMALL,)),
    (8, 128, 576, 16, 16, 0, 2, SILU, 8, (SMALL,)),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "m%d_k%d_n%d_e%d_bm%d_%s" % (
    c[0], c[1], c[2], c[4], c[8], "silu" if c[7] == SILU else "store"))
def test_gemm_gather(case):
    M, K, N, E_total, E_local, begin, topk, epi, bm, paths = case
    zipf = 1.1 if M == 96 else 0.0
    ids, al, x, q, s = _problem(M, K, N, E_total, E_local, begin, topk, 7, bm, zipf)
    up = _upload_align(al, M, topk, E_local, bm)
    packed = prepack(to_device(q), to_device(s), epi == SILU)
    width = N // 2 if epi == SILU else N
    expected = _oracle_rows(x, q, s, al, topk, epi, True)
    for path in paths:
        for _ in range(2):    # twice: the work queue must start from zero again
            C = torch.full((up[0], width), float("nan"), dtype=torch.bfloat16, device="cuda")
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            _run_gemm(to_device(x), True, packed, E_local, N, K, M, topk, up, bm, epi, C, path, status)
            assert status.item() == 0
            Cn = bf16_to_np(C)
            for e, (rows, ref) in expected.items():
                assert_close_to_oracle(Cn[rows], ref, f"path {path} expert {e}", *GEMM_TOL[path])


@pytest.mark.parametrize("path", [SMALL, LARGE])
def test_gemm_direct_rows_and_header_check(path):
    M, K, N, E, topk, bm = 50, 256, 128, 4, 2, 16
    ids, al, _, q, s = _problem(M, K, N, E, E, 0, topk, 9, bm)
    up = _upload_align(al, M, topk, E, bm)
    cap = up[0]
    A = wl.activations(cap, K, 10)          # one row per sorted row
    packed = prepack(to_device(q), to_device(s), False)
    C = torch.zeros((cap, N), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _run_gemm(to_device(A), False, packed, E, N, K, M, topk, up, bm, STORE, C, path, status)
    assert status.item() == 0
    Cn = bf16_to_np(C)
    for e, (rows, ref) in _oracle_rows(A, q, s, al, topk, STORE, False).items():
        assert_close_to_oracle(Cn[rows], ref, f"expert {e}", *GEMM_TOL[path])
    # a blob packed for another K is refused on the device, without a fault
    other = prepack(to_device(wl.int4_weights(E, N, 2 * K, 1, 4)),
                    to_device(wl.group_scales(E, N, 2 * K, 1, 5)), False)
    _run_gemm(to_device(A), False, other, E, N, K, M, topk, up, bm, STORE, C, path, status)
    assert status.item() == chord.CHORD_ERR_PREPACK_MISMATCH
    # a plain blob used for SiLU*mul is refused too
    status.zero_()
    C_half = torch.zeros((cap, N // 2), dtype=torch.bfloat16, device="cuda")
    _run_gemm(to_device(A), False, packed, E, N, K, M, topk, up, bm, SILU, C_half, path, status)
    assert status.item() == chord.CHORD_ERR_PREPACK_MISMATCH


# (M, topk, H, E_total, local experts): one CTA per (token, column block),
# and the streaming form taken from 4096 items on (1100 tokens x 4 column
# blocks, the last one ragged: H = 3976); with rows of 4096 < H <= 8192
# and at least 16 tokens per SM, persistent CTAs that carry the next token's
# slots ahead (3001 tokens, a ragged last pass over the grid, H = 7160)
@pytest.mark.parametrize("M,k,H,E,local", [(37, 4, 1024, 12, (2, 7)), (1100, 6, 3976, 40, (3, 25)),
                                           (3001, 8, 7160, 64, (8, 40))])
def test_moe_sum_against_oracle(M, k, H, E, local):
    logits, bias = wl.router_inputs(M, E, 12)
    w, ids, _ = oracle.route(logits, bias, k)
    al = oracle.moe_align(ids, local[0], local[1], 16)   # some assignments dropped
    cap = max(al["num_tokens_post_padded"], 1)
    y = wl.activations(cap, H, 13)
    out = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    chord.chord_moe_sum(to_device(y), torch.from_numpy(w).cuda(),
                        torch.from_numpy(al["sorted_positions"]).cuda(), out)
    torch.cuda.synchronize()
    ref = oracle.moe_sum(oracle.bf16_to_f64(y), w, al["sorted_positions"], M, k)
    got = bf16_to_np(out)
    # FP32 sum of at most k products, one BF16 rounding
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)
    assert np.all(got[np.all(al["sorted_positions"].reshape(M, k) < 0, axis=1)] == 0)


@pytest.mark.parametrize("M,K,N,epi,path", [
    (1, 256, 128, STORE, SMALL), (37, 512, 192, STORE, SMALL), (37, 512, 256, SILU, SMALL),
    (100, 1024, 256, SILU, LARGE), (300, 256, 384, STORE, LARGE), (300, 256, 384, STORE, 0),
    (5, 7168, 512, SILU, 0),
])
def test_dense_gemm(M, K, N, epi, path):
    """Dense entry (E = 1, no routing) against the oracle's expert GEMM, twice per workspace."""
    x = wl.activations(M, K, 51)
    q = wl.int4_weights(1, N, K, 52, wl.S_Q13)
    s = wl.group_scales(1, N, K, 53, wl.S_S13)
    packed = prepack(to_device(q), to_device(s), epi == SILU)
    acc = oracle.expert_rows_gemm(oracle.bf16_to_f64(x), oracle.dequant_expert(q[0], s[0]))
    ref = oracle.silu_mul(acc) if epi == SILU else acc
    ws = torch.zeros(chord.chord_w4a16_gemm_workspace_bytes(M), dtype=torch.uint8, device="cuda")
    tun = chord.chord_tuning(path, 0, 0, 0)
    for _ in range(2):
        C = torch.full((M, N // 2 if epi == SILU else N), float("nan"), dtype=torch.bfloat16, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        chord.chord_w4a16_gemm(to_device(x), packed, N, K, epi, C, ws, tuning=tun, dev_status=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        assert int(ws[:256].view(torch.int32).abs().sum().item()) == 0
        tol = GEMM_TOL[LARGE] if path == LARGE or (path == 0 and M >= 16 and N % 128 == 0) else GEMM_TOL[SMALL]
        assert_close_to_oracle(bf16_to_np(C), ref, "dense", *tol)


def test_gemm_split_k_counters_and_parity():
    """Three tokens, K = 2048 (four 512-wide stages), 8 experts: 8 or fewer
    work items against hundreds of resident CTAs, so the decode GEMM splits
    K.  The split partials are written (the area is no longer zero), the
    per-item counters are back at zero after the call, every row matches the
    oracle, and a second call gives the same bits."""
    M, K, N, E, topk, bm = 3, 2048, 256, 8, 2, 8
    ids, al, x, q, s = _problem(M, K, N, E, E, 0, topk, 41, bm)
    up = _upload_align(al, M, topk, E, bm)
    cap = up[0]
    packed = prepack(to_device(q), to_device(s), False)
    ws = torch.zeros(chord.chord_w4a16_moe_gemm_workspace_bytes(cap, K, True), dtype=torch.uint8, device="cuda")
    tun = chord.chord_tuning(SMALL, 0, 0, 0)
    outs = []
    for _ in range(2):
        C = torch.full((cap, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        chord.chord_w4a16_moe_gemm(to_device(x), True, packed, E, N, K, M, topk, *up[1:], bm, STORE, C, ws,
                                   tuning=tun, dev_status=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        counters = ws[256:256 + 512 * 4 * 4].view(torch.int32)
        assert int(counters.abs().sum().item()) == 0, "split-K counters must be left at zero"
        assert int(ws[:256].view(torch.int32).abs().sum().item()) == 0
        partials = ws[256 + 512 * 16:256 + 512 * 16 + 512 * 2048 * 4]
        assert int((partials != 0).sum().item()) > 0, "no split-K partials were written"
        outs.append(bf16_to_np(C))
        for e, (rows, ref) in _oracle_rows(x, q, s, al, topk, STORE, True).items():
            assert_close_to_oracle(outs[-1][rows], ref, f"split-K expert {e}", *GEMM_TOL[SMALL])
    n = al["num_tokens_post_padded"]
    assert np.array_equal(outs[0][:n].view(np.uint16), outs[1][:n].view(np.uint16))


@pytest.mark.parametrize("E,K,extra", [(16, 4096, 0.6), (4, 7168, 0.55)])
def test_gemm_tail_wave_split_k(E, K, extra):
    """More work items than resident CTAs, with a last wave of about `extra`
    of the CTAs (more than half): the decode GEMM takes the other items whole
    and splits those of the last wave along K (into three ranges over eight
    stages at 0.6 of a wave, five over fourteen at 0.55).  Every row matches
    the oracle, split partials were written, the counters are back at zero,
    and a second call gives the same bits."""
    M, topk, bm = 64, 2, 8
    logits, bias = wl.router_inputs(M, E, 43)
    _, ids, _ = oracle.route(logits, bias, topk)
    nblocks = oracle.moe_align(ids, 0, E, bm)["num_tokens_post_padded"] // bm
    ctas = 4 * torch.cuda.get_device_properties(0).multi_processor_count   # resident at 8 rows per pass
    N = 64 * -(-int(ctas * (1 + extra)) // nblocks)
    ids, al, x, q, s = _problem(M, K, N, E, E, 0, topk, 43, bm)
    assert al["num_tokens_post_padded"] // bm == nblocks
    up = _upload_align(al, M, topk, E, bm)
    cap = up[0]
    packed = prepack(to_device(q), to_device(s), False)
    ws = torch.zeros(chord.chord_w4a16_moe_gemm_workspace_bytes(cap, K, True), dtype=torch.uint8, device="cuda")
    tun = chord.chord_tuning(SMALL, 8, 0, 0)
    refs = _oracle_rows(x, q, s, al, topk, STORE, True)
    outs = []
    for _ in range(2):
        C = torch.full((cap, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        chord.chord_w4a16_moe_gemm(to_device(x), True, packed, E, N, K, M, topk, *up[1:], bm, STORE, C, ws,
                                   tuning=tun, dev_status=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        assert int(ws[256:256 + 512 * 4 * 4].view(torch.int32).abs().sum().item()) == 0, \
            "split-K counters must be left at zero"
        assert int(ws[:256].view(torch.int32).abs().sum().item()) == 0
        partials = ws[256 + 512 * 16:256 + 512 * 16 + 512 * 2048 * 4]
        assert int((partials != 0).sum().item()) > 0, "the last wave was not split"
        outs.append(bf16_to_np(C))
        for e, (rows, ref) in refs.items():
            assert_close_to_oracle(outs[-1][rows], ref, f"tail split expert {e}", *GEMM_TOL[SMALL])
    n = al["num_tokens_post_padded"]
    assert np.array_equal(outs[0][:n].view(np.uint16), outs[1][:n].view(np.uint16))


@pytest.mark.parametrize("path", [SMALL, LARGE])
@pytest.mark.parametrize("M,K,N,E,topk,bm", [(40, 256, 384, 6, 3, 16), (300, 512, 256, 4, 2, 16)])
def test_weighted_add_epilogue(path, M, K, N, E, topk, bm):
    """CHORD_EPI_WEIGHTED_ADD: the down GEMM over rows in sorted order adds
    topk_weights[f] * row into token f / topk of an FP32 [M, N] accumulator.
    Expected: for every token, the sum over its local assignments of w times
    the oracle's expert GEMM row (FP64).  The accumulator starts from a
    known non-zero value, which the epilogue must add to, not overwrite."""
    logits, bias = wl.router_inputs(M, E, 61)
    w, ids, _ = oracle.route(logits, bias, topk)
    al = oracle.moe_align(ids, 0, E, bm)
    up = _upload_align(al, M, topk, E, bm)
    cap = up[0]
    A = wl.activations(cap, K, 62)           # one row per sorted row (the gate/up output)
    q = wl.int4_weights(E, N, K, 63, wl.S_Q2)
    s = wl.group_scales(E, N, K, 64, wl.S_S2)
    packed = prepack(to_device(q), to_device(s), False)
    rows = _oracle_rows(A, q, s, al, topk, STORE, False)
    ref = np.full((M, N), 0.25)
    st = al["sorted_token_ids"]
    for e, (r, vals) in rows.items():
        for k, row in enumerate(r):
            f = int(st[row])
            ref[f // topk] += float(w.ravel()[f]) * vals[k]
    ws = torch.zeros(chord.chord_w4a16_moe_gemm_workspace_bytes(cap, K, False), dtype=torch.uint8, device="cuda")
    tw = torch.from_numpy(np.ascontiguousarray(w, np.float32)).cuda()
    C = torch.full((M, N), 0.25, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    chord.chord_w4a16_moe_gemm(to_device(A), False, packed, E, N, K, M, topk, *up[1:], bm,
                               chord.CHORD_EPI_WEIGHTED_ADD, C, ws, tuning=chord.chord_tuning(path, 0, 0, 0),
                               dev_status=status, topk_weights=tw)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert int(ws[:256].view(torch.int32).abs().sum().item()) == 0
    assert_close_to_oracle(C.cpu().numpy().astype(np.float64), ref, f"weighted add path {path}", *GEMM_TOL[path])
