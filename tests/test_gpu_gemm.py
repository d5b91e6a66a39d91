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

# GEMM alone: FP32 accumulation of exact products, one BF16 rounding of C.
GEMM_MAXABS = 8e-3
GEMM_FROB = 3e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _problem(M, K, N, E_total, E_local, begin, topk, seed, zipf=0.0):
    logits, bias = wl.router_inputs(M, E_total, seed, zipf)
    _, ids, _ = oracle.route(logits, bias, topk)
    al = oracle.moe_align(ids, begin, E_local, 16)
    x = wl.activations(M, K, seed)
    q = wl.int4_weights(E_local, N, K, seed, wl.S_Q13)
    s = wl.group_scales(E_local, N, K, seed, wl.S_S13)
    return ids, al, x, q, s


def _upload_align(al, M, topk, E_local):
    cap = max(oracle.align_capacity(M, topk, E_local, 16), 16)
    st = np.full(cap, M * topk, np.int32)
    st[:al["num_tokens_post_padded"]] = al["sorted_token_ids"]
    return (cap, torch.from_numpy(st).cuda(), torch.from_numpy(al["expert_counts"]).cuda(),
            torch.from_numpy(al["expert_offsets"]).cuda())


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


@pytest.mark.parametrize("M,K,N,E_total,E_local,begin,topk,epi,path_rows", [
    (40, 320, 384, 8, 8, 0, 2, chord.CHORD_EPI_STORE, None),        # 3 tiles, ragged K stage
    (40, 320, 384, 8, 8, 0, 2, chord.CHORD_EPI_SILU_MUL, None),
    (64, 7168, 256, 384, 48, 0, 8, chord.CHORD_EPI_SILU_MUL, None),  # Kimi K, decode rows
    (300, 256, 144, 6, 3, 2, 2, chord.CHORD_EPI_STORE, None),       # N padded to a tile, many passes
    (300, 512, 256, 6, 6, 0, 3, chord.CHORD_EPI_SILU_MUL, None),    # >32 rows per expert
    (2, 128, 128, 4, 4, 0, 1, chord.CHORD_EPI_STORE, None),
])
def test_gemm_gather(M, K, N, E_total, E_local, begin, topk, epi, path_rows):
    ids, al, x, q, s = _problem(M, K, N, E_total, E_local, begin, topk, 7)
    cap, st, cnt, off = _upload_align(al, M, topk, E_local)
    packed = prepack(to_device(q), to_device(s), epi == chord.CHORD_EPI_SILU_MUL)
    width = N // 2 if epi == chord.CHORD_EPI_SILU_MUL else N
    C = torch.full((cap, width), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    chord.chord_w4a16_moe_gemm(to_device(x), True, packed, E_local, N, K, M, topk, st, cnt, off, epi,
                               C, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    Cn = bf16_to_np(C)
    for e, (rows, ref) in _oracle_rows(x, q, s, al, topk, epi, True).items():
        assert_close_to_oracle(Cn[rows], ref, f"expert {e}", GEMM_MAXABS, GEMM_FROB)


def test_gemm_direct_rows_and_header_check():
    M, K, N, E, topk = 50, 256, 128, 4, 2
    ids, al, _, q, s = _problem(M, K, N, E, E, 0, topk, 9)
    cap, st, cnt, off = _upload_align(al, M, topk, E)
    A = wl.activations(cap, K, 10)          # one row per sorted row
    packed = prepack(to_device(q), to_device(s), False)
    C = torch.zeros((cap, N), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    chord.chord_w4a16_moe_gemm(to_device(A), False, packed, E, N, K, M, topk, st, cnt, off,
                               chord.CHORD_EPI_STORE, C, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    Cn = bf16_to_np(C)
    for e, (rows, ref) in _oracle_rows(A, q, s, al, topk, chord.CHORD_EPI_STORE, False).items():
        assert_close_to_oracle(Cn[rows], ref, f"expert {e}", GEMM_MAXABS, GEMM_FROB)
    # a blob packed for another K is refused on the device, without a fault
    other = prepack(to_device(wl.int4_weights(E, N, 2 * K, 1, 4)),
                    to_device(wl.group_scales(E, N, 2 * K, 1, 5)), False)
    chord.chord_w4a16_moe_gemm(to_device(A), False, other, E, N, K, M, topk, st, cnt, off,
                               chord.CHORD_EPI_STORE, C, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == chord.CHORD_ERR_PREPACK_MISMATCH
    # a plain blob used for SiLU*mul is refused too
    status.zero_()
    chord.chord_w4a16_moe_gemm(to_device(A), False, packed, E, N, K, M, topk, st, cnt, off,
                               chord.CHORD_EPI_SILU_MUL, C, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == chord.CHORD_ERR_PREPACK_MISMATCH


def test_moe_sum_against_oracle():
    M, k, H, E = 37, 4, 1024, 12
    logits, bias = wl.router_inputs(M, E, 12)
    w, ids, _ = oracle.route(logits, bias, k)
    al = oracle.moe_align(ids, 2, 7, 16)          # some assignments dropped
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
