"""GPU tests of the device-side failure paths, made to fail on the host side
or through the library's test hook, never by a GPU fault.

* A bounded barrier wait that runs out: chord_debug_force_timeout makes the
  register-MMA GEMM's producer withhold every work item (no copy is issued),
  so the consumers' waits for an item run out; the kernel must record
  CHORD_ERR_TIMEOUT and return, and leave the work-queue counters at zero,
  so the next call on the same workspace is exact.
* An expert id out of range in the align buffers (corrupted on the host):
  the GEMM records CHORD_ERR_ROUTING_INVALID, skips that block, and computes
  every other block correctly ([Chord] "런타임 고려사항": unsupported input is
  reported, not silently used).
"""
import numpy as np
import pytest
import torch

from w4a16_int4_weight_sigmoid_gb300 import chord
from w4a16_int4_weight_sigmoid_gb300.layer import prepack

from gpu_util import assert_close_to_oracle, bf16_to_np, ensure_lib, to_device
from test_gpu_gemm import GEMM_TOL, _oracle_rows, _problem, _upload_align

pytestmark = pytest.mark.gpu

SMALL, STORE = chord.CHORD_PATH_SMALL_M, chord.CHORD_EPI_STORE


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _run(x, packed, E, N, K, M, topk, up, bm, C, ws, status):
    chord.chord_w4a16_moe_gemm(to_device(x), True, packed, E, N, K, M, topk, *up[1:], bm, STORE, C, ws,
                               tuning=chord.chord_tuning(SMALL, 8, 0, 0), dev_status=status)
    torch.cuda.synchronize()


def test_wait_timeout_is_reported_and_the_next_call_is_exact():
    # enough work items (32 tiles x ~50 blocks) that the GEMM does not split every item along K
    M, K, N, E, topk, bm = 200, 1024, 2048, 8, 2, 8
    ids, al, x, q, s = _problem(M, K, N, E, E, 0, topk, 71, bm)
    up = _upload_align(al, M, topk, E, bm)
    cap = up[0]
    packed = prepack(to_device(q), to_device(s), False)
    ws = torch.zeros(chord.chord_w4a16_moe_gemm_workspace_bytes(cap, K, True), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    C = torch.zeros((cap, N), dtype=torch.bfloat16, device="cuda")
    try:
        chord.chord_debug_force_timeout(True)
        _run(x, packed, E, N, K, M, topk, up, bm, C, ws, status)
    finally:
        chord.chord_debug_force_timeout(False)
    assert status.item() == chord.CHORD_ERR_TIMEOUT
    assert int(ws[:8].view(torch.int32).abs().sum().item()) == 0, "work-queue counters not reset after a timeout"
    status.zero_()
    C = torch.full((cap, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    _run(x, packed, E, N, K, M, topk, up, bm, C, ws, status)
    assert status.item() == 0
    got = bf16_to_np(C)
    for e, (rows, ref) in _oracle_rows(x, q, s, al, topk, STORE, True).items():
        assert_close_to_oracle(got[rows], ref, f"after timeout, expert {e}", *GEMM_TOL[SMALL])


def test_expert_id_out_of_range_is_reported_and_skipped():
    M, K, N, E, topk, bm = 40, 512, 256, 6, 2, 16
    ids, al, x, q, s = _problem(M, K, N, E, E, 0, topk, 72, bm)
    up = list(_upload_align(al, M, topk, E, bm))
    cap = up[0]
    eids = up[2]
    bad_block = 1
    bad_expert = int(eids[bad_block].item())
    eids[bad_block] = 99                      # not a local expert
    packed = prepack(to_device(q), to_device(s), False)
    ws = torch.zeros(chord.chord_w4a16_moe_gemm_workspace_bytes(cap, K, True), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    C = torch.full((cap, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    _run(x, packed, E, N, K, M, topk, up, bm, C, ws, status)
    assert status.item() == chord.CHORD_ERR_ROUTING_INVALID
    got = bf16_to_np(C)
    bad_rows = np.arange(bad_block * bm, (bad_block + 1) * bm)
    assert np.all(np.isnan(got[bad_rows])), "the block with the bad expert id must not be written"
    for e, (rows, ref) in _oracle_rows(x, q, s, al, topk, STORE, True).items():
        keep = ~np.isin(rows, bad_rows)
        if keep.any():
            assert_close_to_oracle(got[rows[keep]], ref[keep], f"expert {e}", *GEMM_TOL[SMALL])
    assert bad_expert >= 0
