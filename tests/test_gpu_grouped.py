"""GPU parity: the grouped-layout W4A16 GEMMs (contiguous and masked) against
the FP64 oracle, on both kernel paths and both epilogues, with ragged and
empty expert groups; rows outside the groups must stay untouched."""
import numpy as np
import pytest
import torch

import oracle
from w4a16_int4_weight_sigmoid_gb300 import chord
from w4a16_int4_weight_sigmoid_gb300 import workload as wl
from w4a16_int4_weight_sigmoid_gb300.layer import prepack

from gpu_util import assert_close_to_oracle, bf16_to_np, ensure_lib, to_device

pytestmark = pytest.mark.gpu

SMALL, LARGE = chord.CHORD_PATH_SMALL_M, chord.CHORD_PATH_LARGE_M
STORE, SILU = chord.CHORD_EPI_STORE, chord.CHORD_EPI_SILU_MUL
# the same bars as the indexed GEMM (test_gpu_gemm.py): FP32 accumulation of
# exact products on the register path; q*s rounded once to BF16 on tcgen05
GEMM_TOL = {SMALL: (8e-3, 3e-3), LARGE: (1e-2, 5e-3)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _weights(E, N, K, seed, silu):
    q = wl.int4_weights(E, N, K, seed, wl.S_Q13)
    s = wl.group_scales(E, N, K, seed + 1, wl.S_S13)
    return q, s, prepack(to_device(q), to_device(s), silu)


def _run(layout, A, counts, packed, N, K, epi, path, max_m=0, expected_m=0):
    E = len(counts)
    rows = A.shape[0]
    g = torch.tensor(counts, dtype=torch.int32, device="cuda")
    ws = torch.zeros(chord.chord_w4a16_grouped_workspace_bytes(E, rows), dtype=torch.uint8, device="cuda")
    C = torch.full((rows, N // 2 if epi == SILU else N), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tun = chord.chord_tuning(path, 0, 0, 0) if path else None
    if layout == "contiguous":
        chord.chord_w4a16_grouped_gemm_contiguous(to_device(A), g, packed, N, K, epi, C, ws, expected_m,
                                                  tuning=tun, dev_status=status)
    else:
        chord.chord_w4a16_grouped_gemm_masked(to_device(A).view(E, max_m, K), g, packed, N, K, epi,
                                              C.view(E, max_m, -1), ws, expected_m, tuning=tun,
                                              dev_status=status)
    torch.cuda.synchronize()
    assert int(ws[:256].view(torch.int32).abs().sum().item()) == 0   # work counters left zero
    return bf16_to_np(C), status.item()


CASES = [
    # layout, counts, max_m
    ("contiguous", [3, 0, 130, 17, 1], 0),
    ("masked", [48, 0, 5, 33], 48),
]


@pytest.mark.parametrize("layout,counts,max_m", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("epi", [STORE, SILU], ids=["store", "silu"])
@pytest.mark.parametrize("path", [SMALL, LARGE], ids=["register", "tcgen05"])
def test_grouped_gemm_parity(layout, counts, max_m, epi, path):
    N, K, E = 256, 512, len(counts)
    starts = oracle.group_starts(counts, layout, max_m)
    rows = E * max_m if layout == "masked" else int(starts[-1] + (-(-counts[-1] // 128)) * 128) + 128
    A = wl.activations(rows, K, 71)
    q, s, packed = _weights(E, N, K, 72, epi == SILU)
    idx, ref = oracle.grouped_gemm(oracle.bf16_to_f64(A), counts, q, s, layout, max_m, epi == SILU)
    for _ in range(2):   # the workspace is reused: its counters must come back zeroed
        got, status = _run(layout, A, counts, packed, N, K, epi, path, max_m)
        assert status == 0
        assert_close_to_oracle(got[idx], ref, f"grouped {layout}", *GEMM_TOL[path])
        other = np.ones(rows, bool)
        other[idx] = False
        assert np.all(np.isnan(got[other])), "rows outside the groups were written"


@pytest.mark.parametrize("layout,counts,max_m", CASES, ids=[c[0] for c in CASES])
def test_grouped_gemm_auto_path_from_expected_m(layout, counts, max_m):
    """No tuning: expected_m picks the path; both choices give the oracle's result."""
    N, K, E = 256, 512, len(counts)
    starts = oracle.group_starts(counts, layout, max_m)
    rows = E * max_m if layout == "masked" else int(starts[-1] + (-(-counts[-1] // 128)) * 128)
    A = wl.activations(rows, K, 73)
    q, s, packed = _weights(E, N, K, 74, False)
    idx, ref = oracle.grouped_gemm(oracle.bf16_to_f64(A), counts, q, s, layout, max_m)
    for expected_m in (2, 200):
        got, status = _run(layout, A, counts, packed, N, K, STORE, 0, max_m, expected_m)
        assert status == 0
        assert_close_to_oracle(got[idx], ref, f"grouped {layout} auto", *GEMM_TOL[LARGE])


def test_grouped_gemm_bad_counts_are_recorded():
    """A masked count above max_m, or contiguous groups that overflow A, set
    CHORD_ERR_INVALID_ARG in the device status and compute nothing."""
    N, K = 256, 256
    q, s, packed = _weights(2, N, K, 75, False)
    A = wl.activations(2 * 32, K, 76)
    got, status = _run("masked", A, [5, 33], packed, N, K, STORE, SMALL, 32)
    assert status == chord.CHORD_ERR_INVALID_ARG and np.all(np.isnan(got))
    A = wl.activations(200, K, 77)     # two groups padded to 128 need 256 rows
    got, status = _run("contiguous", A, [100, 20], packed, N, K, STORE, SMALL)
    assert status == chord.CHORD_ERR_INVALID_ARG and np.all(np.isnan(got))
