"""GPU test of chord_moe_align_noalloc, the allocation-free align.

Some callers cannot allocate device memory at all (an engine or plugin that
owns every allocation and gives out no scratch, or a hot path where
cudaMalloc is forbidden).  For them the library offers an align entry point
whose scratch is a static device array inside the library.  This test calls
it through the C ABI twice in a row, on two different routings that both need
the scratch (more than 4096 assignments), and checks every output against the
regular chord_moe_align run with a caller-provided workspace: bit for bit,
the tolerance of all align tests.  It must pass alone in a fresh process and
after the other tests, so it keeps no state of its own.
"""
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


def _buffers(M, k, E_local, bm):
    cap = chord.chord_moe_align_capacity(M, k, E_local, bm)
    i32 = torch.int32
    return dict(
        sorted_token_ids=torch.full((cap,), -7, dtype=i32, device="cuda"),
        expert_ids=torch.full((cap // bm,), -7, dtype=i32, device="cuda"),
        num_tokens_post_padded=torch.full((1,), -7, dtype=i32, device="cuda"),
        expert_counts=torch.full((E_local,), -7, dtype=i32, device="cuda"),
        expert_offsets=torch.full((E_local + 1,), -7, dtype=i32, device="cuda"),
        sorted_positions=torch.full((M * k,), -7, dtype=i32, device="cuda"),
    )


def _host(b, bm):
    n = int(b["num_tokens_post_padded"].item())
    return dict(ntpp=n, sorted=b["sorted_token_ids"].cpu().numpy()[:n],
                eids=b["expert_ids"].cpu().numpy()[:n // bm],
                counts=b["expert_counts"].cpu().numpy(), offsets=b["expert_offsets"].cpu().numpy(),
                pos=b["sorted_positions"].cpu().numpy())


@pytest.mark.parametrize("calls", [
    [(4096, 8, 384, 0, 384, 16, 4), (1000, 8, 384, 96, 48, 64, 5)],
    [(8192, 8, 384, 0, 48, 16, 3), (6000, 6, 16, 0, 16, 128, 6)],
])
def test_noalloc_align_matches_workspace_align_twice(calls):
    for M, k, E, begin, E_local, bm, seed in calls:
        assert M * k > 4096, "the case must use the scratch"
        logits, bias = wl.router_inputs(M, E, seed)
        _, ids_np, _ = oracle.route(logits, bias, k)
        ids = torch.from_numpy(ids_np).cuda()
        ref = _buffers(M, k, E_local, bm)
        ws = torch.empty(chord.chord_moe_align_workspace_bytes(M, k, E_local), dtype=torch.uint8,
                         device="cuda")
        chord.chord_moe_align(ids, begin, E_local, bm, ref["sorted_token_ids"], ref["expert_ids"],
                              ref["num_tokens_post_padded"], ref["expert_counts"],
                              ref["expert_offsets"], ref["sorted_positions"], ws)
        got = _buffers(M, k, E_local, bm)
        chord.chord_moe_align_noalloc(ids, begin, E_local, bm, got["sorted_token_ids"],
                                      got["expert_ids"], got["num_tokens_post_padded"],
                                      got["expert_counts"], got["expert_offsets"],
                                      got["sorted_positions"])
        torch.cuda.synchronize()
        r, g = _host(ref, bm), _host(got, bm)
        assert g["ntpp"] == r["ntpp"] > 0
        for key in ("sorted", "eids", "counts", "offsets", "pos"):
            assert np.array_equal(g[key], r[key]), key


def test_noalloc_align_rejects_sizes_beyond_its_limit():
    M, k, E = 9000, 8, 384            # 72000 assignments > 65536
    ids = torch.zeros((M, k), dtype=torch.int32, device="cuda")
    b = _buffers(M, k, E, 16)
    with pytest.raises(chord.ChordError) as ei:
        chord.chord_moe_align_noalloc(ids, 0, E, 16, b["sorted_token_ids"], b["expert_ids"],
                                      b["num_tokens_post_padded"], b["expert_counts"],
                                      b["expert_offsets"], b["sorted_positions"])
    assert ei.value.code == chord.CHORD_ERR_INVALID_ARG
    assert "65536" in str(ei.value)
    torch.cuda.synchronize()
    assert int(b["num_tokens_post_padded"].item()) == -7, "nothing may be launched"
