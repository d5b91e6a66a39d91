"""C-ABI checks that need no GPU: the library builds, loads and exports every
entry point include/chord_moe.h declares; host-side sizing functions; argument
checks that reject bad calls before any launch; the header is plain C."""
import ctypes
import os
import re
import subprocess

import pytest

from w4a16_int4_weight_sigmoid_gb300 import build as B
from w4a16_int4_weight_sigmoid_gb300 import chord

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "chord_moe.h")


@pytest.fixture(scope="module")
def L():
    B.build()
    return chord.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(chord_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (chord_\w+)", out))
    assert set(names) <= exported


def test_binding_covers_every_entry_point():
    assert set(_declared()) == set(chord._SIGS)


def test_header_is_plain_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "chord_moe.h"\nint main(void){return CHORD_OK;}\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), "-c",
                        str(src), "-o", str(tmp_path / "t.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_sizing_functions(L):
    assert L.chord_moe_align_capacity(3, 2, 4, 8) == 40             # 6 + 4*7 = 34 -> 40
    assert L.chord_moe_align_capacity(4, 2, 8, 16) == 8 * 16
    assert L.chord_moe_align_capacity(64, 8, 48, 16) == 512 + 48 * 15
    assert L.chord_moe_align_capacity(1, 8, 384, 7) == 0           # bad block_m
    assert L.chord_moe_align_workspace_bytes(128, 8, 384) == 0      # one chunk: none
    assert L.chord_moe_align_workspace_bytes(4096, 8, 384) == (32768 + 32 * 384) * 4   # chunks of 1024
    assert L.chord_w4a16_prepack_bytes(48, 4096, 7168, 32) == 256 + 48 * 64 * 112 * 2304
    assert L.chord_w4a16_prepack_bytes(1, 16, 64, 32) == 256 + 2304
    assert L.chord_w4a16_prepack_bytes(1, 16, 96, 32) == 0          # K % 64
    assert L.chord_w4a16_prepack_bytes(1, 16, 64, 64) == 0          # group 64
    assert L.chord_moe_layer_workspace_bytes(64, 7168, 2048, 48, 8) > 0
    assert L.chord_version() >= 100
    plan = chord.chord_moe_layer_plan(64, 384, 8)
    assert plan.path == chord.CHORD_PATH_SMALL_M and plan.rows_per_pass == 8
    assert chord.chord_moe_layer_plan(8192, 384, 8).path == chord.CHORD_PATH_LARGE_M
    assert chord.chord_moe_layer_plan(128, 4, 2).rows_per_pass == 32
    # 256 B of work-queue counters, the split-K area (512 items x 4 warps of
    # counters, 512 slots of 8 KB partials), then the gathered rows
    split = 512 * 4 * 4 + 512 * 2048 * 4
    assert L.chord_w4a16_moe_gemm_workspace_bytes(1000, 512, 0) == 256 + split
    assert L.chord_w4a16_moe_gemm_workspace_bytes(1000, 512, 1) == 256 + split + 1000 * 512 * 2


def _rc_and_msg(L, rc):
    return rc, L.chord_last_error_string().decode()


def test_argument_checks_reject_before_launch(L):
    P = ctypes.c_void_p(16)   # never dereferenced: the checks fail first
    rc, msg = _rc_and_msg(L, L.chord_moe_route(P, P, 4, 384, 0, P, P, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG and "topk" in msg
    rc, _ = _rc_and_msg(L, L.chord_moe_route(P, P, 4, 384, 33, P, P, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG
    rc, _ = _rc_and_msg(L, L.chord_moe_route(P, P, 4, 2000, 8, P, P, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG
    rc, msg = _rc_and_msg(L, L.chord_moe_align(P, 4, 2, 0, 8, 12, 1000, P, P, P, P, P, None, None, 0, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG and "block_m" in msg
    rc, msg = _rc_and_msg(L, L.chord_moe_align(P, 4, 2, 0, 8, 16, 10, P, P, P, P, P, None, None, 0, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG and "capacity" in msg
    rc, _ = _rc_and_msg(L, L.chord_moe_align(P, 4096, 8, 0, 384, 16, 10 ** 6, P, P, P, P, P, None, None, 0, None))
    assert rc == chord.CHORD_ERR_WORKSPACE_TOO_SMALL
    rc, _ = _rc_and_msg(L, L.chord_w4a16_prepack(P, P, 2, 128, 96, 32, 0, P, 10 ** 9, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG
    rc, _ = _rc_and_msg(L, L.chord_w4a16_prepack(P, P, 2, 128, 128, 128, 0, P, 10 ** 9, None))
    assert rc == chord.CHORD_ERR_UNSUPPORTED
    rc, _ = _rc_and_msg(L, L.chord_w4a16_prepack(P, P, 2, 96, 128, 32, 1, P, 10 ** 9, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG                        # gate_up needs N % 64
    t = chord.chord_tuning(0, 0, 1, 0)
    rc, msg = _rc_and_msg(L, L.chord_w4a16_moe_gemm(P, 1, P, 4, 256, 128, 8, 2, P, P, P, P, P, 16, 100, 0, None,
                                                    P, ctypes.byref(t), P, 1 << 24, None, None))
    assert rc == chord.CHORD_ERR_UNSUPPORTED and "FP16" in msg
    t = chord.chord_tuning(0, 0, 0, 1)
    rc, _ = _rc_and_msg(L, L.chord_w4a16_moe_gemm(P, 1, P, 4, 256, 128, 8, 2, P, P, P, P, P, 16, 100, 0, None,
                                                  P, ctypes.byref(t), P, 1 << 24, None, None))
    assert rc == chord.CHORD_ERR_UNSUPPORTED
    rc, _ = _rc_and_msg(L, L.chord_w4a16_moe_gemm(P, 1, P, 4, 256, 100, 8, 2, P, P, P, P, P, 16, 100, 0, None,
                                                  P, None, P, 1 << 24, None, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG                        # K % 64
    rc, _ = _rc_and_msg(L, L.chord_w4a16_moe_gemm(P, 1, P, 4, 96, 128, 8, 2, P, P, P, P, P, 16, 100, 1, None,
                                                  P, None, P, 1 << 24, None, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG                        # SiLU needs N % 64
    rc, _ = _rc_and_msg(L, L.chord_w4a16_moe_gemm(P, 1, P, 4, 256, 128, 8, 2, P, P, P, P, P, 12, 100, 0, None,
                                                  P, None, P, 1 << 24, None, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG                        # block_m
    rc, _ = _rc_and_msg(L, L.chord_w4a16_moe_gemm(P, 1, P, 4, 256, 128, 8, 2, P, P, P, P, P, 16, 100, 0, None,
                                                  P, None, P, 100, None, None))
    assert rc == chord.CHORD_ERR_WORKSPACE_TOO_SMALL                # < counters + split-K area
    t = chord.chord_tuning(chord.CHORD_PATH_LARGE_M, 0, 0, 0)
    rc, _ = _rc_and_msg(L, L.chord_w4a16_moe_gemm(P, 1, P, 4, 192, 128, 8, 2, P, P, P, P, P, 16, 100, 0, None,
                                                  P, ctypes.byref(t), P, 1 << 24, None, None))
    assert rc == chord.CHORD_ERR_UNSUPPORTED                        # tcgen05 path needs N % 128
    rc, _ = _rc_and_msg(L, L.chord_moe_sum(P, P, P, 4, 2, 100, P, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG                        # H % 8
    rc, _ = _rc_and_msg(L, L.chord_moe_layer(P, P, P, P, P, 4, 256, 128, 8, 4, 8, 2, P, None, None,
                                             P, 10 ** 9, None, None, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG                        # shard exceeds E_total
    rc, _ = _rc_and_msg(L, L.chord_moe_layer(P, P, P, P, P, 4, 256, 128, 8, 0, 8, 2, P, None, None,
                                             P, 10, None, None, None))
    assert rc == chord.CHORD_ERR_WORKSPACE_TOO_SMALL


def test_new_entry_points_reject_before_launch(L):
    """chord_moe_route_align and chord_w4a16_gemm check their arguments on the host."""
    P = ctypes.c_void_p(16)   # never dereferenced: the checks fail first
    # route+align: topk > E_total, local experts outside E_total, bad block_m, small capacity
    rc, msg = _rc_and_msg(L, L.chord_moe_route_align(P, P, 4, 8, 9, 0, 8, 16, 1000, P, P, P, P, P, P, P,
                                                     None, None, 0, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG and "topk" in msg
    rc, msg = _rc_and_msg(L, L.chord_moe_route_align(P, P, 4, 384, 8, 380, 8, 16, 1000, P, P, P, P, P, P, P,
                                                     None, None, 0, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG and "within" in msg
    rc, msg = _rc_and_msg(L, L.chord_moe_route_align(P, P, 4, 384, 8, 0, 48, 24, 1000, P, P, P, P, P, P, P,
                                                     None, None, 0, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG and "block_m" in msg
    rc, msg = _rc_and_msg(L, L.chord_moe_route_align(P, P, 4, 384, 8, 0, 48, 16, 10, P, P, P, P, P, P, P,
                                                     None, None, 0, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG and "capacity" in msg
    # dense GEMM: K % 64, SiLU needs N % 64, workspace too small, tcgen05 path needs N % 128
    rc, _ = _rc_and_msg(L, L.chord_w4a16_gemm(P, P, 256, 100, 8, 0, P, None, P, 1 << 24, None, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG
    rc, _ = _rc_and_msg(L, L.chord_w4a16_gemm(P, P, 96, 128, 8, 1, P, None, P, 1 << 24, None, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG
    need = L.chord_w4a16_gemm_workspace_bytes(1000)
    assert need >= 512 + (1000 // 8) * 4
    rc, _ = _rc_and_msg(L, L.chord_w4a16_gemm(P, P, 256, 128, 1000, 0, P, None, P, need - 1, None, None))
    assert rc == chord.CHORD_ERR_WORKSPACE_TOO_SMALL
    t = chord.chord_tuning(chord.CHORD_PATH_LARGE_M, 0, 0, 0)
    rc, _ = _rc_and_msg(L, L.chord_w4a16_gemm(P, P, 192, 128, 1000, 0, P, ctypes.byref(t), P, need, None, None))
    assert rc == chord.CHORD_ERR_UNSUPPORTED


def test_weighted_add_epilogue_checks(L):
    """CHORD_EPI_WEIGHTED_ADD reads rows in sorted order and needs the routing
    weights; the dense and grouped GEMMs, which have no routing, refuse it."""
    P = ctypes.c_void_p(16)
    WADD = chord.CHORD_EPI_WEIGHTED_ADD
    big = 1 << 24
    rc, _ = _rc_and_msg(L, L.chord_w4a16_moe_gemm(P, 1, P, 4, 256, 128, 8, 2, P, P, P, P, P, 16, 100, WADD, P,
                                                  P, None, P, big, None, None))
    assert rc == chord.CHORD_ERR_UNSUPPORTED                        # gathered rows
    rc, msg = _rc_and_msg(L, L.chord_w4a16_moe_gemm(P, 0, P, 4, 256, 128, 8, 2, P, P, P, P, P, 16, 100, WADD, None,
                                                    P, None, P, big, None, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG and "topk_weights" in msg
    rc, msg = _rc_and_msg(L, L.chord_w4a16_gemm(P, P, 256, 128, 8, WADD, P, None, P, big, None, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG and "routing" in msg
    need = L.chord_w4a16_grouped_workspace_bytes(8, 1024)
    rc, msg = _rc_and_msg(L, L.chord_w4a16_grouped_gemm_contiguous(P, 1024, P, 8, 0, P, 256, 128, WADD, P, None,
                                                                   P, need, None, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG and "routing" in msg
    rc, _ = _rc_and_msg(L, L.chord_w4a16_moe_gemm(P, 0, P, 4, 256, 128, 8, 2, P, P, P, P, P, 16, 100, 3, P,
                                                  P, None, P, big, None, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG                        # unknown epilogue


def test_grouped_entry_points_reject_before_launch(L):
    """The grouped-layout GEMMs check their arguments on the host; every case
    below fails a check, so nothing is launched with these placeholder pointers."""
    P = ctypes.c_void_p(16)
    assert L.chord_w4a16_grouped_workspace_bytes(0, 100) == 0
    need = L.chord_w4a16_grouped_workspace_bytes(8, 1024)
    assert need >= 256 + (2 * 8 + 2) * 4 + (1024 // 8) * 4
    # contiguous: E out of range, K % 64, SiLU with N % 64, small workspace, tcgen05 with N % 128
    rc, msg = _rc_and_msg(L, L.chord_w4a16_grouped_gemm_contiguous(P, 1024, P, 0, 0, P, 256, 128, 0, P, None,
                                                                   P, need, None, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG and "E=" in msg
    rc, _ = _rc_and_msg(L, L.chord_w4a16_grouped_gemm_contiguous(P, 1024, P, 8, 0, P, 256, 100, 0, P, None,
                                                                 P, need, None, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG
    rc, _ = _rc_and_msg(L, L.chord_w4a16_grouped_gemm_contiguous(P, 1024, P, 8, 0, P, 96, 128, 1, P, None,
                                                                 P, need, None, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG
    rc, _ = _rc_and_msg(L, L.chord_w4a16_grouped_gemm_contiguous(P, 1024, P, 8, 0, P, 256, 128, 0, P, None,
                                                                 P, need - 1, None, None))
    assert rc == chord.CHORD_ERR_WORKSPACE_TOO_SMALL
    t = chord.chord_tuning(chord.CHORD_PATH_LARGE_M, 0, 0, 0)
    rc, _ = _rc_and_msg(L, L.chord_w4a16_grouped_gemm_contiguous(P, 1024, P, 8, 0, P, 192, 128, 0, P,
                                                                 ctypes.byref(t), P, need, None, None))
    assert rc == chord.CHORD_ERR_UNSUPPORTED
    # masked: max_m % 16, E out of range, small workspace (rows = E * max_m)
    rc, msg = _rc_and_msg(L, L.chord_w4a16_grouped_gemm_masked(P, P, 8, 24, 0, P, 256, 128, 0, P, None, P,
                                                               need, None, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG and "max_m" in msg
    rc, _ = _rc_and_msg(L, L.chord_w4a16_grouped_gemm_masked(P, P, 2000, 32, 0, P, 256, 128, 0, P, None, P,
                                                             need, None, None))
    assert rc == chord.CHORD_ERR_INVALID_ARG
    rc, _ = _rc_and_msg(L, L.chord_w4a16_grouped_gemm_masked(P, P, 8, 256, 0, P, 256, 128, 0, P, None, P,
                                                             need, None, None))
    assert rc == chord.CHORD_ERR_WORKSPACE_TOO_SMALL


def test_grouped_wrappers_check_shapes_before_the_library():
    """A masked call whose group counts do not match A's experts, or a
    contiguous call with a 3-D A, is refused by the binding itself."""
    import torch
    A3 = torch.zeros((2, 16, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="one group_rows entry per expert"):
        chord.chord_w4a16_grouped_gemm_masked(A3, torch.zeros(3, dtype=torch.int32), None, 64, 64, 0, None, None)
    with pytest.raises(ValueError, match="rows, K"):
        chord.chord_w4a16_grouped_gemm_contiguous(A3, torch.zeros(2, dtype=torch.int32), None, 64, 64, 0, None, None)


def test_gemm_wrappers_check_operands_before_the_library():
    """The C ABI sees raw pointers only, so the binding checks what it cannot:
    BF16 operands, A's last dimension = K, and C large enough for N (STORE) or
    N/2 (SiLU*mul) columns on every row.  Each mismatch raises ValueError
    before any pointer is taken (these tensors are on the CPU)."""
    import torch
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    STORE, SILU = chord.CHORD_EPI_STORE, chord.CHORD_EPI_SILU_MUL
    A = torch.zeros((8, 64), dtype=bf)
    # dense
    with pytest.raises(ValueError, match="bfloat16"):
        chord.chord_w4a16_gemm(A.float(), None, 64, 64, STORE, torch.zeros((8, 64), dtype=bf), None)
    with pytest.raises(ValueError, match="bfloat16"):
        chord.chord_w4a16_gemm(A, None, 64, 64, STORE, torch.zeros((8, 64), dtype=f32), None)
    with pytest.raises(ValueError, match="last dimension"):
        chord.chord_w4a16_gemm(A, None, 64, 128, STORE, torch.zeros((8, 64), dtype=bf), None)
    with pytest.raises(ValueError, match="C's last dimension"):
        chord.chord_w4a16_gemm(A, None, 64, 64, SILU, torch.zeros((8, 64), dtype=bf), None)
    with pytest.raises(ValueError, match="same rows"):
        chord.chord_w4a16_gemm(A, None, 64, 64, STORE, torch.zeros((4, 64), dtype=bf), None)
    # contiguous
    g2 = torch.zeros(2, dtype=i32)
    with pytest.raises(ValueError, match="rows of A"):
        chord.chord_w4a16_grouped_gemm_contiguous(A, g2, None, 64, 64, STORE, torch.zeros((7, 64), dtype=bf), None)
    with pytest.raises(ValueError, match="last dimension"):
        chord.chord_w4a16_grouped_gemm_contiguous(A, g2, None, 64, 128, STORE, torch.zeros((8, 64), dtype=bf), None)
    with pytest.raises(ValueError, match="C's last dimension"):
        chord.chord_w4a16_grouped_gemm_contiguous(A, g2, None, 128, 64, STORE, torch.zeros((8, 64), dtype=bf), None)
    # masked
    A3 = torch.zeros((2, 16, 64), dtype=bf)
    with pytest.raises(ValueError, match="experts and rows"):
        chord.chord_w4a16_grouped_gemm_masked(A3, g2, None, 64, 64, STORE, torch.zeros((2, 8, 64), dtype=bf), None)
    with pytest.raises(ValueError, match="bfloat16"):
        chord.chord_w4a16_grouped_gemm_masked(A3, g2, None, 64, 64, STORE, torch.zeros((2, 16, 64), dtype=f32), None)
    with pytest.raises(ValueError, match="C's last dimension"):
        chord.chord_w4a16_grouped_gemm_masked(A3, g2, None, 128, 64, SILU, torch.zeros((2, 16, 32), dtype=bf), None)
    # indexed: gathered A needs M token rows, C needs capacity rows
    st = torch.zeros(48, dtype=i32)
    e = torch.zeros(3, dtype=i32)
    with pytest.raises(ValueError, match="A holds"):
        chord.chord_w4a16_moe_gemm(A, True, None, 2, 64, 64, 16, 2, st, e, e, e, e, 16, STORE,
                                   torch.zeros((48, 64), dtype=bf), None)
    with pytest.raises(ValueError, match="C holds"):
        chord.chord_w4a16_moe_gemm(A, True, None, 2, 64, 64, 8, 2, st, e, e, e, e, 16, STORE,
                                   torch.zeros((40, 64), dtype=bf), None)
    with pytest.raises(ValueError, match="A holds"):
        chord.chord_w4a16_moe_gemm(A, False, None, 2, 64, 64, 8, 2, st, e, e, e, e, 16, STORE,
                                   torch.zeros((48, 64), dtype=bf), None)


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(chord, "_lib", None)
    monkeypatch.setattr(chord, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        chord.lib()


def test_product_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "w4a16_int4_weight_sigmoid_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "oracle/" not in text, f
