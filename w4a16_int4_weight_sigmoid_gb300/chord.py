"""Thin Python binding of libchord_moe.so (ctypes).

Argument marshalling only: every function here checks tensor dtypes and
devices, passes raw device pointers and the current CUDA stream to the C
entry point of the same name, and raises ChordError on a non-zero status.
All computation happens in the library's CUDA kernels; there is no CPU
fallback, and a missing library is an error.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libchord_moe.so")

CHORD_OK = 0
CHORD_ERR_INVALID_ARG = -1
CHORD_ERR_UNSUPPORTED = -2
CHORD_ERR_CUDA = -3
CHORD_ERR_WORKSPACE_TOO_SMALL = -4
CHORD_ERR_PREPACK_MISMATCH = -5
CHORD_ERR_TIMEOUT = -6
CHORD_ERR_ROUTING_INVALID = -7

CHORD_EPI_STORE = 0
CHORD_EPI_SILU_MUL = 1
CHORD_EPI_WEIGHTED_ADD = 2

CHORD_PATH_AUTO = 0
CHORD_PATH_SMALL_M = 1
CHORD_PATH_LARGE_M = 2


class ChordError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"chord error {code}: {msg}")
        self.code = code


class chord_tuning(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("rows_per_pass", ctypes.c_int),
                ("use_f16_accum", ctypes.c_int), ("batch_invariant", ctypes.c_int)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_Z = ctypes.c_size_t
_SIGS = {
    "chord_last_error_string": (ctypes.c_char_p, []),
    "chord_version": (_I, []),
    "chord_debug_force_timeout": (_I, [_I]),
    "chord_moe_route": (_I, [_P, _P, _I, _I, _I, _P, _P, _P]),
    "chord_moe_align_capacity": (_Z, [_I, _I, _I, _I]),
    "chord_moe_align_workspace_bytes": (_Z, [_I, _I, _I]),
    "chord_moe_align": (_I, [_P, _I, _I, _I, _I, _I, _Z, _P, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "chord_moe_align_noalloc": (_I, [_P, _I, _I, _I, _I, _I, _Z, _P, _P, _P, _P, _P, _P, _P]),
    "chord_moe_route_align": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _Z, _P, _P, _P, _P, _P, _P, _P, _P,
                                   _P, _Z, _P]),
    "chord_w4a16_prepack_bytes": (_Z, [_I, _I, _I, _I]),
    "chord_w4a16_prepack": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "chord_w4a16_moe_gemm_workspace_bytes": (_Z, [_Z, _I, _I]),
    "chord_w4a16_moe_gemm": (_I, [_P, _I, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _Z, _I,
                                  _P, _P, _P, _P, _Z, _P, _P]),
    "chord_moe_sum": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "chord_w4a16_gemm_workspace_bytes": (_Z, [_I]),
    "chord_w4a16_gemm": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _Z, _P, _P]),
    "chord_w4a16_grouped_workspace_bytes": (_Z, [_I, _Z]),
    "chord_w4a16_grouped_gemm_contiguous": (_I, [_P, _Z, _P, _I, _I, _P, _I, _I, _I, _P, _P, _P, _Z,
                                                 _P, _P]),
    "chord_w4a16_grouped_gemm_masked": (_I, [_P, _P, _I, _I, _I, _P, _I, _I, _I, _P, _P, _P, _Z, _P, _P]),
    "chord_moe_layer_workspace_bytes": (_Z, [_I, _I, _I, _I, _I]),
    "chord_moe_layer_plan": (_I, [_I, _I, _I, _P]),
    "chord_moe_layer": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _Z,
                             _P, _P, _P]),
}

_lib = None


def lib():
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "w4a16_int4_weight_sigmoid_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(rc: int):
    if rc != CHORD_OK:
        raise ChordError(rc, lib().chord_last_error_string().decode())


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _check_operands(A, C, K: int, N: int, epilogue: int, a_rows: int, c_rows: int, what: str):
    """Shape and dtype checks the C ABI cannot make (it sees raw pointers):
    A holds a_rows rows of K BF16 values and C holds c_rows rows of N (STORE)
    or N/2 (SiLU*mul) BF16 values.  Raises ValueError before anything runs."""
    for name, t in (("A", A), ("C", C)):
        if not isinstance(t, torch.Tensor):
            raise ValueError(f"{what}: {name} must be a torch.Tensor")
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{what}: {name} must be bfloat16, got {t.dtype}")
    if A.shape[-1] != K:
        raise ValueError(f"{what}: A's last dimension {A.shape[-1]} != K={K}")
    if A.numel() < a_rows * K:
        raise ValueError(f"{what}: A holds {A.numel()} values, needs {a_rows} rows of K={K}")
    ncols = N // 2 if epilogue == CHORD_EPI_SILU_MUL else N
    if C.shape[-1] != ncols:
        raise ValueError(f"{what}: C's last dimension {C.shape[-1]} != {ncols} "
                         f"({'N/2 for SiLU*mul' if epilogue == CHORD_EPI_SILU_MUL else 'N'})")
    if C.numel() < c_rows * ncols:
        raise ValueError(f"{what}: C holds {C.numel()} values, needs {c_rows} rows of {ncols}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _tuning(tuning):
    """None, a chord_tuning, or a path id."""
    if tuning is None:
        return None
    t = tuning if isinstance(tuning, chord_tuning) else chord_tuning(int(tuning), 0, 0, 0)
    return ctypes.byref(t), t


def chord_version() -> int:
    return lib().chord_version()


def chord_debug_force_timeout(enable: bool) -> None:
    """Test hook: later register-MMA GEMM launches withhold their work items,
    so their consumers' waits run out (CHORD_ERR_TIMEOUT, nothing computed)."""
    _check(lib().chord_debug_force_timeout(int(bool(enable))))


def chord_moe_route(logits, bias, topk: int, topk_weights, topk_ids, stream=None):
    M, E = logits.shape
    _check(lib().chord_moe_route(_ptr(logits, torch.float32, "logits"), _ptr(bias, torch.float32, "bias"),
                                 M, E, topk, _ptr(topk_weights, torch.float32, "topk_weights"),
                                 _ptr(topk_ids, torch.int32, "topk_ids"), _stream(stream)))


def chord_moe_align_capacity(M: int, topk: int, E_local: int, block_m: int) -> int:
    return lib().chord_moe_align_capacity(M, topk, E_local, block_m)


def chord_moe_align_workspace_bytes(M: int, topk: int, E_local: int) -> int:
    return lib().chord_moe_align_workspace_bytes(M, topk, E_local)


def chord_moe_align(topk_ids, expert_begin: int, E_local: int, block_m: int, sorted_token_ids,
                    expert_ids, num_tokens_post_padded, expert_counts, expert_offsets,
                    sorted_positions=None, workspace=None, stream=None):
    M, k = topk_ids.shape
    i32 = torch.int32
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().chord_moe_align(
        _ptr(topk_ids, i32, "topk_ids"), M, k, expert_begin, E_local, block_m,
        sorted_token_ids.numel(), _ptr(sorted_token_ids, i32, "sorted_token_ids"),
        _ptr(expert_ids, i32, "expert_ids"), _ptr(num_tokens_post_padded, i32, "ntpp"),
        _ptr(expert_counts, i32, "expert_counts"), _ptr(expert_offsets, i32, "expert_offsets"),
        _ptr(sorted_positions, i32, "sorted_positions"), _ptr(workspace, None, "workspace"),
        ws_bytes, _stream(stream)))


def chord_moe_route_align(logits, bias, topk: int, expert_begin: int, E_local: int, block_m: int,
                          topk_weights, topk_ids, sorted_token_ids, expert_ids, num_tokens_post_padded,
                          expert_counts, expert_offsets, sorted_positions=None, workspace=None,
                          stream=None):
    """chord_moe_route then chord_moe_align in one call (one launch for small M)."""
    M, E_total = logits.shape
    i32 = torch.int32
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().chord_moe_route_align(
        _ptr(logits, torch.float32, "logits"), _ptr(bias, torch.float32, "bias"), M, E_total, topk,
        expert_begin, E_local, block_m, sorted_token_ids.numel(),
        _ptr(topk_weights, torch.float32, "topk_weights"), _ptr(topk_ids, i32, "topk_ids"),
        _ptr(sorted_token_ids, i32, "sorted_token_ids"), _ptr(expert_ids, i32, "expert_ids"),
        _ptr(num_tokens_post_padded, i32, "ntpp"), _ptr(expert_counts, i32, "expert_counts"),
        _ptr(expert_offsets, i32, "expert_offsets"), _ptr(sorted_positions, i32, "sorted_positions"),
        _ptr(workspace, None, "workspace"), ws_bytes, _stream(stream)))


def chord_moe_align_noalloc(topk_ids, expert_begin: int, E_local: int, block_m: int,
                            sorted_token_ids, expert_ids, num_tokens_post_padded, expert_counts,
                            expert_offsets, sorted_positions=None, stream=None):
    """chord_moe_align without a workspace argument: for callers that cannot
    allocate device memory; its scratch is a static array in the library."""
    M, k = topk_ids.shape
    i32 = torch.int32
    _check(lib().chord_moe_align_noalloc(
        _ptr(topk_ids, i32, "topk_ids"), M, k, expert_begin, E_local, block_m,
        sorted_token_ids.numel(), _ptr(sorted_token_ids, i32, "sorted_token_ids"),
        _ptr(expert_ids, i32, "expert_ids"), _ptr(num_tokens_post_padded, i32, "ntpp"),
        _ptr(expert_counts, i32, "expert_counts"), _ptr(expert_offsets, i32, "expert_offsets"),
        _ptr(sorted_positions, i32, "sorted_positions"), _stream(stream)))


def chord_w4a16_prepack_bytes(E: int, N: int, K: int, group: int = 32) -> int:
    return lib().chord_w4a16_prepack_bytes(E, N, K, group)


def chord_w4a16_prepack(qweight, scales, gate_up: bool, packed, group: int = 32, stream=None):
    E, N, K2 = qweight.shape
    _check(lib().chord_w4a16_prepack(
        _ptr(qweight, torch.uint8, "qweight"), _ptr(scales, None, "scales"), E, N, 2 * K2, group,
        int(gate_up), _ptr(packed, torch.uint8, "packed"), packed.numel(), _stream(stream)))


def chord_w4a16_moe_gemm_workspace_bytes(capacity: int, K: int, a_gather: bool) -> int:
    return lib().chord_w4a16_moe_gemm_workspace_bytes(capacity, K, int(a_gather))


def chord_w4a16_moe_gemm(A, a_gather: bool, packed_w, E_local: int, N: int, K: int, M: int,
                         topk: int, sorted_token_ids, expert_ids, num_tokens_post_padded,
                         expert_counts, expert_offsets, block_m: int, epilogue: int, C, workspace,
                         tuning=None, dev_status=None, stream=None, topk_weights=None):
    """workspace: uint8 tensor of chord_w4a16_moe_gemm_workspace_bytes() bytes, zeroed once
    when allocated (the library keeps its counters zero).  CHORD_EPI_WEIGHTED_ADD: C is a
    float32 [M, N] accumulator the caller initialises, topk_weights float32 [M, topk]."""
    cap = sorted_token_ids.numel()
    if epilogue == CHORD_EPI_WEIGHTED_ADD:
        if not isinstance(C, torch.Tensor) or C.dtype != torch.float32 or C.numel() < M * N:
            raise ValueError("chord_w4a16_moe_gemm: the weighted add needs a float32 C of M x N values")
        if not isinstance(topk_weights, torch.Tensor) or topk_weights.numel() < M * topk:
            raise ValueError("chord_w4a16_moe_gemm: the weighted add needs topk_weights [M, topk]")
        _check_operands(A, A, K, K, CHORD_EPI_STORE, cap, 0, "chord_w4a16_moe_gemm")
    else:
        _check_operands(A, C, K, N, epilogue, M if a_gather else cap, cap, "chord_w4a16_moe_gemm")
    tun = _tuning(tuning)
    _check(lib().chord_w4a16_moe_gemm(
        _ptr(A, None, "A"), int(a_gather), _ptr(packed_w, torch.uint8, "packed_w"), E_local, N, K, M,
        topk, _ptr(sorted_token_ids, torch.int32, "sorted_token_ids"),
        _ptr(expert_ids, torch.int32, "expert_ids"),
        _ptr(num_tokens_post_padded, torch.int32, "num_tokens_post_padded"),
        _ptr(expert_counts, torch.int32, "expert_counts"),
        _ptr(expert_offsets, torch.int32, "expert_offsets"), block_m, sorted_token_ids.numel(),
        epilogue, _ptr(topk_weights, torch.float32, "topk_weights"), _ptr(C, None, "C"),
        tun[0] if tun else None, _ptr(workspace, torch.uint8, "workspace"),
        workspace.numel(), _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def chord_w4a16_gemm_workspace_bytes(M: int) -> int:
    return lib().chord_w4a16_gemm_workspace_bytes(M)


def chord_w4a16_gemm(A, packed_w, N: int, K: int, epilogue: int, C, workspace, tuning=None,
                     dev_status=None, stream=None):
    """Dense C = A (q*s)^T with a one-expert packed blob; workspace zeroed once when allocated."""
    if A.dim() != 2 or C.dim() != 2 or C.shape[0] != A.shape[0]:
        raise ValueError("chord_w4a16_gemm: A must be [M, K] and C [M, N or N/2] with the same rows")
    _check_operands(A, C, K, N, epilogue, A.shape[0], A.shape[0], "chord_w4a16_gemm")
    tun = _tuning(tuning)
    _check(lib().chord_w4a16_gemm(
        _ptr(A, None, "A"), _ptr(packed_w, torch.uint8, "packed_w"), N, K, A.shape[0], epilogue,
        _ptr(C, None, "C"), tun[0] if tun else None, _ptr(workspace, torch.uint8, "workspace"),
        workspace.numel(), _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def chord_w4a16_grouped_workspace_bytes(E: int, rows: int) -> int:
    return lib().chord_w4a16_grouped_workspace_bytes(E, rows)


def chord_w4a16_grouped_gemm_contiguous(A, group_rows, packed_w, N: int, K: int, epilogue: int, C, workspace,
                                        expected_m: int = 0, tuning=None, dev_status=None, stream=None):
    """Contiguous layout: A [rows, K], expert groups in order, each padded to 128 rows."""
    if A.dim() != 2:
        raise ValueError("contiguous layout: A must be [rows, K]")
    if C.dim() != 2 or C.shape[0] != A.shape[0]:
        raise ValueError("contiguous layout: C must be [rows, N or N/2] with the rows of A")
    _check_operands(A, C, K, N, epilogue, A.shape[0], A.shape[0], "chord_w4a16_grouped_gemm_contiguous")
    tun = _tuning(tuning)
    _check(lib().chord_w4a16_grouped_gemm_contiguous(
        _ptr(A, None, "A"), A.shape[0], _ptr(group_rows, torch.int32, "group_rows"), group_rows.numel(),
        expected_m, _ptr(packed_w, torch.uint8, "packed_w"), N, K, epilogue, _ptr(C, None, "C"),
        tun[0] if tun else None, _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def chord_w4a16_grouped_gemm_masked(A, group_rows, packed_w, N: int, K: int, epilogue: int, C, workspace,
                                    expected_m: int = 0, tuning=None, dev_status=None, stream=None):
    """Masked layout: A [E, max_m, K], the first group_rows[e] rows of expert e are used."""
    if A.dim() != 3 or group_rows.numel() != A.shape[0]:
        raise ValueError("masked layout: A must be [E, max_m, K] with one group_rows entry per expert")
    if C.dim() != 3 or C.shape[:2] != A.shape[:2]:
        raise ValueError("masked layout: C must be [E, max_m, N or N/2] with the experts and rows of A")
    _check_operands(A, C, K, N, epilogue, A.shape[0] * A.shape[1], A.shape[0] * A.shape[1],
                    "chord_w4a16_grouped_gemm_masked")
    tun = _tuning(tuning)
    _check(lib().chord_w4a16_grouped_gemm_masked(
        _ptr(A, None, "A"), _ptr(group_rows, torch.int32, "group_rows"), A.shape[0], A.shape[1], expected_m,
        _ptr(packed_w, torch.uint8, "packed_w"), N, K, epilogue, _ptr(C, None, "C"),
        tun[0] if tun else None, _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _ptr(dev_status, torch.int32, "dev_status"), _stream(stream)))


def chord_moe_sum(y, topk_weights, sorted_positions, out, stream=None):
    M, k = topk_weights.shape
    H = out.shape[1]
    _check(lib().chord_moe_sum(_ptr(y, None, "y"), _ptr(topk_weights, torch.float32, "topk_weights"),
                               _ptr(sorted_positions, torch.int32, "sorted_positions"), M, k, H,
                               _ptr(out, None, "out"), _stream(stream)))


def chord_moe_layer_workspace_bytes(M: int, H: int, I: int, E_local: int, topk: int) -> int:
    return lib().chord_moe_layer_workspace_bytes(M, H, I, E_local, topk)


def chord_moe_layer_plan(M: int, E_total: int, topk: int) -> chord_tuning:
    plan = chord_tuning()
    _check(lib().chord_moe_layer_plan(M, E_total, topk, ctypes.byref(plan)))
    return plan


def chord_moe_layer(x, logits, bias, w13_packed, w2_packed, H: int, I: int, E_total: int,
                    expert_begin: int, E_local: int, topk: int, out, workspace,
                    topk_weights_out=None, topk_ids_out=None, tuning=None, dev_status=None,
                    stream=None):
    M = x.shape[0]
    tun = _tuning(tuning)
    _check(lib().chord_moe_layer(
        _ptr(x, None, "x"), _ptr(logits, torch.float32, "logits"), _ptr(bias, torch.float32, "bias"),
        _ptr(w13_packed, torch.uint8, "w13_packed"), _ptr(w2_packed, torch.uint8, "w2_packed"),
        M, H, I, E_total, expert_begin, E_local, topk, _ptr(out, None, "out"),
        _ptr(topk_weights_out, torch.float32, "topk_weights_out"),
        _ptr(topk_ids_out, torch.int32, "topk_ids_out"), _ptr(workspace, torch.uint8, "workspace"),
        workspace.numel(), tun[0] if tun else None, _ptr(dev_status, torch.int32, "dev_status"),
        _stream(stream)))
