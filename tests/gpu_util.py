"""Helpers for the GPU parity tests: device upload, the parity bar, oracle
results for sampled tokens."""
import numpy as np
import torch

from w4a16_int4_weight_sigmoid_gb300 import build as B
from w4a16_int4_weight_sigmoid_gb300 import chord
from w4a16_int4_weight_sigmoid_gb300.layer import to_device  # noqa: F401

# Parity bar for layer outputs against the FP64 oracle.
MAXABS_FRAC = 1e-2      # max |gpu - oracle| <= 1e-2 * max |oracle|
REL_FROB = 5e-3         # ||gpu - oracle||_F <= 5e-3 * ||oracle||_F


def ensure_lib():
    B.build()
    chord.lib()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close_to_oracle(got: np.ndarray, ref: np.ndarray, what: str,
                           maxabs_frac=MAXABS_FRAC, rel_frob=REL_FROB):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    scale = np.abs(ref).max()
    if scale == 0:
        assert np.all(got == 0), f"{what}: expected zeros"
        return
    maxabs = np.abs(got - ref).max()
    fro = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert maxabs <= maxabs_frac * scale, f"{what}: max abs err {maxabs:.3e} > {maxabs_frac} * {scale:.3e}"
    assert fro <= rel_frob, f"{what}: rel Frobenius err {fro:.3e} > {rel_frob}"
