"""Helpers shared by the GPU parity tests (conversion and comparison only)."""
import numpy as np
import torch

REL_TOL = 1e-2      # relative Frobenius error of O against the oracle
ABS_TOL = 2e-2      # per-element absolute error of O against the oracle


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns on the host."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def compare_o(got: np.ndarray, ref: np.ndarray):
    """(relative Frobenius error, max abs error) of got against ref."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nr = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / nr if nr > 0 else np.linalg.norm(got)
    return float(rel), float(np.abs(got - ref).max()) if got.size else 0.0


def assert_o_close(got, ref, what=""):
    rel, mx = compare_o(got, ref)
    assert rel <= REL_TOL and mx <= ABS_TOL, f"{what}: rel {rel:.3e}, max abs {mx:.3e}"
    return rel, mx
