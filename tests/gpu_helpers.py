"""Shared helpers of the GPU parity tests: tolerances and comparisons."""
import numpy as np
import torch

# Spec bounds: fp32 inputs max-abs 1e-5; bf16 inputs (fp32 accumulation)
# max-abs 2e-2 and relative L2 5e-3.
F32_ATOL = 1e-5
BF16_ATOL = 2e-2
BF16_RL2 = 5e-3


def dev():
    return torch.device("cuda:0")


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def assert_bf16_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    rl2 = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)) if got.size else 0.0
    assert err <= BF16_ATOL and rl2 <= BF16_RL2, f"{what}: max-abs {err:.3e}, rel-L2 {rl2:.3e}"
    return err, rl2


def assert_f32_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = float(np.max(np.abs(got - ref)))
    assert err <= F32_ATOL, f"{what}: max-abs {err:.3e}"
    return err
