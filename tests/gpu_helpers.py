"""Shared helpers of the GPU parity tests: tolerances and comparisons."""
import math

import numpy as np
import torch

# Parity bounds: fp32 inputs max-abs 1e-5; bf16 inputs (fp32 accumulation)
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


def half_ulp_bf16(x) -> float:
    """Half a bf16 ulp at |x| (8 significant bits): 2^(e-8) for |x| in [2^e, 2^(e+1))."""
    x = abs(float(x))
    return 0.0 if x == 0.0 else math.ldexp(1.0, math.frexp(x)[1] - 9)


def assert_grad_close(got, ref, what, rl2_tol=BF16_RL2, abs_tol=BF16_ATOL, floor=1e-3,
                      bf16_storage=True):
    """Gradient comparison of the backward tests: relative L2 against
    max(||ref||, floor * sqrt(n)) and max-abs against abs_tol plus, for gradients
    stored in bf16, half an ulp of the largest reference entry (the rounding of the
    stored value alone; the derivation is in tests/test_gpu_bwd.py)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite"
    err = float(np.max(np.abs(got - ref)))
    rl2 = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), floor * math.sqrt(ref.size)))
    ref_max = float(np.max(np.abs(ref)))
    bound = abs_tol + (half_ulp_bf16(ref_max) if bf16_storage else 0.0)
    assert rl2 <= rl2_tol and err <= bound, \
        f"{what}: max-abs {err:.3e} (bound {bound:.3e}, ref max {ref_max:.3e}), rel-L2 {rl2:.3e}"
    return err, rl2
