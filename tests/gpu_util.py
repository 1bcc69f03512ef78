"""Helpers shared by the GPU parity tests (comparison against the fp64 oracle)."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances of the parity bar (bf16 inputs, fp32 accumulation):
LOSS_REL = 1e-3      # |loss - oracle| <= 1e-3 * |oracle|
LSE_ABS = 2e-3       # max |lse - oracle|
GRAD_REL = 1e-2      # max |dX - oracle| <= 1e-2 * max |oracle|


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def check_loss(got: float, exp: float):
    assert abs(got - exp) <= LOSS_REL * max(abs(exp), 1e-30) or (exp == 0.0 and got == 0.0), \
        f"loss {got} vs oracle {exp}"


def check_lse(got, exp):
    err = np.abs(np.asarray(got, dtype=np.float64) - exp).max() if np.size(exp) else 0.0
    assert err <= LSE_ABS, f"lse max abs err {err}"


def check_grad(name: str, got, exp):
    got = np.asarray(got, dtype=np.float64)
    scale = np.abs(exp).max() if np.size(exp) else 0.0
    err = np.abs(got - exp).max() if np.size(exp) else 0.0
    if scale == 0.0:
        assert err == 0.0, f"{name}: expected zeros, max abs {err}"
    else:
        assert err <= GRAD_REL * scale, f"{name}: max abs err {err} > {GRAD_REL} * {scale}"
    return err / scale if scale else 0.0
