"""Shared helpers of the test-suite: run the oracle on the same seeded
inputs that the CUDA path gets, and compare."""
import numpy as np
import torch

from oracle import oracle


def rel_l2(got, want) -> float:
    g = got.detach().double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    w = np.asarray(want, np.float64)
    fin = np.isfinite(w)
    num = np.linalg.norm((g - w)[fin])
    den = np.linalg.norm(w[fin])
    return float(num / den) if den > 0 else float(num)


def max_abs(got, want) -> float:
    g = got.detach().double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    w = np.asarray(want, np.float64)
    fin = np.isfinite(w)
    return float(np.max(np.abs(g - w)[fin])) if fin.any() else 0.0


def f64(t):
    return t.detach().double().cpu().numpy()


def problem_of(x, w, H, p_drop=0.0, seed=0, offset=0):
    """oracle.Problem for synth inputs x of workload w."""
    return oracle.Problem(x.cu_seqlens.cpu().numpy(), H, w.D, w.span, w.nb, w.mp,
                          qmask=None if x.qmask is None else x.qmask.cpu().numpy(),
                          kmask=None if x.kmask is None else x.kmask.cpu().numpy(),
                          p_drop=p_drop, seed=seed, offset=offset)


def lse_to_oracle_layout(lse, packed, B, H, L):
    """GPU LSE ([B,H,L] padded or [H,T] packed) -> oracle [H,T]."""
    a = lse.detach().double().cpu().numpy()
    if packed:
        return a
    return a.transpose(1, 0, 2).reshape(H, B * L)
