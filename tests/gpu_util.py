"""Helpers shared by the GPU parity tests (no arithmetic of the method here)."""
import numpy as np


def to_dev(arrs, device="cuda"):
    import torch
    return {k: torch.from_numpy(np.ascontiguousarray(v)).to(device) for k, v in arrs.items()}


def np64(t):
    return t.detach().cpu().numpy().astype(np.float64)


def max_abs(x, ref):
    return float(np.max(np.abs(np.asarray(x, np.float64) - np.asarray(ref, np.float64))))


def rel_l2(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


# Tolerances stated for this method (potentials as a fraction of max C; plan
# applications as relative L2):
F_TOL_FMA = 1e-4        # FP32-FMA path
F_TOL_TENSOR = 1e-3     # tensor-core path
APPLY_TOL = 1e-3
