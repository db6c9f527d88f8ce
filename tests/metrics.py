"""Comparison metrics shared by the tests (no method arithmetic)."""
import numpy as np


def cosine(a, b):
    a = np.asarray(a, np.float64).ravel(); b = np.asarray(b, np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))


def rel_l2(a, ref):
    a = np.asarray(a, np.float64).ravel(); ref = np.asarray(ref, np.float64).ravel()
    return float(np.linalg.norm(a - ref) / max(np.linalg.norm(ref), 1e-300))


def norm_max_err(a, ref):
    """max|a - ref| / max|ref| (the parity tolerance's form)."""
    a = np.asarray(a, np.float64); ref = np.asarray(ref, np.float64)
    m = np.abs(ref).max(initial=0.0)
    return float(np.abs(a - ref).max(initial=0.0) / (m if m > 0 else 1.0))
