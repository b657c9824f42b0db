"""Error metric and small helpers shared by the tests."""
import numpy as np


def max_rel_err(y: np.ndarray, o: np.ndarray) -> float:
    """max_i |y_i - o_i| / max(|o_i|, tau), tau = 1e-2 * rms(o).

    The floor tau keeps cancellation near zero from dominating a relative
    measure; rows that are exactly zero in both give 0.
    """
    y = np.asarray(y, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    if o.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(o * o)))
    tau = max(1e-2 * rms, np.finfo(np.float64).tiny)
    return float(np.max(np.abs(y - o) / np.maximum(np.abs(o), tau)))


# Acceptance tolerances for combine (max relative error as defined above).
TOL_BF16_OUT = 1e-2
TOL_F32_OUT = 1e-5
