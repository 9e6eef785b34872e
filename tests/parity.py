"""Helpers shared by the GPU parity tests: tolerance checks against the oracle.

Tolerances (stated for the decode path): for every batch row b,
    max_n |y_gpu - y_oracle| <= 2e-3 * max_n |y_oracle|
    max_n |y_gpu - y_oracle| <= 1e-3 * sqrt(K) * max_k |x|
"""
import numpy as np

REL = 2e-3
ABS_PER_SQRTK = 1e-3


def tol_limits(y_ref: np.ndarray, x: np.ndarray, K: int) -> np.ndarray:
    y_ref = np.atleast_2d(y_ref)
    x = np.atleast_2d(x)
    lim = []
    for b in range(y_ref.shape[0]):
        lim.append(min(REL * np.abs(y_ref[b]).max(), ABS_PER_SQRTK * np.sqrt(K) * np.abs(x[b]).max()))
    return np.array(lim)


def assert_close(y_gpu: np.ndarray, y_ref: np.ndarray, x: np.ndarray, K: int, what: str = ""):
    y_gpu = np.atleast_2d(np.asarray(y_gpu, np.float64))
    y_ref = np.atleast_2d(y_ref)
    assert y_gpu.shape == y_ref.shape, (y_gpu.shape, y_ref.shape)
    assert np.all(np.isfinite(y_gpu)), f"{what}: non-finite output"
    lim = tol_limits(y_ref, x, K)
    err = np.abs(y_gpu - y_ref).max(axis=1)
    bad = np.nonzero(err > lim)[0]
    assert bad.size == 0, f"{what}: batch rows {bad.tolist()} err {err[bad]} > limit {lim[bad]}"
    return err, lim


def top2_margin(v: np.ndarray) -> float:
    s = np.sort(v)[::-1]
    return float(s[0] - s[1]) if s.size > 1 else float("inf")
