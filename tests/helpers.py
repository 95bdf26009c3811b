"""Shared helpers of the parity tests (tolerances, uploads, oracle runs)."""

from __future__ import annotations

import numpy as np

REL_TOL = 1e-3      # |gpu - oracle| <= REL_TOL * max(|oracle_i|, rms(oracle))
MARGIN_TOL = 1e-4   # tokens may differ only where the oracle's top-2 margin is below this


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    scale = np.maximum(np.abs(ref), rms if rms > 0 else 1e-30)
    return np.abs(got - ref) / scale


def assert_close(got, ref, name="", tol=REL_TOL):
    err = rel_err(got, ref)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= tol, f"{name}: max scaled error {worst:.3e} > {tol:.1e} at flat index {int(err.argmax())}"
    return worst


def assert_token(gpu_tok, ref_tok, ref_margin, name=""):
    assert gpu_tok == ref_tok or ref_margin < MARGIN_TOL, (
        f"{name}: token {gpu_tok} != oracle {ref_tok} (oracle top-2 margin {ref_margin:.3e})")


def seeded_affine(rng, n, k):
    """Affine weight with the benchmark's value distributions from a numpy Generator."""
    q = rng.integers(0, 2 ** 32, size=(n, k // 8), dtype=np.uint64).astype(np.uint32)
    s = (np.abs(0.02 * rng.standard_normal((n, k // 32))) / 8).astype(np.float32)
    b = (-8.0 * s + 1e-3 * rng.standard_normal((n, k // 32))).astype(np.float32)
    return q, s, b
