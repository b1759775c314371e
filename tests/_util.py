"""Shared test helpers: parity metrics with the stated tolerances, and the
oracle-side input plumbing (re-exported from oracle.harness)."""
from __future__ import annotations

import numpy as np

from oracle.harness import bits, f64, oracle_pool, seq_token_mask  # noqa: F401

# Tolerances for bf16-in / fp32-accumulate outputs against the fp64 oracle
REL_L2 = 5e-3
MAX_ABS = 2e-2


def rel_l2(x, ref) -> float:
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm((x - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))


def max_abs(x, ref) -> float:
    return float(np.max(np.abs(np.asarray(x, np.float64) - np.asarray(ref, np.float64))))


def assert_close(x, ref, rel=REL_L2, mabs=MAX_ABS, what=""):
    r, m = rel_l2(x, ref), max_abs(x, ref)
    assert np.all(np.isfinite(np.asarray(x, np.float64))), f"{what}: non-finite values"
    assert r <= rel and m <= mabs, f"{what}: rel_l2={r:.3e} (<= {rel}) max_abs={m:.3e} (<= {mabs})"
    return r, m
