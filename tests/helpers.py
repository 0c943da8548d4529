"""Shared test helpers: case conversion, oracle calls, error metrics."""

from __future__ import annotations

import json
import os

import numpy as np


from oracle.cases import np64, packed, run_oracle, run_oracle_pairs  # noqa: F401,E402


def rel_err(x, ref):
    """Normwise relative error ||x - ref||_2 / ||ref||_2 (float64)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((x - ref).ravel())
    if den == 0.0:
        return num
    return num / den


def check_close(name, x, ref, tol, abs_floor=1e-6):
    """Normwise relative error <= tol; for a near-zero reference the max-abs
    difference must stay below abs_floor. All values must be finite."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(x)), f"{name}: non-finite values"
    den = np.linalg.norm(ref.ravel())
    if den < abs_floor * np.sqrt(max(ref.size, 1)):
        err = float(np.max(np.abs(x - ref))) if x.size else 0.0
        assert err <= abs_floor, f"{name}: max-abs {err:.3e} > {abs_floor}"
        return err
    err = rel_err(x, ref)
    assert err <= tol, f"{name}: normwise relative error {err:.3e} > {tol}"
    return err


def record_errors(case_name, errs, **extra):
    """Appends one JSON line {case, errors per tensor, ...} to the file named by the environment
    variable KDA_PARITY_REPORT (nothing when it is unset): the per-tensor error margins of a GPU
    parity run, kept for the record."""
    path = os.environ.get("KDA_PARITY_REPORT")
    if not path:
        return
    rec = {"case": case_name, "errors": {k: float(v) for k, v in errs.items()}}
    rec.update(extra)
    with open(path, "a") as fh:
        fh.write(json.dumps(rec) + "\n")
