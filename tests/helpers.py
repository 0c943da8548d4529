"""Shared test helpers: case conversion, oracle calls, error metrics."""

from __future__ import annotations

import numpy as np
import torch


def np64(x):
    if x is None:
        return None
    return x.detach().to("cpu", torch.float64).numpy()


def packed(case):
    """Case tensors as float64 numpy arrays on the packed token axis."""
    B, T, H = case.B, case.T, case.H
    d = dict(
        q=np64(case.q).reshape(B * T, H, case.K),
        k=np64(case.k).reshape(B * T, H, case.K),
        v=np64(case.v).reshape(B * T, H, case.V),
        beta=np64(case.beta).reshape(B * T, H),
        do=np64(case.do).reshape(B * T, H, case.V),
        h0=np64(case.h0),
        dht=np64(case.dht),
        g=None,
    )
    if case.g is not None:
        d["g"] = np64(case.g).reshape((B * T, H) + tuple(case.g.shape[3:]))
    return d


def run_oracle(case, backward=True, items=None, nthreads=None):
    from oracle import run_recurrence
    p = packed(case)
    return run_recurrence(p["q"], p["k"], p["v"], p["beta"], p["g"], case.seq_starts,
                          gate=case.gate, scale=case.scale, h0=p["h0"], do=p["do"],
                          dht=p["dht"], backward=backward, nthreads=nthreads, items=items)


def run_oracle_pairs(case, pairs, backward=True, nthreads=None):
    """Oracle on selected (sequence, head) pairs only; returns a dict of lists
    (one float64 array per pair) with the pair's token slice / state."""
    from oracle import run_recurrence
    p = packed(case)
    ss = case.seq_starts
    parts = {k: [] for k in ("q", "k", "v", "beta", "g", "do")}
    h0s, dhts, starts = [], [], [0]
    for (n, h) in pairs:
        a, b = ss[n], ss[n + 1]
        for key in parts:
            if p[key] is None:
                continue
            parts[key].append(p[key][a:b, h:h + 1])
        h0s.append(None if p["h0"] is None else p["h0"][n, h:h + 1])
        dhts.append(None if p["dht"] is None else p["dht"][n, h:h + 1])
        starts.append(starts[-1] + (b - a))
    cat = {k: (np.concatenate(v, axis=0) if v else None) for k, v in parts.items()}
    h0 = None if p["h0"] is None else np.stack(h0s, axis=0)
    dht = None if p["dht"] is None else np.stack(dhts, axis=0)
    res = run_recurrence(cat["q"], cat["k"], cat["v"], cat["beta"], cat["g"], starts,
                         gate=case.gate, scale=case.scale, h0=h0, do=cat["do"], dht=dht,
                         backward=backward, nthreads=nthreads)
    out = {}
    for key, val in res.items():
        if val is None:
            out[key] = None
            continue
        if key in ("ht", "dh0"):
            out[key] = [val[i, 0] for i in range(len(pairs))]
        else:
            out[key] = [val[starts[i]:starts[i + 1], 0] for i in range(len(pairs))]
    return out


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
