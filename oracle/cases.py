"""Case-level helpers around the recurrence oracle (packed arrays, sampled
(sequence, head) pairs).

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""

from __future__ import annotations

import numpy as np
import torch

from .recurrence import run_recurrence


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
    p = packed(case)
    return run_recurrence(p["q"], p["k"], p["v"], p["beta"], p["g"], case.seq_starts,
                          gate=case.gate, scale=case.scale, h0=p["h0"], do=p["do"],
                          dht=p["dht"], backward=backward, nthreads=nthreads, items=items)


def pairs_arrays(case, pairs):
    """float64 arrays of the selected (sequence, head) pairs, each pair one
    sequence of a single-head problem, plus its sequence starts."""
    ss = case.seq_starts
    B, T, H = case.B, case.T, case.H

    def sl(x, a, b, h):
        flat = x.reshape((B * T, H) + tuple(x.shape[3:]))
        return flat[a:b, h:h + 1].to(torch.float64).numpy()

    parts = {k: [] for k in ("q", "k", "v", "beta", "g", "do")}
    h0s, dhts, starts = [], [], [0]
    for (n, h) in pairs:
        a, b = ss[n], ss[n + 1]
        for key in parts:
            x = getattr(case, key)
            if x is not None:
                parts[key].append(sl(x, a, b, h))
        if case.h0 is not None:
            h0s.append(case.h0[n, h:h + 1].to(torch.float64).numpy())
        if case.dht is not None:
            dhts.append(case.dht[n, h:h + 1].to(torch.float64).numpy())
        starts.append(starts[-1] + (b - a))
    cat = {k: (np.concatenate(v, axis=0) if v else None) for k, v in parts.items()}
    cat["h0"] = np.stack(h0s, axis=0) if h0s else None
    cat["dht"] = np.stack(dhts, axis=0) if dhts else None
    return cat, starts


def run_pairs_arrays(case, cat, starts, backward=True, nthreads=None):
    return run_recurrence(cat["q"], cat["k"], cat["v"], cat["beta"], cat["g"], starts,
                          gate=case.gate, scale=case.scale, h0=cat["h0"], do=cat["do"],
                          dht=cat["dht"], backward=backward, nthreads=nthreads)


def run_oracle_pairs(case, pairs, backward=True, nthreads=None):
    """Oracle on selected (sequence, head) pairs only; returns a dict of lists
    (one float64 array per pair) with the pair's token slice / state."""
    cat, starts = pairs_arrays(case, pairs)
    res = run_pairs_arrays(case, cat, starts, backward=backward, nthreads=nthreads)
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


def run_oracle_prologue_arrays(q, k, v, beta, g_raw, *, A_log, dt_bias, lower_bound, eps, scale, gate,
                               seq_starts, h0=None, do=None, dht=None, backward=True, qk_norm=True,
                               nthreads=None, erase=None, write=None):
    """The operator with its prologue on, as a composition: q, k normalised
    per (token, head) (``qk_norm``), the decay activated from the raw gate
    (``A_log`` not None), then the recurrence; with ``backward`` the
    recurrence's gradients are carried back through the prologue
    (``oracle.prologue``). Adds dA_log and ddt_bias (None without dt_bias)."""
    from .prologue import gate_bwd, gate_fwd, l2norm_bwd, l2norm_fwd
    qh = l2norm_fwd(q, eps)[0] if qk_norm else np.asarray(q, dtype=np.float64)
    kh = l2norm_fwd(k, eps)[0] if qk_norm else np.asarray(k, dtype=np.float64)
    g = g_raw if (A_log is None or g_raw is None) else gate_fwd(g_raw, A_log, dt_bias, lower_bound)
    res = run_recurrence(qh, kh, v, beta, g, seq_starts, gate=gate, scale=scale, h0=h0, do=do, dht=dht,
                         backward=backward, nthreads=nthreads, erase=erase, write=write)
    if backward:
        if qk_norm:
            res["dq"] = l2norm_bwd(res["dq"], q, eps)
            res["dk"] = l2norm_bwd(res["dk"], k, eps)
        if A_log is not None and g_raw is not None:
            res["dg"], res["dA_log"], res["ddt_bias"] = gate_bwd(res["dg"], g_raw, A_log, dt_bias, lower_bound)
    return res
