"""FP64 oracle of the operator's optional prologue: the gate activation and
the per-(token, head) L2 normalisation of q and k, with their backward.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "GatedDeltaNet-2 (NVlabs) — official spec transcription", §2.0 (q and
k normalised before the chunk pipeline), §3 (the per-token gate-in-kernel
body: the head's A_log, the per-channel dt_bias added to the raw gate, then
either the softplus form or the lower-bound sigmoid form) and §4.2 (the
normalisation's eps sits inside the square root):

    z = g_raw + dt_bias
    softplus form:    g = -exp(A_log) * softplus(z)
    lower-bound form: g = lower_bound * sigmoid(exp(A_log) * z)      (-5 <= lower_bound < 0)
    x_hat = x / sqrt(sum_c x_c^2 + eps)

The backward is the chain rule of these closed forms, written out by hand:

    d/dz softplus(z) = sigmoid(z);  d/dz sigmoid(u) = s (1 - s)
    softplus form:    dg/dz = -exp(A) sigmoid(z),            dg/dA = g
    lower-bound form: dg/dz = lb s (1 - s) exp(A),  s = sigmoid(exp(A) z),
                      dg/dA = lb s (1 - s) exp(A) z
    dx = r (dx_hat - x_hat <x_hat, dx_hat>),  r = (sum x^2 + eps)^(-1/2)

dt_bias gets the sum over tokens of dg/dz times the upstream gradient (it
enters z additively); A_log the sum over tokens and channels of dg/dA times
it. Pinned in ``tests/test_oracle_prologue.py``.
"""

from __future__ import annotations

import numpy as np


def _softplus(z):
    # log(1 + e^z) without overflow
    return np.logaddexp(0.0, z)


def _sigmoid(z):
    return 0.5 * (1.0 + np.tanh(0.5 * z))


def gate_fwd(g_raw, A_log, dt_bias=None, lower_bound=0.0):
    """g_raw: [T, H, K] (per-channel) or [T, H] (scalar); A_log: [H];
    dt_bias: None, [H, K] or [H] (matching g_raw's trailing shape).
    Returns the natural-log decay g with g_raw's shape."""
    g_raw = np.asarray(g_raw, dtype=np.float64)
    A = np.asarray(A_log, dtype=np.float64)
    scalar = g_raw.ndim == 2
    z = g_raw + (0.0 if dt_bias is None else np.asarray(dt_bias, dtype=np.float64)[None])
    eA = np.exp(A)[None, :] if scalar else np.exp(A)[None, :, None]
    if lower_bound == 0.0:
        return -eA * _softplus(z)
    return lower_bound * _sigmoid(eA * z)


def gate_bwd(dg, g_raw, A_log, dt_bias=None, lower_bound=0.0):
    """Gradients of <dg, gate_fwd(...)>: (dg_raw, dA_log [H], ddt_bias or None)."""
    g_raw = np.asarray(g_raw, dtype=np.float64)
    dg = np.asarray(dg, dtype=np.float64)
    A = np.asarray(A_log, dtype=np.float64)
    scalar = g_raw.ndim == 2
    z = g_raw + (0.0 if dt_bias is None else np.asarray(dt_bias, dtype=np.float64)[None])
    eA = np.exp(A)[None, :] if scalar else np.exp(A)[None, :, None]
    if lower_bound == 0.0:
        dgdz = -eA * _sigmoid(z)
        dgdA = -eA * _softplus(z)
    else:
        s = _sigmoid(eA * z)
        dgdz = lower_bound * s * (1.0 - s) * eA
        dgdA = dgdz * z
    dz = dg * dgdz
    dA = dg * dgdA
    dA_log = dA.sum(axis=0) if scalar else dA.sum(axis=(0, 2))
    ddt = None if dt_bias is None else dz.sum(axis=0)
    return dz, dA_log, ddt


def l2norm_fwd(x, eps):
    """x: [..., C]; returns (x_hat, r) with r = (sum x^2 + eps)^(-1/2) per row."""
    x = np.asarray(x, dtype=np.float64)
    r = 1.0 / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)
    return x * r, r[..., 0]


def l2norm_bwd(dx_hat, x, eps):
    """Gradient of <dx_hat, x_hat(x)> with respect to x."""
    xh, r = l2norm_fwd(x, eps)
    dx_hat = np.asarray(dx_hat, dtype=np.float64)
    dot = np.sum(xh * dx_hat, axis=-1, keepdims=True)
    return r[..., None] * (dx_hat - xh * dot)
