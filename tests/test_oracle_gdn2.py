"""Pins of the GatedDeltaNet-2 branch of the recurrence oracle (erase vector b
on the key axis, write vector w on the value axis; "GatedDeltaNet-2 (NVlabs) —
official spec transcription", §3): reduction to the scalar-beta rule, the
chain rule of that reduction for beta's gradient, a one-token closed form
written out independently, and central finite differences of every gradient."""

import numpy as np
import pytest

from oracle import run_recurrence


def _case(rng, T, H, K, V, gate):
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, V))
    b = rng.uniform(0.0, 2.0, (T, H, K))
    w = rng.uniform(0.0, 1.0, (T, H, V))
    g = {"channel": rng.uniform(-2, 0, (T, H, K)), "scalar": rng.uniform(-2, 0, (T, H)), "none": None}[gate]
    return dict(q=q, k=k, v=v, b=b, w=w, g=g, h0=0.3 * rng.standard_normal((1, H, K, V)),
                do=rng.standard_normal((T, H, V)), dht=rng.standard_normal((1, H, K, V)), ss=[0, T])


def _run(d, gate, backward=True, beta=None):
    if beta is not None:
        return run_recurrence(d["q"], d["k"], d["v"], beta, d["g"], d["ss"], gate=gate, scale=0.6, h0=d["h0"],
                              do=d["do"], dht=d["dht"], backward=backward, nthreads=1)
    return run_recurrence(d["q"], d["k"], d["v"], None, d["g"], d["ss"], gate=gate, scale=0.6, h0=d["h0"],
                          do=d["do"], dht=d["dht"], backward=backward, nthreads=1, erase=d["b"], write=d["w"])


@pytest.mark.parametrize("gate", ["channel", "scalar", "none"])
def test_tied_vectors_reduce_to_the_beta_rule(gate):
    rng = np.random.default_rng(11)
    T, H, K, V = 9, 2, 4, 3
    d = _case(rng, T, H, K, V, gate)
    beta = rng.uniform(0.1, 0.9, (T, H))
    d["b"] = np.repeat(beta[:, :, None], K, axis=2)
    d["w"] = np.repeat(beta[:, :, None], V, axis=2)
    r2 = _run(d, gate)
    r1 = _run(d, gate, beta=beta)
    for name in ("o", "ht", "dq", "dk", "dv", "dh0") + (("dg",) if gate != "none" else ()):
        assert np.allclose(r2[name], r1[name], rtol=1e-12, atol=1e-12), name
    # d/dbeta of the tied parameterisation: every erase and write entry moves with beta
    tied = r2["derase"].sum(-1) + r2["dwrite"].sum(-1)
    assert np.allclose(tied, r1["dbeta"], rtol=1e-12, atol=1e-12)


def test_one_token_closed_form():
    rng = np.random.default_rng(12)
    K, V = 4, 3
    d = _case(rng, 1, 1, K, V, "channel")
    r = _run(d, "channel", backward=False)
    S = np.exp(d["g"][0, 0])[:, None] * d["h0"][0, 0]                 # decay
    rr = d["w"][0, 0] * d["v"][0, 0] - S.T @ (d["b"][0, 0] * d["k"][0, 0])
    S = S + np.outer(d["k"][0, 0], rr)                                 # write with k
    assert np.allclose(r["ht"][0, 0], S, rtol=1e-13, atol=1e-13)
    assert np.allclose(r["o"][0, 0], S.T @ (0.6 * d["q"][0, 0]), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("gate", ["channel", "scalar"])
def test_gdn2_gradients_match_finite_differences(gate):
    rng = np.random.default_rng(13)
    d = _case(rng, 6, 2, 4, 3, gate)
    ref = _run(d, gate)

    def loss(name, x):
        e = dict(d)
        e[name] = x
        r = _run(e, gate, backward=False)
        return float(np.sum(d["do"] * r["o"]) + np.sum(d["dht"] * r["ht"]))

    for name, key in (("b", "derase"), ("w", "dwrite"), ("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"),
                      ("h0", "dh0")):
        x = d[name]
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[i] += 1e-6
            xm[i] -= 1e-6
            fd[i] = (loss(name, xp) - loss(name, xm)) / 2e-6
        assert np.allclose(ref[key], fd, rtol=1e-6, atol=1e-8), name
