"""Pins of the prologue oracle (gate activation, q/k L2 normalisation) against
closed forms, invariants and central finite differences, and of its
composition with the recurrence oracle (the full operator with the prologue
on) against finite differences of the whole loss."""

import numpy as np
import pytest

from oracle.prologue import gate_bwd, gate_fwd, l2norm_bwd, l2norm_fwd


def _fd(f, x, eps=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        xp = x.copy()
        xm = x.copy()
        xp[i] += eps
        xm[i] -= eps
        g[i] = (f(xp) - f(xm)) / (2 * eps)
    return g


def test_gate_closed_forms():
    # softplus form: A_log = log 4, z = log 3 -> softplus(z) = log 4, g = -4 log 4
    g = gate_fwd(np.array([[np.log(3.0)]]), np.array([np.log(4.0)]))
    assert abs(g[0, 0] + 4.0 * np.log(4.0)) < 1e-14
    # z = 0: g = -exp(A) ln 2
    g = gate_fwd(np.zeros((1, 2)), np.array([0.0, np.log(2.0)]))
    assert np.allclose(g, [[-np.log(2.0), -2.0 * np.log(2.0)]], rtol=0, atol=1e-14)
    # lower-bound form: z = 0 gives lb / 2; every value lies in (lb, 0)
    g = gate_fwd(np.zeros((1, 1, 3)), np.array([0.7]), lower_bound=-5.0)
    assert np.allclose(g, -2.5, rtol=0, atol=1e-14)
    z = np.linspace(-10, 10, 41).reshape(41, 1, 1)
    g = gate_fwd(z, np.array([1.0]), lower_bound=-3.0)
    assert np.all(g > -3.0) and np.all(g < 0.0)
    # dt_bias enters additively: g(g_raw, dt) = g(g_raw + dt, 0)
    rng = np.random.default_rng(0)
    gr, dt, A = rng.normal(size=(4, 2, 3)), rng.normal(size=(2, 3)), rng.normal(size=2)
    assert np.allclose(gate_fwd(gr, A, dt), gate_fwd(gr + dt[None], A), rtol=0, atol=1e-14)


@pytest.mark.parametrize("scalar", [False, True])
@pytest.mark.parametrize("lb", [0.0, -4.0])
def test_gate_backward_matches_finite_differences(scalar, lb):
    rng = np.random.default_rng(1)
    shp = (5, 2) if scalar else (5, 2, 3)
    gr = rng.normal(size=shp)
    A = np.log(rng.uniform(1, 16, size=2))
    dt = rng.normal(size=shp[1:]) * 0.5
    dg = rng.normal(size=shp)

    def loss(gr_, A_, dt_):
        return float(np.sum(dg * gate_fwd(gr_, A_, dt_, lb)))

    dz, dA, ddt = gate_bwd(dg, gr, A, dt, lb)
    assert np.allclose(dz, _fd(lambda x: loss(x, A, dt), gr), rtol=1e-6, atol=1e-8)
    assert np.allclose(dA, _fd(lambda x: loss(gr, x, dt), A), rtol=1e-6, atol=1e-8)
    assert np.allclose(ddt, _fd(lambda x: loss(gr, A, x), dt), rtol=1e-6, atol=1e-8)


def test_l2norm_invariants_and_backward():
    rng = np.random.default_rng(2)
    x = rng.normal(size=(6, 4, 8))
    xh, r = l2norm_fwd(x, 0.0)
    assert np.allclose(np.sum(xh * xh, -1), 1.0, rtol=0, atol=1e-13)
    assert np.allclose(l2norm_fwd(3.7 * x, 0.0)[0], xh, rtol=0, atol=1e-13)   # scale invariance
    assert np.allclose(r, 1.0 / np.linalg.norm(x, axis=-1), rtol=1e-14)
    # eps sits inside the square root: a zero row stays zero and finite
    z, rz = l2norm_fwd(np.zeros((1, 8)), 1e-6)
    assert np.all(z == 0.0) and np.isclose(rz[0], 1e3)
    dxh = rng.normal(size=x.shape)
    dx = l2norm_bwd(dxh, x, 0.0)
    assert np.allclose(np.sum(dx * x, -1), 0.0, atol=1e-12)   # orthogonal to x without eps
    eps = 1e-3
    xs = x[:2, :1]
    ds = dxh[:2, :1]
    fd = _fd(lambda y: float(np.sum(ds * l2norm_fwd(y, eps)[0])), xs)
    assert np.allclose(l2norm_bwd(ds, xs, eps), fd, rtol=1e-6, atol=1e-9)


@pytest.mark.parametrize("gate,lb", [("channel", 0.0), ("channel", -4.0), ("scalar", 0.0)])
def test_prologue_composed_with_the_recurrence_matches_finite_differences(gate, lb):
    """The full operator with the prologue on: loss <do, o> + <dht, ht> of
    (l2norm(q), l2norm(k), v, beta, gate(g_raw)); its oracle gradients (the
    recurrence's BPTT composed with the prologue backward) against central
    differences of the loss in every raw input and parameter."""
    from oracle.cases import run_oracle_prologue_arrays
    rng = np.random.default_rng(3)
    T, H, K, V = 5, 2, 4, 3
    q = rng.normal(size=(T, H, K))
    k = rng.normal(size=(T, H, K))
    v = rng.normal(size=(T, H, V))
    beta = rng.uniform(0.2, 0.9, size=(T, H))
    gshape = (T, H, K) if gate == "channel" else (T, H)
    gr = rng.normal(size=gshape) * 0.5
    A = np.log(rng.uniform(1, 4, size=H))
    dt = rng.normal(size=gshape[1:]) * 0.3 - 1.0
    h0 = rng.normal(size=(1, H, K, V)) * 0.1
    do = rng.normal(size=(T, H, V))
    dht = rng.normal(size=(1, H, K, V))
    kw = dict(lower_bound=lb, eps=1e-6, scale=0.7, gate=gate, seq_starts=[0, T], h0=h0, do=do, dht=dht)

    def loss(q_=q, k_=k, gr_=gr, dt_=dt, A_=A):
        r = run_oracle_prologue_arrays(q_, k_, v, beta, gr_, A_log=A_, dt_bias=dt_, backward=False, **kw)
        return float(np.sum(do * r["o"]) + np.sum(dht * r["ht"]))

    ref = run_oracle_prologue_arrays(q, k, v, beta, gr, A_log=A, dt_bias=dt, backward=True, **kw)
    checks = (("dq", q, lambda y: loss(q_=y)), ("dk", k, lambda y: loss(k_=y)), ("dg", gr, lambda y: loss(gr_=y)),
              ("ddt_bias", dt, lambda y: loss(dt_=y)), ("dA_log", A, lambda y: loss(A_=y)))
    for key, x, f in checks:
        assert np.allclose(ref[key], _fd(f, x), rtol=1e-5, atol=1e-7), key
