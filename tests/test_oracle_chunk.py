"""Pins for the numpy chunk-form restatement (CPU only).

The chunk form is pinned against the recurrence oracle (the pages call the
recurrent and chunkwise programs two schedules of one recurrence), against
the printed FLOP counts, and its alternative backward evaluations (ReWY vs
the seven-product graph; direct, centered and pairwise matrix intra; Gram
elimination vs the explicit key Gram matrix) against each other.
"""

import os

import numpy as np
import pytest

from oracle import chunk_ref, run_recurrence

GOLD = os.path.join(os.path.dirname(__file__), "golden", "wy_backward_flops.txt")


def _one_head(rng, L, K, V, gate, gmin=-1.0):
    q = rng.standard_normal((L, K))
    k = rng.standard_normal((L, K))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((L, V))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(L)))
    if gate == "channel":
        g = rng.uniform(gmin, 0.0, (L, K))
    elif gate == "scalar":
        g = np.repeat(rng.uniform(gmin, 0.0, (L, 1)), K, axis=1)
    else:
        g = np.zeros((L, K))
    h0 = 0.3 * rng.standard_normal((K, V))
    do = rng.standard_normal((L, V))
    dht = rng.standard_normal((K, V))
    return q, k, v, beta, g, h0, do, dht


def _oracle(q, k, v, beta, g, h0, do, dht, gate, scale):
    L = q.shape[0]
    gg = None if gate == "none" else (g[:, :1] if gate == "scalar" else g)
    gg = None if gg is None else (gg[:, None, 0] if gate == "scalar" else gg[:, None, :])
    return run_recurrence(q[:, None], k[:, None], v[:, None], beta[:, None], gg,
                          [0, L], gate=gate, scale=scale, h0=h0[None, None],
                          do=do[:, None], dht=dht[None, None], nthreads=1)


@pytest.mark.parametrize("C", [1, 4, 16, 64])
def test_chunk_forward_equals_recurrence(C):
    rng = np.random.default_rng(C)
    q, k, v, beta, g, h0, do, dht = _one_head(rng, 150, 12, 7, "channel")
    o, ht, chunks = chunk_ref.forward(q, k, v, beta, g, 0.4, h0=h0, C=C)
    r = _oracle(q, k, v, beta, g, h0, do, dht, "channel", 0.4)
    np.testing.assert_allclose(o, r["o"][:, 0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(ht, r["ht"][0, 0], rtol=1e-10, atol=1e-12)
    for ch in chunks:
        n = ch["a1"] - ch["a0"]
        np.testing.assert_allclose(ch["A"] @ (np.eye(n) + ch["L"]), np.eye(n), atol=1e-12)
        assert np.all(np.triu(ch["L"]) == 0.0)


@pytest.mark.parametrize("gate", ["channel", "scalar", "none"])
@pytest.mark.parametrize("graph", ["rewy", "seven"])
@pytest.mark.parametrize("C", [16, 64])
def test_chunk_backward_equals_bptt(gate, graph, C):
    rng = np.random.default_rng(100 + C)
    L = 141                                   # several chunks and a ragged tail
    q, k, v, beta, g, h0, do, dht = _one_head(rng, L, 10, 6, gate)
    beta[5] = 0.0
    res = chunk_ref.backward(q, k, v, beta, g, 0.3, do, h0=h0, dht=dht, C=C, graph=graph)
    r = _oracle(q, k, v, beta, g, h0, do, dht, gate, 0.3)
    for key in ("o", "dq", "dk", "dv", "dbeta"):
        np.testing.assert_allclose(res[key], r[key][:, 0], rtol=1e-9, atol=1e-11, err_msg=key)
    np.testing.assert_allclose(res["ht"], r["ht"][0, 0], rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(res["dh0"], r["dh0"][0, 0], rtol=1e-9, atol=1e-11)
    if gate == "channel":
        np.testing.assert_allclose(res["dg"], r["dg"][:, 0], rtol=1e-9, atol=1e-11)
    elif gate == "scalar":
        np.testing.assert_allclose(res["dg"].sum(axis=1), r["dg"][:, 0], rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("intra", ["centered", "pairwise"])
def test_matrix_intra_evaluations_agree(intra):
    """Centering by any per-feature midpoint and the pairwise evaluation give
    the directly factored contractions (paper: matrix-intra equivalence and
    centering)."""
    rng = np.random.default_rng(21)
    q, k, v, beta, g, h0, do, dht = _one_head(rng, 64, 8, 5, "channel", gmin=-0.5)
    a = chunk_ref.backward(q, k, v, beta, g, 0.5, do, h0=h0, dht=dht, C=64, intra="direct")
    b = chunk_ref.backward(q, k, v, beta, g, 0.5, do, h0=h0, dht=dht, C=64, intra=intra)
    for key in ("dq", "dk", "dbeta", "dg"):
        np.testing.assert_allclose(b[key], a[key], rtol=1e-10, atol=1e-12, err_msg=key)


def test_centered_factors_stay_bounded():
    """With the midpoint center the factors are bounded by exp(Delta/2)."""
    rng = np.random.default_rng(22)
    G = np.cumsum(rng.uniform(-3.0, 0.0, (64, 16)), axis=0)
    c = 0.5 * (G.max(axis=0) + G.min(axis=0))
    delta = G.max(axis=0) - G.min(axis=0)
    al = np.exp(G - c)
    ze = np.exp(c - G)
    bound = np.exp(delta / 2) * (1 + 1e-12)
    assert np.all(al <= bound) and np.all(ze <= bound)


def test_gram_elimination_equals_explicit_gram():
    rng = np.random.default_rng(23)
    n, K = 64, 16
    Kc = rng.standard_normal((n, K))
    beta = rng.uniform(0, 1, n)
    beta[3] = 0.0
    G = np.cumsum(rng.uniform(-0.3, 0.0, n))
    D = np.tril(rng.standard_normal((n, n)), -1)
    explicit, gram_free = chunk_ref.gram_free_gate_terms(D, Kc, beta, G)
    np.testing.assert_allclose(gram_free, explicit, rtol=1e-11, atol=1e-11)


def test_wy_flop_counts_match_printed_figures():
    rows = [l.split() for l in open(GOLD) if l.strip() and not l.startswith("#")]
    hdr, vals = rows[0], rows[1]
    rec = dict(zip(hdr, vals))
    n, dk, dv = int(rec["n"]), int(rec["dk"]), int(rec["dv"])
    seven, rewy = chunk_ref.wy_backward_flops(n, dk, dv)
    assert round(seven / 1e6, 2) == float(rec["seven_mflop"])
    assert round(rewy / 1e6, 2) == float(rec["rewy_mflop"])
    assert round(100 * (seven - rewy) / seven, 1) == float(rec["removed_percent"])
    # the difference is 4 n^2 dk + 4 n^3 (paper, "Arithmetic accounting")
    assert seven - rewy == 4 * n * n * dk + 4 * n ** 3
