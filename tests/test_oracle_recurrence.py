"""Pins for the FP64 recurrence oracle (CPU only).

Each test checks the oracle against something other than itself: central
finite differences, exact identities of the map, special cases with closed
forms from the pages, and the four-token chunk expansion of the "Kimi Delta
Attention" blog (section 6). A dropped term, a wrong sign, a transposed
operand or a decay applied after the prediction fails at least one of them.
"""

import numpy as np
import pytest

from oracle import run_recurrence


def _rand(rng, lens, H, K, V, gate, h0=True, dht=True, gmin=-2.0):
    T = sum(lens)
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, V))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    if gate == "channel":
        g = rng.uniform(gmin, 0.0, (T, H, K))
    elif gate == "scalar":
        g = rng.uniform(gmin, 0.0, (T, H))
    else:
        g = None
    N = len(lens)
    d = dict(q=q, k=k, v=v, beta=beta, g=g,
             h0=0.3 * rng.standard_normal((N, H, K, V)) if h0 else None,
             do=rng.standard_normal((T, H, V)),
             dht=rng.standard_normal((N, H, K, V)) if dht else None,
             ss=np.concatenate([[0], np.cumsum(lens)]).astype(np.int64))
    return d


def _run(d, gate, scale, backward=True, nthreads=1):
    return run_recurrence(d["q"], d["k"], d["v"], d["beta"], d["g"], d["ss"], gate=gate,
                          scale=scale, h0=d["h0"], do=d["do"], dht=d["dht"],
                          backward=backward, nthreads=nthreads)


def _loss(d, gate, scale):
    r = _run(d, gate, scale, backward=False)
    L = float(np.sum(d["do"] * r["o"]))
    if d["dht"] is not None:
        L += float(np.sum(d["dht"] * r["ht"]))
    return L


@pytest.mark.parametrize("gate", ["channel", "scalar", "none"])
@pytest.mark.parametrize("lens", [[1], [5, 3], [67]])
def test_central_differences(gate, lens):
    """Every gradient equals central finite differences of <do,o> + <dht,ht>."""
    rng = np.random.default_rng(7 + len(lens) + sum(lens))
    H, K, V = 2, 4, 3
    scale = 0.7
    d = _rand(rng, lens, H, K, V, gate)
    # one beta exactly zero: the undivided beta derivative must still hold
    d["beta"][0, 0] = 0.0
    an = _run(d, gate, scale)
    names = [("q", "dq"), ("k", "dk"), ("v", "dv"), ("beta", "dbeta"), ("h0", "dh0")]
    if gate != "none":
        names.append(("g", "dg"))
    h = 1e-6
    for x, dx in names:
        arr = d[x]
        fd = np.zeros_like(arr)
        flat = arr.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + h
            lp = _loss(d, gate, scale)
            flat[i] = old - h
            lm = _loss(d, gate, scale)
            flat[i] = old
            fd.reshape(-1)[i] = (lp - lm) / (2 * h)
        err = np.linalg.norm(fd - an[dx]) / max(np.linalg.norm(fd), 1e-300)
        assert err < 1e-7, (x, err)


@pytest.mark.parametrize("gate", ["channel", "scalar", "none"])
def test_linearity_identities(gate):
    """(o, ht) is linear in (v, h0) and o is linear in q while ht ignores q, so
    <dv,v> + <dh0,h0> = <do,o> + <dht,ht> and <dq,q> = <do,o> exactly."""
    rng = np.random.default_rng(11)
    d = _rand(rng, [130, 64, 1], 3, 16, 8, gate)
    r = _run(d, gate, 0.25, nthreads=3)
    lhs = np.sum(r["dv"] * d["v"]) + np.sum(r["dh0"] * d["h0"])
    rhs = np.sum(d["do"] * r["o"]) + np.sum(d["dht"] * r["ht"])
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(rhs))
    assert abs(np.sum(r["dq"] * d["q"]) - np.sum(d["do"] * r["o"])) <= 1e-10 * max(1.0, abs(rhs))


def test_beta_zero_only_decays():
    """beta = 0: nothing is written; the state only decays and each output is a
    read of the decayed initial state."""
    rng = np.random.default_rng(3)
    d = _rand(rng, [9], 1, 5, 4, "channel")
    d["beta"][:] = 0.0
    r = _run(d, "channel", 0.5)
    cum = np.exp(np.cumsum(d["g"][:, 0, :], axis=0))        # [T, K]
    S0 = d["h0"][0, 0]
    np.testing.assert_allclose(r["ht"][0, 0], cum[-1][:, None] * S0, rtol=1e-13, atol=1e-15)
    o_ref = np.stack([(cum[t][:, None] * S0).T @ (0.5 * d["q"][t, 0]) for t in range(9)])
    np.testing.assert_allclose(r["o"][:, 0], o_ref, rtol=1e-12, atol=1e-14)
    assert np.all(r["dv"] == 0.0)
    assert np.all(np.isfinite(r["dbeta"]))


def test_orthonormal_keys_recall():
    """No decay, beta = 1, orthonormal keys: after each write the state maps
    its key exactly to its value, and later orthogonal writes keep it so
    (blog, section 2.1: the write can be read back)."""
    rng = np.random.default_rng(5)
    K, V, T = 8, 6, 8
    Qm, _ = np.linalg.qr(rng.standard_normal((K, K)))
    k = Qm.T[:T][:, None, :]                         # rows orthonormal
    d = dict(q=k.copy(), k=k, v=rng.standard_normal((T, 1, V)), beta=np.ones((T, 1)), g=None,
             h0=rng.standard_normal((1, 1, K, V)), do=np.zeros((T, 1, V)), dht=None,
             ss=np.array([0, T], dtype=np.int64))
    r = _run(d, "none", 1.0, backward=False)
    # reading with q_t = k_t right after the write returns v_t
    np.testing.assert_allclose(r["o"][:, 0], d["v"][:, 0], rtol=0, atol=1e-12)
    S = r["ht"][0, 0]
    for j in range(T):
        np.testing.assert_allclose(S.T @ k[j, 0], d["v"][j, 0], rtol=0, atol=1e-12)


def test_write_is_local_in_key_space():
    """Without decay a write changes the state only along its key: for x
    orthogonal to k_0, x^T (S_0 - h0) = 0 (blog, section 2.1)."""
    rng = np.random.default_rng(6)
    K, V = 6, 5
    d = _rand(rng, [1], 1, K, V, "none")
    r = _run(d, "none", 1.0, backward=False)
    k0 = d["k"][0, 0]
    x = rng.standard_normal(K)
    x -= (x @ k0) * k0
    delta = r["ht"][0, 0] - d["h0"][0, 0]
    np.testing.assert_allclose(x @ delta, 0.0, atol=1e-13)
    # and along k_0 the read moves (1 - beta) of the way from old to v
    b = d["beta"][0, 0]
    old = d["h0"][0, 0].T @ k0
    np.testing.assert_allclose(r["ht"][0, 0].T @ k0, (1 - b) * old + b * d["v"][0, 0], atol=1e-13)


def test_single_token_closed_form():
    rng = np.random.default_rng(8)
    K, V = 5, 3
    d = _rand(rng, [1], 1, K, V, "channel")
    r = _run(d, "channel", 0.3, backward=False)
    a = np.exp(d["g"][0, 0])
    St = a[:, None] * d["h0"][0, 0]
    k0, v0, b0, q0 = d["k"][0, 0], d["v"][0, 0], d["beta"][0, 0], d["q"][0, 0]
    S1 = St + np.outer(k0, b0 * (v0 - St.T @ k0))
    np.testing.assert_allclose(r["ht"][0, 0], S1, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(r["o"][0, 0], S1.T @ (0.3 * q0), rtol=1e-14, atol=1e-15)


def test_four_token_chunk_expansion():
    """The blog's four-token chunk derivation (section 6): provisional errors
    from the decayed incoming state, causal substitution with
    rho_ij = beta_i <k_j| D_{j+1:i} |k_i>, outputs from chi_ij and the
    boundary-decayed queries, and the fast-forwarded end state. Written in the
    blog's value-by-key orientation and compared with the recurrence."""
    rng = np.random.default_rng(9)
    K, V, n, s = 6, 4, 4, 0.4
    d = _rand(rng, [n], 1, K, V, "channel")
    r = _run(d, "channel", s, backward=False)
    al = np.exp(d["g"][:, 0, :])                     # alpha_i, [n, K]
    Sc = d["h0"][0, 0].T                              # value x key
    kk, qq, vv, bb = d["k"][:, 0], d["q"][:, 0], d["v"][:, 0], d["beta"][:, 0]

    def Dr(a, b):                                     # D_a ... D_b (diagonal), identity if a > b
        out = np.ones(K)
        for t in range(a, b + 1):
            out = out * al[t]
        return out

    ebar = [bb[i] * (vv[i] - Sc @ (Dr(0, i) * kk[i])) for i in range(n)]
    rho = np.zeros((n, n))
    for i in range(n):
        for j in range(i):
            rho[i, j] = bb[i] * np.dot(kk[j], Dr(j + 1, i) * kk[i])
    e = []
    for i in range(n):
        e.append(ebar[i] - sum(rho[i, j] * e[j] for j in range(i)))
    S_end = Sc * Dr(0, n - 1)[None, :] + sum(np.outer(e[j], Dr(j + 1, n - 1) * kk[j]) for j in range(n))
    o = []
    for i in range(n):
        oi = s * Sc @ (Dr(0, i) * qq[i])
        for j in range(i + 1):
            oi = oi + s * np.dot(kk[j], Dr(j + 1, i) * qq[i]) * e[j]
        o.append(oi)
    np.testing.assert_allclose(r["o"][:, 0], np.stack(o), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["ht"][0, 0], S_end.T, rtol=1e-12, atol=1e-13)


def test_gate_family_reductions():
    """A per-channel gate broadcast from a scalar is GDN, and a zero gate is
    DeltaNet (ReWY paper, Table 1); the scalar log-gate gradient is the sum
    of the per-channel one over features."""
    rng = np.random.default_rng(10)
    d = _rand(rng, [70, 3], 2, 6, 5, "scalar")
    rs = _run(d, "scalar", 0.5)
    dc = dict(d)
    dc["g"] = np.repeat(d["g"][:, :, None], 6, axis=2)
    rc = _run(dc, "channel", 0.5)
    for key in ("o", "ht", "dq", "dk", "dv", "dbeta", "dh0"):
        np.testing.assert_allclose(rc[key], rs[key], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(rc["dg"].sum(axis=2), rs["dg"], rtol=1e-11, atol=1e-12)
    dz = dict(d)
    dz["g"] = np.zeros_like(dc["g"])
    rz = _run(dz, "channel", 0.5)
    rn = _run(d, "none", 0.5)
    for key in ("o", "ht", "dq", "dk", "dv", "dbeta", "dh0"):
        np.testing.assert_allclose(rz[key], rn[key], rtol=1e-13, atol=1e-14)


def test_thread_count_and_item_selection_do_not_change_results():
    rng = np.random.default_rng(12)
    d = _rand(rng, [100, 37, 64], 3, 8, 8, "channel")
    r1 = _run(d, "channel", 0.3, nthreads=1)
    r4 = _run(d, "channel", 0.3, nthreads=4)
    for key in r1:
        if r1[key] is not None:
            assert np.array_equal(r1[key], r4[key]), key
    rs = run_recurrence(d["q"], d["k"], d["v"], d["beta"], d["g"], d["ss"], gate="channel",
                        scale=0.3, h0=d["h0"], do=d["do"], dht=d["dht"], items=[(1, 2)])
    a, b = d["ss"][1], d["ss"][2]
    assert np.array_equal(rs["o"][a:b, 2], r1["o"][a:b, 2])
    assert np.array_equal(rs["dk"][a:b, 2], r1["dk"][a:b, 2])
    assert np.array_equal(rs["dh0"][1, 2], r1["dh0"][1, 2])
    assert np.all(rs["o"][a:b, 1] == 0.0)


def test_split_call_equals_one_call():
    """Resuming a sequence from its final state equals one call (forward), and
    the reverse pass chains dh0 of the later part into dht of the earlier."""
    rng = np.random.default_rng(13)
    d = _rand(rng, [90], 2, 6, 4, "channel")
    full = _run(d, "channel", 0.5)
    cut = 37
    a = {x: (None if d[x] is None else d[x][:cut]) for x in ("q", "k", "v", "beta", "g", "do")}
    b = {x: (None if d[x] is None else d[x][cut:]) for x in ("q", "k", "v", "beta", "g", "do")}
    a.update(h0=d["h0"], ss=np.array([0, cut], dtype=np.int64))
    b.update(ss=np.array([0, 90 - cut], dtype=np.int64), dht=d["dht"])
    a_f = _run(dict(a, dht=None), "channel", 0.5, backward=False)
    b.update(h0=a_f["ht"])
    rb = _run(b, "channel", 0.5)
    ra = _run(dict(a, dht=rb["dh0"]), "channel", 0.5)
    np.testing.assert_allclose(np.concatenate([ra["o"], rb["o"]]), full["o"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(rb["ht"], full["ht"], rtol=1e-12, atol=1e-13)
    for key in ("dq", "dk", "dv", "dbeta", "dg"):
        np.testing.assert_allclose(np.concatenate([ra[key], rb[key]]), full[key], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(ra["dh0"], full["dh0"], rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("gate", ["channel", "scalar", "none"])
def test_value_columns_are_independent_subproblems(gate):
    """The delta-rule update acts on each value column of the state on its own
    ("ReWY" paper, the state recurrence): splitting v, h0, do and dht into
    value blocks gives o, ht, dv, dh0 as the blocks' results side by side and
    dq, dk, dbeta, dg as the sums of the blocks' ones (the loss is the sum of
    the blocks' losses). This is what lets value widths above the kernels'
    tile run as value blocks."""
    rng = np.random.default_rng(17)
    d = _rand(rng, [70, 9], 2, 6, 11, gate)
    full = _run(d, gate, 0.5)
    cuts = [0, 4, 11]
    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        blk = dict(d, v=d["v"][..., a:b], do=d["do"][..., a:b], h0=d["h0"][..., a:b], dht=d["dht"][..., a:b])
        parts.append(_run(blk, gate, 0.5))
    for key in ("o", "ht", "dv", "dh0"):
        np.testing.assert_allclose(np.concatenate([p[key] for p in parts], axis=-1), full[key],
                                   rtol=1e-12, atol=1e-13)
    keys = ("dq", "dk", "dbeta") + (("dg",) if gate != "none" else ())
    for key in keys:
        np.testing.assert_allclose(sum(p[key] for p in parts), full[key], rtol=1e-10, atol=1e-12)
