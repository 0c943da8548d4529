"""FP64 numpy restatement of the chunk form (forward WY, ReWY backward).

TEST INFRASTRUCTURE ONLY (see the package docstring).

One sequence, one head. Notation of "ReWY: Faster Backpropagation for
Delta-Rule Attention" (sections "The chunk system and conventional WY
backward", "ReWY: Algorithm and Analysis", Appendices A and "Complete
Gradients and Equivalence"), rows stacked, state S in R^{dk x dv}:

    G_i = sum_{t<=i} g_t (in-chunk, inclusive)      gamma = exp(G)
    X = K*gamma   E = diag(beta) X   Y = K/gamma   Z = diag(beta) V
    Q_g = scale*Q*gamma                  (the query scale is absorbed in Q)
    L = L_<(E Y^T)   M = I + L   A = M^{-1}
    W = A E   U = A Z   R = U - W S       (so M R = Z - E S)
    C_q = L_<=(Q_g Y^T)
    O = Q_g S + C_q R                     (read includes the current write)
    Lambda = diag(gamma_last)   F = Y Lambda
    S+ = Lambda S + F^T R

Those display equations were lost from the paper's text; they are rebuilt
here from its surrounding prose, from the four-token expansion of the "Kimi
Delta Attention" blog (section 6) and from the GatedDeltaNet-2 spec
transcription (section 2.5: u = A(beta v), w = A(beta exp(g) k)). The tests pin
the rebuilt forms against the recurrence oracle and against the paper's FLOP
counts.

Backward for one chunk, given the output adjoint O_bar and the adjoint S+_bar
of the outgoing state (accumulated from later chunks and dht):

    R_bar = C_q^T O_bar + F S+_bar            (both uses of R, before the pullback)
    H_q   = L_<=(O_bar R^T)
    ReWY (Algorithm 1):  P = A^T R_bar ;  D = -L_<(P R^T) ;  Z_bar = P ;
                         E_bar = -P S^T + D Y ;  Y_bar += D^T E ;
                         S_bar_res = -E^T P (supplied once)
    Q_g_bar = O_bar S^T + H_q Y ;  Y_bar += H_q^T Q_g + F_bar Lambda ;
    F_bar = R S+_bar^T ;  lambda_bar = rowsum(S .* S+_bar) + sum_i Y_i .* F_bar_i
    S_bar = Lambda S+_bar + Q_g^T O_bar - E^T P
    chain rule: dq = scale*gamma*Q_g_bar ; dk = beta*gamma*E_bar + Y_bar/gamma ;
                dv = beta*P ; dbeta = <X_i, E_bar_i> + <V_i, P_i> (undivided) ;
                G_bar = Q_g*Q_g_bar + E*E_bar - Y*Y_bar, plus gamma_last*lambda_bar
                at the last token ; dg = reverse in-chunk cumsum of G_bar.

The seven-product graph (same section) replaces the ReWY block by
    W_bar = -R_bar S^T ; A_bar = R_bar Z^T + W_bar E^T ; M_bar = -A^T A_bar A^T ;
    D = L_<(M_bar) ; Z_bar = A^T R_bar ; E_bar_dir = A^T W_bar ;
    S_bar_res = -W^T R_bar.
"""

from __future__ import annotations

import numpy as np


def tril(x, k=0):
    return np.tril(x, k)


def chunk_bounds(L: int, C: int):
    return [(a, min(a + C, L)) for a in range(0, L, C)]


def forward(q, k, v, beta, g, scale, h0=None, C=64):
    """Chunk-form forward. q,k [L,dk]; v [L,dv]; beta [L]; g [L,dk] (natural-log
    decay per channel; pass zeros for no gate and a broadcast column for a
    scalar gate). Returns o [L,dv], ht, and the per-chunk intermediates."""
    L, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if h0 is None else np.array(h0, dtype=np.float64)
    o = np.zeros((L, dv))
    chunks = []
    for a0, a1 in chunk_bounds(L, C):
        Q, Kc, Vc, b, gc = q[a0:a1], k[a0:a1], v[a0:a1], beta[a0:a1], g[a0:a1]
        n = a1 - a0
        G = np.cumsum(gc, axis=0)
        gam = np.exp(G)
        X = Kc * gam
        E = b[:, None] * X
        Y = Kc / gam
        Z = b[:, None] * Vc
        Qg = scale * Q * gam
        Lm = tril(E @ Y.T, -1)
        A = np.linalg.inv(np.eye(n) + Lm)
        W = A @ E
        U = A @ Z
        R = U - W @ S
        Cq = tril(Qg @ Y.T, 0)
        o[a0:a1] = Qg @ S + Cq @ R
        lam = gam[-1]
        F = Y * lam[None, :]
        chunks.append(dict(a0=a0, a1=a1, G=G, gam=gam, X=X, E=E, Y=Y, Z=Z, Qg=Qg, L=Lm, A=A,
                           W=W, U=U, R=R, Cq=Cq, lam=lam, F=F, S=S.copy()))
        S = lam[:, None] * S + F.T @ R
    return o, S, chunks


def intra_contractions(Hq, D, Kc, E, Qg, G, mode="direct", Y=None, gam=None, beta=None,
                       scale=None, Q=None):
    """The four matrix-intra contractions, already in physical coordinates:

        T_q = gamma * (H_q Y)      T_e = gamma * (D Y)
        T_y = (D^T E + H_q^T Q_g) / gamma

    "direct" evaluates them with gamma and 1/gamma as written; "centered"
    uses alpha = exp(G - c), zeta = exp(c - G) with the per-feature midpoint
    c = (max_i G + min_i G)/2 (the paper's centered factors); "pairwise" sums
    the per-pair factor exp(G_i - G_j) token pair by token pair.
    """
    n, dk = Kc.shape
    if mode == "direct":
        return gam * (Hq @ Y), gam * (D @ Y), (D.T @ E + Hq.T @ Qg) / gam
    if mode == "centered":
        c = 0.5 * (G.max(axis=0) + G.min(axis=0))
        al = np.exp(G - c[None, :])
        ze = np.exp(c[None, :] - G)
        Kz = Kc * ze
        Ea = beta[:, None] * Kc * al
        Qa = scale * Q * al
        return al * (Hq @ Kz), al * (D @ Kz), ze * (D.T @ Ea + Hq.T @ Qa)
    if mode == "pairwise":
        Tq = np.zeros((n, dk))
        Te = np.zeros((n, dk))
        Ty = np.zeros((n, dk))
        for i in range(n):
            for j in range(n):
                f = np.exp(G[i] - G[j])       # decay from token j to token i
                Tq[i] += Hq[i, j] * Kc[j] * f
                Te[i] += D[i, j] * Kc[j] * f
                # transposed contractions land on row j
                Ty[j] += D[i, j] * beta[i] * Kc[i] * f + Hq[i, j] * scale * Q[i] * f
        return Tq, Te, Ty
    raise ValueError(mode)


def backward(q, k, v, beta, g, scale, do, h0=None, dht=None, C=64, graph="rewy",
             intra="direct"):
    """Chunk-form backward. ``graph``: "rewy" (Algorithm 1) or "seven"
    (expanded WY graph). ``intra``: how the four interaction contractions are
    evaluated ("direct", "centered" or "pairwise"). Returns a dict of dq, dk,
    dv, dbeta, dg ([L, dk], per channel) and dh0, plus the outputs o, ht."""
    L, dk = k.shape
    dv = v.shape[1]
    o, ht, chunks = forward(q, k, v, beta, g, scale, h0=h0, C=C)
    Sb = np.zeros((dk, dv)) if dht is None else np.array(dht, dtype=np.float64)
    dq = np.zeros_like(q, dtype=np.float64)
    dk_ = np.zeros_like(k, dtype=np.float64)
    dv_ = np.zeros_like(v, dtype=np.float64)
    db = np.zeros(L)
    dg = np.zeros((L, dk))
    for ch in reversed(chunks):
        a0, a1 = ch["a0"], ch["a1"]
        Ob = do[a0:a1]
        S, R, A, E, Y, Z, Qg, Cq, F, W = (ch[x] for x in ("S", "R", "A", "E", "Y", "Z", "Qg", "Cq", "F", "W"))
        gam, lam, X, G = ch["gam"], ch["lam"], ch["X"], ch["G"]
        Kc, Vc, b, Q = k[a0:a1], v[a0:a1], beta[a0:a1], q[a0:a1]
        Sp = Sb                                   # adjoint of the outgoing state
        Rb = Cq.T @ Ob + F @ Sp
        Hq = tril(Ob @ R.T, 0)
        Fb = R @ Sp.T
        if graph == "rewy":
            P = A.T @ Rb
            D = -tril(P @ R.T, -1)
            Zb = P
            Eb_dir = -P @ S.T
            S_res = -E.T @ P
        elif graph == "seven":
            Wb = -Rb @ S.T
            Ab = Rb @ Z.T + Wb @ E.T
            Mb = -A.T @ Ab @ A.T
            D = tril(Mb, -1)
            Zb = A.T @ Rb
            Eb_dir = A.T @ Wb
            S_res = -W.T @ Rb
            P = Zb
        else:
            raise ValueError(graph)
        Tq, Te, Ty = intra_contractions(Hq, D, Kc, E, Qg, G, mode=intra, Y=Y, gam=gam,
                                        beta=b, scale=scale, Q=Q)
        # physical (gamma-scaled) adjoints: gamma*Q_g_bar, gamma*E_bar, Y_bar/gamma
        Qt = gam * (Ob @ S.T) + Tq
        Et = gam * Eb_dir + Te
        Yt = Ty + Fb * (lam[None, :] / gam)
        dq[a0:a1] = scale * Qt
        dk_[a0:a1] = b[:, None] * Et + Yt
        dv_[a0:a1] = b[:, None] * Zb
        db[a0:a1] = np.sum(Kc * Et, axis=1) + np.sum(Vc * Zb, axis=1)
        Gb = scale * Q * Qt + b[:, None] * Kc * Et - Kc * Yt
        lam_b = np.sum(S * Sp, axis=1) + np.sum(Y * Fb, axis=0)
        Gb[-1] += lam * lam_b
        dg[a0:a1] = np.cumsum(Gb[::-1], axis=0)[::-1]
        Sb = lam[:, None] * Sp + Qg.T @ Ob + S_res
    return dict(o=o, ht=ht, dq=dq, dk=dk_, dv=dv_, dbeta=db, dg=dg, dh0=Sb)


def gram_free_gate_terms(D, Kc, beta, G):
    """Scalar gate: the log-gate contributions of the erase coefficients
    L = L_<(diag(beta) Gamma-weighted K K^T), computed two ways.

    Returns (explicit, gram_free): explicit forms the key Gram matrix and takes
    row minus column sums of D .* L; gram_free uses only the key-gradient
    contractions A_K = C K and B_K = C^T K with C = diag(beta) Gamma,
    Gamma_ij = D_ij exp(G_i - G_j) ("Gram elimination for scalar-gate
    gradients" and its appendix proof)."""
    n = Kc.shape[0]
    Gs = G.reshape(n)
    Ex = np.exp(Gs[:, None] - Gs[None, :])
    Lm = tril(beta[:, None] * Ex * (Kc @ Kc.T), -1)
    J = D * Lm
    explicit = J.sum(axis=1) - J.sum(axis=0)
    Cm = beta[:, None] * D * Ex
    AK = Cm @ Kc
    BK = Cm.T @ Kc
    gram_free = np.sum(Kc * AK, axis=1) - np.sum(Kc * BK, axis=1)
    return explicit, gram_free


def wy_backward_flops(n: int, dk: int, dv: int):
    """Dense FLOPs (2 per multiply-add) of the local WY backward products.

    Seven-product graph: W_bar = -R_bar S^T (2 n dk dv); A_bar = R_bar Z^T +
    W_bar E^T (2 n^2 dv + 2 n^2 dk); -A^T A_bar A^T (4 n^3); Z_bar = A^T R_bar
    (2 n^2 dv); E_bar_dir = A^T W_bar (2 n^2 dk).
    ReWY: P = A^T R_bar (2 n^2 dv); P R^T (2 n^2 dv); P S^T (2 n dk dv)."""
    seven = 2 * n * dk * dv + 2 * n * n * dv + 2 * n * n * dk + 4 * n ** 3 + 2 * n * n * dv + 2 * n * n * dk
    rewy = 2 * n * n * dv + 2 * n * n * dv + 2 * n * dk * dv
    return seven, rewy
