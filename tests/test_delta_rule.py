"""The delta rule with a decay per head (Gated DeltaNet; "Parallel Scan", "What
one combine costs": a transition that is the identity minus a rank-one matrix
and overwrites what the state stores under a key; "At real scale": the layer)
-- the oracle pinned, and the chunkwise form a kernel implements checked
against it.

Reading (the pages name the structure but print no formula): in their row
convention (S [dk][dv], o_t = q_t S_t)
    S_t = a_t (I - beta_t k_t^T k_t) S_{t-1} + beta_t k_t^T v_t,
the form in which a unit-norm key written with beta = 1 stores exactly v_t:
k_t S_t = v_t.

Pins (each from outside the oracle's own formula): the overwrite property;
mutually orthogonal keys reduce it to decayed linear attention with values
beta_t v_t (the linear-attention oracle); beta = 0 leaves only the decay
(closed form); central finite differences for every gradient.

Chunkwise form ("What one combine costs": a product of rank-one corrections
stored as two thin factors, the WY representation): inside a chunk with
cumulative decays gamma_r = prod_{u<=r} a_u, the strictly lower triangular
A_rs = beta_r (gamma_r / gamma_s) k_r . k_s gives
    U = (I + A)^-1 diag(beta) V,   W = (I + A)^-1 diag(beta gamma) K,
and then, from the chunk's incoming state S,
    O = diag(gamma) Q S + ((Q K^T) . D) (U - W S)
    S' = gamma_L S + K^T diag(gamma_L / gamma) (U - W S)
with D_rs = gamma_r / gamma_s for s <= r -- the decayed linear-attention chunk
with the values U - W S.
"""
import numpy as np
import pytest

import oracle


def _rand(T=23, dk=5, dv=4, seed=0, unit_keys=True):
    rng = np.random.default_rng(seed)
    q = rng.normal(size=(1, 2, T, dk))
    k = rng.normal(size=(1, 2, T, dk))
    if unit_keys:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.normal(size=(1, 2, T, dv))
    la = -rng.uniform(0.0, 0.3, (1, 2, T))
    beta = rng.uniform(0.0, 1.0, (1, 2, T))
    S0 = rng.normal(size=(1, 2, dk, dv))
    return q, k, v, la, beta, S0


def test_overwrite_stores_the_value_under_its_key():
    """beta = 1, unit keys: reading with the key just written gives the value just written,
    whatever the state held and whatever the decay."""
    q, k, v, la, beta, S0 = _rand()
    o, _ = oracle.delta_fwd(k, k, v, la, np.ones_like(beta), S0)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-12)


def test_orthogonal_keys_reduce_to_decayed_linear_attention():
    """Keys orthogonal to every earlier key correct nothing (k_t S_{t-1} = 0 from a zero state),
    so the layer is decayed linear attention with values beta_t v_t."""
    rng = np.random.default_rng(3)
    T, dk, dv = 6, 6, 3
    Qm, _ = np.linalg.qr(rng.normal(size=(dk, dk)))
    k = (Qm * rng.uniform(0.5, 2.0, (dk, 1)))[None, None]  # orthogonal rows, any norms
    q = rng.normal(size=(1, 1, T, dk))
    v = rng.normal(size=(1, 1, T, dv))
    la = -rng.uniform(0, 0.5, (1, 1, T))
    beta = rng.uniform(0.1, 1.0, (1, 1, T))
    o, ST = oracle.delta_fwd(q, k, v, la, beta)
    ro, rST = oracle.la_fwd(q, k, v * beta[..., None], la)
    np.testing.assert_allclose(o, ro, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ST, rST, rtol=1e-12, atol=1e-12)


def test_beta_zero_leaves_only_the_decay():
    """beta = 0: S_t = (prod_{u<=t} a_u) S0, so o_t = (prod a) q_t S0."""
    q, k, v, la, beta, S0 = _rand()
    o, ST = oracle.delta_fwd(q, k, v, la, np.zeros_like(beta), S0)
    g = np.exp(np.cumsum(la, axis=-1))
    np.testing.assert_allclose(o, g[..., None] * np.einsum("bhti,bhij->bhtj", q, S0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ST, g[..., -1, None, None] * S0, rtol=1e-12, atol=1e-12)


def test_backward_matches_central_differences():
    q, k, v, la, beta, S0 = _rand(T=9, dk=3, dv=2, seed=5, unit_keys=False)
    rng = np.random.default_rng(9)
    dO = rng.normal(size=(1, 2, 9, 2))
    dST = rng.normal(size=(1, 2, 3, 2))
    grads = oracle.delta_bwd(q, k, v, la, beta, S0, dO, dST)

    def loss(q_, k_, v_, la_, b_, S0_):
        o, ST = oracle.delta_fwd(q_, k_, v_, la_, b_, S0_)
        return float(np.sum(o * dO) + np.sum(ST * dST))

    args = [q, k, v, la, beta, S0]
    h = 1e-6
    for which, g in zip((0, 1, 2, 3, 4, 5), grads[:3] + grads[3:5] + grads[5:]):
        x = args[which]
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            ap = list(args)
            am = list(args)
            ap[which], am[which] = xp, xm
            num[idx] = (loss(*ap) - loss(*am)) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-7, err_msg=f"argument {which}")


# ---------------------------------------------------------------- chunkwise form
def chunked_delta_fwd(q, k, v, la, beta, S0, C):
    """The chunkwise Gated DeltaNet forward (the module docstring's equations), float64."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, T, dv))
    ST = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            S = S0[b, h].copy() if S0 is not None else np.zeros((dk, dv))
            for c0 in range(0, T, C):
                sl = slice(c0, min(c0 + C, T))
                Q, K, V = q[b, h, sl], k[b, h, sl], v[b, h, sl]
                c = np.cumsum(la[b, h, sl])  # in-chunk log decays
                bt = beta[b, h, sl]
                n = len(c)
                G = np.exp(c[:, None] - c[None, :])  # gamma_r / gamma_s
                A = np.tril(bt[:, None] * G * (K @ K.T), -1)
                Tinv = np.linalg.inv(np.eye(n) + A)
                U = Tinv @ (bt[:, None] * V)
                W = Tinv @ ((bt * np.exp(c))[:, None] * K)
                Veff = U - W @ S
                D = np.tril(G)
                o[b, h, sl] = np.exp(c)[:, None] * (Q @ S) + ((Q @ K.T) * D) @ Veff
                S = np.exp(c[-1]) * S + K.T @ (np.exp(c[-1] - c)[:, None] * Veff)
            ST[b, h] = S
    return o, ST


@pytest.mark.parametrize("C", [1, 2, 3, 5, 8, 23, 64])
def test_chunkwise_wy_form_equals_the_recurrence(C):
    q, k, v, la, beta, S0 = _rand(T=23)
    o, ST = chunked_delta_fwd(q, k, v, la, beta, S0, C)
    ro, rST = oracle.delta_fwd(q, k, v, la, beta, S0)
    np.testing.assert_allclose(o, ro, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(ST, rST, rtol=1e-10, atol=1e-11)


def test_wy_factors_are_the_product_of_rank_one_corrections():
    """prod_{s = r..0} (I - beta_s k_s^T k_s) = I - K_r^T W_r (W without decay, from the same
    triangular system), of rank at most r + 1 -- the two thin factors of the pages."""
    rng = np.random.default_rng(2)
    n, dk = 5, 7
    K = rng.normal(size=(n, dk))
    bt = rng.uniform(0.1, 1.0, n)
    A = np.tril(bt[:, None] * (K @ K.T), -1)
    W = np.linalg.inv(np.eye(n) + A) @ (bt[:, None] * K)
    P = np.eye(dk)
    for r in range(n):
        P = (np.eye(dk) - bt[r] * np.outer(K[r], K[r])) @ P
        np.testing.assert_allclose(P, np.eye(dk) - K[: r + 1].T @ W[: r + 1], rtol=1e-12, atol=1e-12)
        assert np.linalg.matrix_rank(np.eye(dk) - P) <= r + 1


def chunked_delta_bwd(q, k, v, la, beta, S0, dO, dST, C):
    """The adjoint of the chunkwise form, chunk by chunk in reverse, float64: the states entering
    each chunk from a forward pass, then per chunk (n tokens, in-chunk log decays c, w = gamma_L / gamma)
        dU = P^T dO + diag(w) K dS',     dX = (I + A)^-T dU,     dV = diag(beta) dX
        dP = dO U^T (s <= r),            dA = -dX U^T (s < r)
        dQ = (dP . D) K + diag(gamma) dO S^T
        dK = (dP . D)^T Q + (F + F^T) K + diag(w) U dS'^T - diag(beta gamma) dX S^T,  F = beta_r dA_rs D_rs
        dbeta_r = (V - diag(gamma) K S)_r . dX_r + sum_s dA_rs D_rs k_r . k_s
        dS = gamma_L dS' + Q^T diag(gamma) dO - K^T diag(beta gamma) dX
    and the gradient on the in-chunk sums c (each product of decays differentiated in c),
    whose suffix sums inside the chunk are the gradient on each token's log decay."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dq, dkk = np.zeros((B, H, T, dk)), np.zeros((B, H, T, dk))
    dvv = np.zeros((B, H, T, dv))
    dl, db = np.zeros((B, H, T)), np.zeros((B, H, T))
    dS0 = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            S = S0[b, h].copy() if S0 is not None else np.zeros((dk, dv))
            starts = []
            for c0 in range(0, T, C):  # the states entering every chunk
                sl = slice(c0, min(c0 + C, T))
                starts.append(S.copy())
                _, S = chunked_delta_fwd(q[None, None, b, h, sl], k[None, None, b, h, sl], v[None, None, b, h, sl],
                                         la[None, None, b, h, sl], beta[None, None, b, h, sl], S[None, None], C)
                S = S[0, 0]
            dS = dST[b, h].copy() if dST is not None else np.zeros((dk, dv))
            for j, c0 in reversed(list(enumerate(range(0, T, C)))):
                sl = slice(c0, min(c0 + C, T))
                Q, K, V, dOc = q[b, h, sl], k[b, h, sl], v[b, h, sl], dO[b, h, sl]
                S = starts[j]
                c = np.cumsum(la[b, h, sl])
                bt = beta[b, h, sl]
                n = len(c)
                gam = np.exp(c)
                G = np.exp(c[:, None] - c[None, :])
                E = np.tril(G * (K @ K.T), -1)
                A = bt[:, None] * E
                Ti = np.linalg.inv(np.eye(n) + A)
                Yv = V - gam[:, None] * (K @ S)
                U = Ti @ (bt[:, None] * Yv)
                Dl = np.tril(G)
                P = (Q @ K.T) * Dl
                w = np.exp(c[-1] - c)
                KdS = K @ dS
                dU = P.T @ dOc + w[:, None] * KdS
                dX = Ti.T @ dU
                dP = np.tril(dOc @ U.T)
                dA = -np.tril(dX @ U.T, -1)
                G1 = dP * Dl
                F = bt[:, None] * dA * G
                dOSt = dOc @ S.T
                dq[b, h, sl] = G1 @ K + gam[:, None] * dOSt
                dkk[b, h, sl] = (G1.T @ Q + (F + F.T) @ K + (w[:, None] * U) @ dS.T
                                 - ((bt * gam)[:, None] * dX) @ S.T)
                dvv[b, h, sl] = bt[:, None] * dX
                db[b, h, sl] = np.sum(Yv * dX, 1) + np.sum(dA * E, 1)
                M1, M2 = dP * P, dA * A
                e = w * np.sum(KdS * U, 1)
                dc = (M1.sum(1) - M1.sum(0) + M2.sum(1) - M2.sum(0) + gam * np.sum(Q * dOSt, 1) - e
                      - bt * np.sum((V - Yv) * dX, 1))
                dc[-1] += e.sum() + gam[-1] * np.sum(S * dS)
                dl[b, h, sl] = np.cumsum(dc[::-1])[::-1]
                dS = gam[-1] * dS + Q.T @ (gam[:, None] * dOc) - K.T @ ((bt * gam)[:, None] * dX)
            dS0[b, h] = dS
    return dq, dkk, dvv, dl, db, dS0


@pytest.mark.parametrize("C", [1, 2, 3, 5, 8, 23, 64])
def test_chunkwise_adjoint_equals_the_recurrence_adjoint(C):
    """The chunk-by-chunk adjoint (what a backward kernel computes per chunk) gives the
    oracle's per-token adjoint for every chunking, short last chunks included."""
    q, k, v, la, beta, S0 = _rand(T=23, unit_keys=False)
    rng = np.random.default_rng(11)
    dO = rng.normal(size=(1, 2, 23, 4))
    dST = rng.normal(size=(1, 2, 5, 4))
    got = chunked_delta_bwd(q, k, v, la, beta, S0, dO, dST, C)
    want = oracle.delta_bwd(q, k, v, la, beta, S0, dO, dST)
    for name, g, r in zip(("dq", "dk", "dv", "dlog_a", "dbeta", "dS0"), got, want):
        np.testing.assert_allclose(g, r, rtol=1e-9, atol=1e-10, err_msg=name)
