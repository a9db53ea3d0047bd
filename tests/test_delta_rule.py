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
