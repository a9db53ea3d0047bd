"""The chunkwise decomposition the CUDA kernels implement, written out in
float64 NumPy and checked against the oracle's per-token recurrence.

This pins the reading of "Parallel Scan", "The chunkwise algorithm" (three
decays per chunk: the mask D with unit diagonal, the decay from the chunk start
lambda that includes the first token's decay, the decay to the chunk end gamma
that excludes the writing token's own decay) and of the two-traversal backward
of "Lightning Attention-2", Algorithm 2, with those decays in place of powers
of one lambda.  Every chunk length, including 1 (the recurrence) and T (the
quadratic form) and ragged last chunks, must give the recurrence's outputs to
rounding.  It also checks the segment-level state passing ("Splitting one
sequence across devices") that the kernels use for chunk parallelism.
"""
import numpy as np
import pytest

import oracle


def _chunk_decays(log_a_chunk):
    """The three decays of one chunk from the segment-sum construction of
    "Long products without underflow": put log a in rows below the diagonal,
    take cumulative sums down each column, so entry (t, s) is the sum of log a
    over (s, t] from its own terms.  A virtual position 0 before the chunk
    gives the decays from the chunk start.  A reset (log a = -inf) yields 0."""
    L = len(log_a_chunk)
    ell = np.concatenate([[0.0], log_a_chunk])  # position 0 = before the chunk
    low = np.where(np.tril(np.ones((L + 1, L + 1)), -1) > 0, ell[:, None], 0.0)
    seg = np.cumsum(low, axis=0)  # seg[t, s] = sum_{u=s+1..t} ell_u, t >= s
    seg = np.where(np.tril(np.ones((L + 1, L + 1))) > 0, seg, -np.inf)
    D = np.exp(seg[1:, 1:])  # within-chunk mask, unit diagonal
    lam = np.exp(seg[1:, 0])  # from the chunk start, includes first decay
    gam = np.exp(seg[L, 1:])  # to the chunk end, excludes own decay
    return lam, gam, D, np.exp(seg[L, 0])


def chunked_fwd(Q, K, V, ell, S0, Tc):
    T = Q.shape[0]
    S = S0.copy()
    O = np.zeros((T, V.shape[1]))
    for t0 in range(0, T, Tc):
        sl = slice(t0, min(t0 + Tc, T))
        lam, gam, D, alpha = _chunk_decays(ell[sl])
        Qj, Kj, Vj = Q[sl], K[sl], V[sl]
        O[sl] = (Qj @ Kj.T * D) @ Vj + lam[:, None] * (Qj @ S)
        S = alpha * S + Kj.T @ (gam[:, None] * Vj)
    return O, S


def chunked_bwd(Q, K, V, ell, S0, dO, dST, Tc):
    """Two traversals: forward order for dQ (rebuilding S), reverse order for
    dK, dV with the adjoint state; then the closed-form decay gradient."""
    T, dk = Q.shape
    dv = V.shape[1]
    starts = list(range(0, T, Tc))
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    S = S0.copy()
    for t0 in starts:
        sl = slice(t0, min(t0 + Tc, T))
        lam, gam, D, alpha = _chunk_decays(ell[sl])
        Kj, Vj, dOj = K[sl], V[sl], dO[sl]
        dQ[sl] = (dOj @ Vj.T * D) @ Kj + lam[:, None] * (dOj @ S.T)
        S = alpha * S + Kj.T @ (gam[:, None] * Vj)
    ST = S
    dS = dST.copy()
    for t0 in reversed(starts):
        sl = slice(t0, min(t0 + Tc, T))
        lam, gam, D, alpha = _chunk_decays(ell[sl])
        Qj, Kj, Vj, dOj = Q[sl], K[sl], V[sl], dO[sl]
        dK[sl] = (dOj @ Vj.T * D).T @ Qj + gam[:, None] * (Vj @ dS.T)
        dV[sl] = (Qj @ Kj.T * D).T @ dOj + gam[:, None] * (Kj @ dS)
        dS = alpha * dS + (lam[:, None] * Qj).T @ dOj
    delta = np.sum(Q * dQ, 1) - np.sum(K * dK, 1)
    dl = np.cumsum(delta[::-1])[::-1] + np.sum(dST * ST)
    return dQ, dK, dV, dl, dS


def _inputs(seed, T, dk, dv, decay=(0.5, 1.0)):
    rng = np.random.default_rng(seed)
    Q = rng.standard_normal((T, dk))
    K = rng.standard_normal((T, dk))
    V = rng.standard_normal((T, dv))
    ell = np.log(rng.uniform(*decay, T))
    S0 = rng.standard_normal((dk, dv))
    dO = rng.standard_normal((T, dv))
    dST = rng.standard_normal((dk, dv))
    return Q, K, V, ell, S0, dO, dST


def _ora(Q, K, V, ell, S0, dO=None, dST=None):
    e = lambda x: x[None, None]
    o, ST = oracle.la_fwd(e(Q), e(K), e(V), e(ell), e(S0))
    if dO is None:
        return o[0, 0], ST[0, 0]
    g = oracle.la_bwd(e(Q), e(K), e(V), e(ell), e(S0), e(dO), e(dST))
    return (o[0, 0], ST[0, 0]) + tuple(x[0, 0] for x in g)


@pytest.mark.parametrize("Tc", [1, 2, 3, 4, 5, 8, 13, 19])
def test_every_chunk_length_gives_the_recurrence(Tc):
    T = 19
    Q, K, V, ell, S0, dO, dST = _inputs(Tc, T, 4, 3)
    o, ST, dq, dk, dv, dl, dS0 = _ora(Q, K, V, ell, S0, dO, dST)
    O2, S2 = chunked_fwd(Q, K, V, ell, S0, Tc)
    np.testing.assert_allclose(O2, o, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(S2, ST, rtol=1e-11, atol=1e-11)
    g = chunked_bwd(Q, K, V, ell, S0, dO, dST, Tc)
    for got, ref in zip(g, (dq, dk, dv, dl, dS0)):
        np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-10)


def test_constant_decay_la2_block_form():
    """Lightning Attention-2, eqs. 8 and 10 with lambda_r = lambda^r (r
    counted from 1) and gamma_r = lambda^(B - r): the block form reaches the
    per-token recurrence."""
    T, Bk, lam = 24, 8, 0.93
    Q, K, V, _, _, _, _ = _inputs(3, T, 5, 5)
    ell = np.full(T, np.log(lam))
    o, ST = _ora(Q, K, V, ell, np.zeros((5, 5)))
    r = np.arange(1, Bk + 1)
    M = np.tril(lam ** (r[:, None] - r[None, :]))
    KV = np.zeros((5, 5))
    O = np.zeros((T, 5))
    for i in range(0, T, Bk):
        sl = slice(i, i + Bk)
        O[sl] = (Q[sl] @ K[sl].T * M) @ V[sl] + (lam ** r)[:, None] * (Q[sl] @ KV)
        KV = lam ** Bk * KV + ((lam ** (Bk - r))[:, None] * K[sl]).T @ V[sl]
    np.testing.assert_allclose(O, o, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(KV, ST, rtol=1e-11, atol=1e-11)


def test_segment_state_passing():
    """Each segment runs from a zero state, giving its total decay and local
    final state; an exclusive scan of those pairs gives every segment's true
    incoming state; the correction diag(lambda) Q S_in completes the output."""
    T, Tc, seg = 50, 4, 3  # segments of 3 chunks; last segment ragged
    Q, K, V, ell, S0, _, _ = _inputs(11, T, 3, 4)
    o, ST = _ora(Q, K, V, ell, S0)
    L = Tc * seg
    pieces = []
    for p0 in range(0, T, L):
        sl = slice(p0, min(p0 + L, T))
        O_loc, S_loc = chunked_fwd(Q[sl], K[sl], V[sl], ell[sl], np.zeros_like(S0), Tc)
        pieces.append((sl, O_loc, S_loc, np.exp(np.sum(ell[sl]))))
    S_in = S0.copy()
    O = np.zeros_like(o)
    for sl, O_loc, S_loc, alpha in pieces:
        lam_seg = np.exp(np.cumsum(ell[sl]))
        O[sl] = O_loc + lam_seg[:, None] * (Q[sl] @ S_in)
        S_in = alpha * S_in + S_loc
    np.testing.assert_allclose(O, o, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(S_in, ST, rtol=1e-11, atol=1e-11)


def test_reset_decay_gives_zero_not_nan():
    """A reset (log a = -inf) inside a chunk: products become 0, never NaN,
    because every segment product is a sum of its own log terms."""
    T, Tc = 12, 4
    Q, K, V, ell, S0, _, _ = _inputs(5, T, 3, 3)
    ell[4] = -np.inf  # first token of the second chunk
    ell[10] = -np.inf  # inside the third chunk
    o, ST = _ora(Q, K, V, ell, S0)
    O2, S2 = chunked_fwd(Q, K, V, ell, S0, Tc)
    assert np.all(np.isfinite(O2))
    np.testing.assert_allclose(O2, o, rtol=1e-11, atol=1e-11)
