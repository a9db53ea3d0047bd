"""The chunkwise algorithm for gated linear attention (one decay per key dimension), written
out in float64 NumPy and checked against the oracle's per-token recurrence.

"Parallel Scan", "The chunkwise algorithm", takes the matrix state with "a scalar, or a
diagonal over the keys" transition through the same chunk decomposition; this file fixes how
the diagonal case factors so that no term overflows however strong the decay.  With c_r[i] the
in-chunk sum of log a over tokens 1..r for key dimension i (every difference of two of them
formed as a segment sum from its own terms, so a reset gives 0, not NaN):

* inter-chunk: o_r += (q_r * e^{c_r}) S_in;  S_out = diag(e^{c_L}) S_in + sum_s (k_s * e^{c_L - c_s})^T v_s
  (every factor <= 1);
* intra-chunk, between a query sub-chunk R and an earlier key sub-chunk S' (sub-chunks of Bc
  tokens): P_{R,S'} = (Q_R * e^{C_R - c_e}) (K_S' * e^{c_e - C_S'})^T with e the last token of
  S', both factors <= 1;  inside a sub-chunk, P[r, s] = sum_i q_r[i] k_s[i] e^{c_r[i] - c_s[i]}
  term by term;
* backward: a forward-order traversal for dQ (rebuilding the state), a reverse-order one for
  dK and dV (carrying the adjoint), each with the same factorisations, and the decay gradient
  by the per-dimension closed form sum_{t>=u} (q_t * dq_t - k_t * dk_t) (+ the dS_T term).

Every chunk length (1 is the recurrence, T the quadratic form) and sub-chunk length must give
the recurrence's results to rounding.  This is the algebra a GLA kernel would implement.
"""
import numpy as np
import pytest

import oracle


class _Decays:
    """Per-dimension decays inside one chunk by segment sums ("Long products without
    underflow"): positions p = 0..L, p = 0 before the chunk's first token, p = r + 1 after token
    r.  between(p, q) = prod of a over the tokens q .. p - 1 (q <= p), one value per key
    dimension, from its own terms; a reset (log a = -inf) among them gives 0, never NaN."""

    def __init__(self, ell):
        L, dk = ell.shape
        reset = np.isneginf(ell)
        self.cs = np.vstack([np.zeros((1, dk)), np.cumsum(np.where(reset, 0.0, ell), axis=0)])
        last = np.full((L + 1, dk), -1)
        for r in range(L):
            last[r + 1] = np.where(reset[r], r, last[r])
        self.last = last  # last[p] = the last reset among tokens < p (-1: none)

    def between(self, p, q):
        d = np.exp(self.cs[p] - self.cs[q])
        d = np.where(self.last[p] >= q, 0.0, d)
        assert np.all(d <= 1.0 + 1e-12), "a factor above 1: the factorisation would overflow"
        return d

    def rows(self, ps, q):  # between(p, q) for p in ps, stacked
        return np.stack([self.between(p, q) for p in ps])

    def cols(self, p, qs):  # between(p, q) for q in qs, stacked
        return np.stack([self.between(p, q) for q in qs])


def _intra_scores(Qj, Kj, dec, Bc):
    """P[r, s] = sum_i q_r[i] k_s[i] a_{s+1..r}[i] for s <= r (0 above), by sub-chunks.  Between a
    query sub-chunk R and an earlier key sub-chunk S' the decay splits at S's last token e:
    a_{e+1..r} (a row factor) times a_{s+1..e} (a column factor), both <= 1."""
    L = Qj.shape[0]
    P = np.zeros((L, L))
    for r0 in range(0, L, Bc):
        R = range(r0, min(r0 + Bc, L))
        for s0 in range(0, r0, Bc):
            S = range(s0, min(s0 + Bc, L))
            e = S[-1]
            qf = Qj[R.start:R.stop] * dec.rows([r + 1 for r in R], e + 1)
            kf = Kj[S.start:S.stop] * dec.cols(e + 1, [s + 1 for s in S])
            P[R.start:R.stop, S.start:S.stop] = qf @ kf.T
        for r in R:  # the diagonal sub-block, term by term
            for s in range(R.start, r + 1):
                P[r, s] = np.sum(Qj[r] * Kj[s] * dec.between(r + 1, s + 1))
    return P


def _intra_weighted(A, Kj, dec, Bc):
    """X[r, i] = sum_{s<=r} A[r, s] k_s[i] a_{s+1..r}[i], by sub-chunks."""
    L, dk = Kj.shape
    X = np.zeros((L, dk))
    for r0 in range(0, L, Bc):
        R = range(r0, min(r0 + Bc, L))
        for s0 in range(0, r0, Bc):
            S = range(s0, min(s0 + Bc, L))
            e = S[-1]
            kf = Kj[S.start:S.stop] * dec.cols(e + 1, [s + 1 for s in S])
            X[R.start:R.stop] += (A[R.start:R.stop, S.start:S.stop] @ kf) * dec.rows([r + 1 for r in R], e + 1)
        for r in R:
            for s in range(R.start, r + 1):
                X[r] += A[r, s] * Kj[s] * dec.between(r + 1, s + 1)
    return X


def _intra_weighted_rev(A, Qj, dec, Bc):
    """Y[s, i] = sum_{r>=s} A[r, s] q_r[i] a_{s+1..r}[i], by sub-chunks (split at S's last token)."""
    L, dk = Qj.shape
    Y = np.zeros((L, dk))
    for s0 in range(0, L, Bc):
        S = range(s0, min(s0 + Bc, L))
        e = S[-1]
        for r0 in range(S.stop, L, Bc):
            R = range(r0, min(r0 + Bc, L))
            qf = Qj[R.start:R.stop] * dec.rows([r + 1 for r in R], e + 1)
            Y[S.start:S.stop] += (A[R.start:R.stop, S.start:S.stop].T @ qf) * dec.cols(e + 1, [s + 1 for s in S])
        for s in S:
            for r in range(s, S.stop):
                Y[s] += A[r, s] * Qj[r] * dec.between(r + 1, s + 1)
    return Y


def gla_chunked_fwd(Q, K, V, ell, S0, Tc, Bc):
    T = Q.shape[0]
    S = S0.copy()
    O = np.zeros((T, V.shape[1]))
    for t0 in range(0, T, Tc):
        sl = slice(t0, min(t0 + Tc, T))
        Qj, Kj, Vj = Q[sl], K[sl], V[sl]
        L = Qj.shape[0]
        dec = _Decays(ell[sl])
        lam = dec.rows(range(1, L + 1), 0)  # from the chunk's start through token r
        gam = dec.cols(L, range(1, L + 1))  # after token s to the chunk's end
        O[sl] = _intra_scores(Qj, Kj, dec, Bc) @ Vj + (Qj * lam) @ S
        S = dec.between(L, 0)[:, None] * S + (Kj * gam).T @ Vj
    return O, S


def gla_chunked_bwd(Q, K, V, ell, S0, dO, dST, Tc, Bc):
    T, dk = Q.shape
    starts = list(range(0, T, Tc))
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    S = S0.copy()
    for t0 in starts:  # forward order: dQ
        sl = slice(t0, min(t0 + Tc, T))
        Kj, Vj, dOj = K[sl], V[sl], dO[sl]
        L = Kj.shape[0]
        dec = _Decays(ell[sl])
        lam, gam = dec.rows(range(1, L + 1), 0), dec.cols(L, range(1, L + 1))
        dQ[sl] = _intra_weighted(np.tril(dOj @ Vj.T), Kj, dec, Bc) + (dOj @ S.T) * lam
        S = dec.between(L, 0)[:, None] * S + (Kj * gam).T @ Vj
    ST = S
    dS = dST.copy()
    for t0 in reversed(starts):  # reverse order: dK, dV with the adjoint state
        sl = slice(t0, min(t0 + Tc, T))
        Qj, Kj, Vj, dOj = Q[sl], K[sl], V[sl], dO[sl]
        L = Qj.shape[0]
        dec = _Decays(ell[sl])
        lam, gam = dec.rows(range(1, L + 1), 0), dec.cols(L, range(1, L + 1))
        dK[sl] = _intra_weighted_rev(np.tril(dOj @ Vj.T), Qj, dec, Bc) + (Vj @ dS.T) * gam
        dV[sl] = _intra_scores(Qj, Kj, dec, Bc).T @ dOj + (Kj * gam) @ dS
        dS = dec.between(L, 0)[:, None] * dS + (Qj * lam).T @ dOj
    dl = np.cumsum((Q * dQ - K * dK)[::-1], axis=0)[::-1] + np.sum(dST * ST, axis=1)[None, :]
    return dQ, dK, dV, dl, dS


def _inputs(seed, T, dk, dv, decay=(0.3, 1.0)):
    rng = np.random.default_rng(seed)
    Q = rng.standard_normal((T, dk))
    K = rng.standard_normal((T, dk))
    V = rng.standard_normal((T, dv))
    ell = np.log(rng.uniform(*decay, (T, dk)))
    S0 = rng.standard_normal((dk, dv))
    dO = rng.standard_normal((T, dv))
    dST = rng.standard_normal((dk, dv))
    return Q, K, V, ell, S0, dO, dST


def _oracle(Q, K, V, ell, S0, dO, dST):
    e = lambda x: x[None, None]
    o, ST = oracle.gla_fwd(e(Q), e(K), e(V), e(ell), e(S0))
    g = oracle.gla_bwd(e(Q), e(K), e(V), e(ell), e(S0), e(dO), e(dST))
    return o[0, 0], ST[0, 0], [x[0, 0] for x in g]


@pytest.mark.parametrize("Tc,Bc", [(1, 1), (2, 1), (4, 2), (8, 4), (16, 4), (16, 16), (13, 4), (37, 37)])
def test_gla_every_chunking_gives_the_recurrence(Tc, Bc):
    T, dk, dv = 37, 5, 3  # ragged last chunk for most Tc
    Q, K, V, ell, S0, dO, dST = _inputs(31, T, dk, dv)
    ro, rST, (rdq, rdk, rdv, rdl, rdS0) = _oracle(Q, K, V, ell, S0, dO, dST)
    O, ST = gla_chunked_fwd(Q, K, V, ell, S0, Tc, Bc)
    np.testing.assert_allclose(O, ro, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(ST, rST, rtol=1e-10, atol=1e-10)
    dq, dk_, dv_, dl, dS0 = gla_chunked_bwd(Q, K, V, ell, S0, dO, dST, Tc, Bc)
    for x, r in zip((dq, dk_, dv_, dl, dS0), (rdq, rdk, rdv, rdl, rdS0)):
        np.testing.assert_allclose(x, r, rtol=1e-9, atol=1e-9)


def test_gla_strong_decay_stays_finite():
    """Decays near 0 (log a down to -30 per token): e^{-c_s} alone would overflow within a few
    chunks' worth of tokens; the factorised form never forms it."""
    T, dk, dv = 48, 4, 3
    Q, K, V, _, S0, dO, dST = _inputs(32, T, dk, dv)
    ell = -np.random.default_rng(33).uniform(5.0, 30.0, (T, dk))
    ro, rST, (rdq, rdk, rdv, rdl, rdS0) = _oracle(Q, K, V, ell, S0, dO, dST)
    O, ST = gla_chunked_fwd(Q, K, V, ell, S0, 16, 4)
    assert np.all(np.isfinite(O))
    np.testing.assert_allclose(O, ro, rtol=1e-10, atol=1e-10)
    dq, dk_, dv_, dl, dS0 = gla_chunked_bwd(Q, K, V, ell, S0, dO, dST, 16, 4)
    for x, r in zip((dq, dk_, dv_, dl, dS0), (rdq, rdk, rdv, rdl, rdS0)):
        np.testing.assert_allclose(x, r, rtol=1e-9, atol=1e-9)


def test_gla_reset_in_one_dimension():
    """a = 0 in one key dimension at one token: writes before it stop reaching later reads
    through that dimension only."""
    T, dk, dv = 30, 4, 2
    Q, K, V, ell, S0, dO, dST = _inputs(34, T, dk, dv)
    ell[11, 2] = -np.inf
    ro, rST, _ = _oracle(Q, K, V, ell, S0, dO, dST)
    O, ST = gla_chunked_fwd(Q, K, V, ell, S0, 8, 4)
    np.testing.assert_allclose(O, ro, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(ST, rST, rtol=1e-10, atol=1e-10)
