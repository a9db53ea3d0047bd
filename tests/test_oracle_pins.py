"""Pins of the float64 oracle against what the pages and the mathematics fix.

None of these compare the oracle with itself: each checks it against a printed
worked example, a closed form, a brute-force evaluation of a different formula
(the quadratic mixing-matrix form, explicit segment products), or central
finite differences of the forward pass.
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------- diagonal scan
def test_composition_worked_example():
    """(0.5,1) then (0.5,0) is the single step (0.25,0.5): running the oracle
    over those two steps from any h0 gives 0.25 h0 + 0.5 exactly."""
    (a1, b1, a2, b2, A, Bc), = [list(map(float, r)) for r in _golden_rows("composition_example.txt")]
    for h0 in (0.0, 1.0, 2.0, -3.0, 1024.0):
        a = np.array([[[a1], [a2]]])
        b = np.array([[[b1], [b2]]])
        h, hT = oracle.scan_diag_fwd(a, b, np.array([[h0]]))
        assert hT[0, 0] == A * h0 + Bc
        assert h[0, 1, 0] == A * h0 + Bc


def test_identity_step_changes_nothing():
    rng = _rng(0)
    h0 = rng.standard_normal((2, 5))
    h, _ = oracle.scan_diag_fwd(np.ones((2, 1, 5)), np.zeros((2, 1, 5)), h0)
    assert np.array_equal(h[:, 0], h0)


def test_fold_example():
    (h0, a1, b1, h1), = [list(map(float, r)) for r in _golden_rows("fold_example.txt")]
    h, _ = oracle.scan_diag_fwd(np.array([[[a1]]]), np.array([[[b1]]]), np.array([[h0]]))
    assert h[0, 0, 0] == h1
    # folding h0 into b1 and scanning from 0 gives the same state
    hf, _ = oracle.scan_diag_fwd(np.array([[[a1]]]), np.array([[[b1 + a1 * h0]]]))
    assert hf[0, 0, 0] == h1


@pytest.mark.parametrize("a,b,h0", [(0.9, 1.0, 0.0), (0.5, -2.0, 3.0), (0.999, 0.25, -1.0)])
def test_geometric_closed_form(a, b, h0):
    """Constant decay and input: h_t = a^t h0 + b (1 - a^t) / (1 - a)."""
    T = 300
    h, hT = oracle.scan_diag_fwd(np.full((1, T, 1), a), np.full((1, T, 1), b), np.array([[h0]]))
    t = np.arange(1, T + 1)
    ref = a ** t * h0 + b * (1 - a ** t) / (1 - a)
    np.testing.assert_allclose(h[0, :, 0], ref, rtol=1e-12, atol=1e-12)
    assert hT[0, 0] == h[0, -1, 0]


def test_brute_force_segment_products():
    """h_t = prod_{u<=t} a_u h0 + sum_{s<=t} (prod_{u=s+1..t} a_u) b_s, each
    product formed from its own terms."""
    rng = _rng(1)
    B, T, D = 2, 9, 3
    a = rng.uniform(-1.2, 1.2, (B, T, D))
    b = rng.standard_normal((B, T, D))
    h0 = rng.standard_normal((B, D))
    h, _ = oracle.scan_diag_fwd(a, b, h0)
    for bi in range(B):
        for d in range(D):
            for t in range(T):
                ref = np.prod(a[bi, : t + 1, d]) * h0[bi, d]
                for s in range(t + 1):
                    ref += np.prod(a[bi, s + 1 : t + 1, d]) * b[bi, s, d]
                assert abs(h[bi, t, d] - ref) <= 1e-12 * (1 + abs(ref))


def test_split_run_equals_single_run():
    """Processing a sequence in two pieces, the second starting from the
    state where the first ended, gives the single run's states exactly."""
    rng = _rng(2)
    B, T, D = 2, 40, 4
    a, b, h0 = rng.uniform(0.5, 1, (B, T, D)), rng.standard_normal((B, T, D)), rng.standard_normal((B, D))
    h, hT = oracle.scan_diag_fwd(a, b, h0)
    for cut in (1, 17, 39):
        h1, hT1 = oracle.scan_diag_fwd(a[:, :cut], b[:, :cut], h0)
        h2, hT2 = oracle.scan_diag_fwd(a[:, cut:], b[:, cut:], hT1)
        assert np.array_equal(np.concatenate([h1, h2], 1), h)
        assert np.array_equal(hT2, hT)


def _fd_check(loss, params, grads, eps=1e-6, tol=1e-7, sample=None, seed=0):
    """Central differences of loss() w.r.t. each array in params (modified in
    place) against the analytic grads."""
    rng = _rng(seed)
    for name, p in params.items():
        g = grads[name]
        flat = p.reshape(-1)
        idxs = range(flat.size) if sample is None or flat.size <= sample else rng.choice(flat.size, sample, replace=False)
        for i in idxs:
            old = flat[i]
            flat[i] = old + eps
            lp = loss()
            flat[i] = old - eps
            lm = loss()
            flat[i] = old
            fd = (lp - lm) / (2 * eps)
            an = g.reshape(-1)[i]
            assert abs(fd - an) <= tol * (1 + abs(fd)), f"{name}[{i}]: fd {fd} vs analytic {an}"


def test_scan_backward_finite_differences():
    """A random recurrence of 50 steps: all three gradients against central
    finite differences of the forward pass."""
    rng = _rng(3)
    B, T, D = 2, 50, 3
    a = rng.uniform(0.6, 1.05, (B, T, D))
    b = rng.standard_normal((B, T, D))
    h0 = rng.standard_normal((B, D))
    g = rng.standard_normal((B, T, D))
    dhT = rng.standard_normal((B, D))

    def loss():
        h, hT = oracle.scan_diag_fwd(a, b, h0)
        return float(np.sum(g * h) + np.sum(dhT * hT))

    da, db, dh0 = oracle.scan_diag_bwd(a, b, h0, g, dhT)
    _fd_check(loss, dict(a=a, b=b, h0=h0), dict(a=da, b=db, h0=dh0), sample=60)


def test_scan_backward_is_reverse_scan():
    """The adjoint is the forward recurrence on reversed time with decays
    shifted by one: hbar = reversed scan of (a_{t+1}, g_t)."""
    rng = _rng(4)
    B, T, D = 1, 30, 2
    a, b, g = rng.uniform(0.5, 1, (B, T, D)), rng.standard_normal((B, T, D)), rng.standard_normal((B, T, D))
    da, db, _ = oracle.scan_diag_bwd(a, b, None, g)
    a_shift = np.concatenate([a[:, 1:], np.zeros((B, 1, D))], 1)
    hbar_rev, _ = oracle.scan_diag_fwd(a_shift[:, ::-1], g[:, ::-1])
    np.testing.assert_allclose(db, hbar_rev[:, ::-1], rtol=1e-13, atol=1e-13)


def test_pair_combine_associative_not_commutative():
    """The operator on pairs is associative; for dense 3x3 steps it is not
    commutative (later step's matrix on the left)."""
    rng = _rng(5)

    def comb(p1, p2):  # (A1,b1) then (A2,b2)
        return (p2[0] @ p1[0], p2[0] @ p1[1] + p2[1])

    ps = [(rng.standard_normal((3, 3)), rng.standard_normal(3)) for _ in range(3)]
    l = comb(comb(ps[0], ps[1]), ps[2])
    r = comb(ps[0], comb(ps[1], ps[2]))
    np.testing.assert_allclose(l[0], r[0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l[1], r[1], rtol=1e-12, atol=1e-12)
    x, y = comb(ps[0], ps[1]), comb(ps[1], ps[0])
    assert not np.allclose(x[0], y[0])
    # scalar pairs on dyadic values: exact associativity
    q = [(0.5, 1.0), (0.25, -3.0), (0.75, 0.5)]
    c = lambda p1, p2: (p1[0] * p2[0], p2[0] * p1[1] + p2[1])
    assert c(c(q[0], q[1]), q[2]) == c(q[0], c(q[1], q[2]))


def _hillis_steele_count(T):
    combines, rounds, shift = 0, 0, 1
    while shift < T:
        combines += T - shift
        rounds += 1
        shift *= 2
    return combines, rounds


def _blelloch_count(T):
    n = 1
    while n < T:
        n *= 2
    up = down = 0
    step = 1
    while step < n:
        up += n // (2 * step)
        step *= 2
    step = n // 2
    while step >= 1:
        down += n // (2 * step)
        step //= 2
    depth = 2 * int(math.log2(n))
    return up, down, T, depth


def test_scan_schedule_counts():
    """Work and depth of the two schedules at T = 1000, as printed."""
    g = {k: int(v) for k, v in _golden_rows("scan_schedule_counts.txt")}
    hs, hs_depth = _hillis_steele_count(g["T"])
    up, down, fix, depth = _blelloch_count(g["T"])
    assert hs == g["hillis_steele_combines"] and hs_depth == g["hillis_steele_depth"]
    assert (up, down, fix) == (g["blelloch_up"], g["blelloch_down"], g["blelloch_inclusive_fixup"])
    assert up + down + fix == g["blelloch_combines"] and depth == g["blelloch_depth"]
    assert g["T"] - 1 == g["loop_combines"]


def test_fp32_underflow_facts():
    """The float32 facts that rule out dividing running products."""
    g = {k: float(v) for k, v in _golden_rows("fp32_underflow_facts.txt")}
    P = np.cumprod(np.full(1200, 0.9, dtype=np.float32), dtype=np.float32)
    tiny = np.finfo(np.float32).tiny
    first_sub = int(np.argmax(P < tiny)) + 1  # 1-based step
    assert first_sub == int(g["decay_0.9_first_subnormal_step"])
    # first 1-based step s whose value persists: P_s == P_{s+1}
    stuck = next(t for t in range(1, 1200) if P[t] == P[t - 1])
    assert stuck == int(g["decay_0.9_first_stuck_step"])
    assert abs(float(P[stuck - 1]) - g["decay_0.9_stuck_value_approx"]) < 0.1e-45
    assert P[1099] / P[999] == g["decay_0.9_ratio_P1100_over_P1000"]
    e = np.float32(np.exp(np.float32(-0.5)))
    Q = np.cumprod(np.full(400, e, dtype=np.float32), dtype=np.float32)
    stuck_e = next(t for t in range(1, 400) if Q[t] == Q[t - 1])
    assert stuck_e == int(g["decay_exp(-0.5)_stuck_after_steps"])


# ----------------------------------------------------------------- selective scan
def _sel_inputs(rng, B, T, D, N):
    x = rng.standard_normal((B, T, D))
    delta = np.log1p(np.exp(rng.normal(-1.0, 0.5, (B, T, D))))
    A = -rng.uniform(0.2, 3.0, (D, N))
    Bm = rng.standard_normal((B, T, N))
    Cm = rng.standard_normal((B, T, N))
    h0 = rng.standard_normal((B, D, N))
    return x, delta, A, Bm, Cm, h0


def test_selective_brute_force():
    """y_t = sum_n C_t[n] (prod_{u<=t} a_u h0 + sum_{s<=t} prod_{u=s+1..t} a_u b_s)
    with a = exp(Delta A), b = Delta B x, from explicit products."""
    rng = _rng(6)
    B, T, D, N = 2, 7, 3, 4
    x, delta, A, Bm, Cm, h0 = _sel_inputs(rng, B, T, D, N)
    y, hT = oracle.selective_fwd(x, delta, A, Bm, Cm, h0)
    for bi in range(B):
        for d in range(D):
            hfin = np.zeros(N)
            for t in range(T):
                acc = 0.0
                for n in range(N):
                    a = np.exp(delta[bi, :, d] * A[d, n])
                    bb = delta[bi, :, d] * Bm[bi, :, n] * x[bi, :, d]
                    h = np.prod(a[: t + 1]) * h0[bi, d, n] + sum(np.prod(a[s + 1 : t + 1]) * bb[s] for s in range(t + 1))
                    acc += Cm[bi, t, n] * h
                    hfin[n] = h
                assert abs(y[bi, t, d] - acc) <= 1e-12 * (1 + abs(acc))
            np.testing.assert_allclose(hT[bi, d], hfin, rtol=1e-12, atol=1e-12)


def test_selective_reduces_to_diag_scan():
    """N = 1 and C = 1: y is the diagonal scan of (exp(Delta A), Delta B x)."""
    rng = _rng(7)
    B, T, D = 2, 33, 5
    x, delta, A, Bm, Cm, h0 = _sel_inputs(rng, B, T, D, 1)
    Cm = np.ones_like(Cm)
    y, _ = oracle.selective_fwd(x, delta, A, Bm, Cm, h0)
    h, _ = oracle.scan_diag_fwd(np.exp(delta * A[None, None, :, 0]), delta * Bm * x, h0[:, :, 0])
    np.testing.assert_allclose(y, h, rtol=1e-13, atol=1e-13)


def test_selective_backward_finite_differences():
    rng = _rng(8)
    B, T, D, N = 2, 12, 3, 4
    x, delta, A, Bm, Cm, h0 = _sel_inputs(rng, B, T, D, N)
    dy = rng.standard_normal((B, T, D))
    dhT = rng.standard_normal((B, D, N))

    def loss():
        y, hT = oracle.selective_fwd(x, delta, A, Bm, Cm, h0)
        return float(np.sum(dy * y) + np.sum(dhT * hT))

    dx, dd, dA, dB, dC, dh0 = oracle.selective_bwd(x, delta, A, Bm, Cm, h0, dy, dhT)
    _fd_check(loss, dict(x=x, delta=delta, A=A, Bm=Bm, Cm=Cm, h0=h0),
              dict(x=dx, delta=dd, A=dA, Bm=dB, Cm=dC, h0=dh0), sample=25, tol=2e-7)


# ----------------------------------------------------------------- linear attention
def _la_inputs(rng, B, H, T, dk, dv, decay=(0.6, 1.0)):
    q = rng.standard_normal((B, H, T, dk))
    k = rng.standard_normal((B, H, T, dk))
    v = rng.standard_normal((B, H, T, dv))
    log_a = np.log(rng.uniform(*decay, (B, H, T)))
    S0 = rng.standard_normal((B, H, dk, dv))
    return q, k, v, log_a, S0


def test_la_matches_quadratic_mixing_form():
    """T_c = T limit: O = (Q K^T * M) V + diag(lambda) Q S0 with
    M_ts = a_{t:s} = prod_{u=s+1..t} a_u (s <= t, diagonal 1) and
    lambda_t = prod_{u<=t} a_u, every product from its own terms."""
    rng = _rng(9)
    B, H, T, dk, dv = 1, 2, 11, 3, 4
    q, k, v, log_a, S0 = _la_inputs(rng, B, H, T, dk, dv)
    o, ST = oracle.la_fwd(q, k, v, log_a, S0)
    a = np.exp(log_a)
    for bi in range(B):
        for h in range(H):
            M = np.zeros((T, T))
            lam = np.zeros(T)
            for t in range(T):
                lam[t] = np.prod(a[bi, h, : t + 1])
                for s in range(t + 1):
                    M[t, s] = np.prod(a[bi, h, s + 1 : t + 1])
            Q, K, V = q[bi, h], k[bi, h], v[bi, h]
            ref = (Q @ K.T * M) @ V + lam[:, None] * (Q @ S0[bi, h])
            np.testing.assert_allclose(o[bi, h], ref, rtol=1e-12, atol=1e-12)
            ST_ref = lam[-1] * S0[bi, h] + (K * M[-1][:, None]).T @ V
            np.testing.assert_allclose(ST[bi, h], ST_ref, rtol=1e-12, atol=1e-12)


def test_la_no_decay_is_causal_linear_attention():
    """a = 1, S0 = 0: unnormalised causal linear attention tril(Q K^T) V."""
    rng = _rng(10)
    q, k, v, _, _ = _la_inputs(rng, 2, 1, 16, 5, 3)
    o, _ = oracle.la_fwd(q, k, v, np.zeros((2, 1, 16)))
    for bi in range(2):
        Q, K, V = q[bi, 0], k[bi, 0], v[bi, 0]
        np.testing.assert_allclose(o[bi, 0], np.tril(Q @ K.T) @ V, rtol=1e-12, atol=1e-12)


def test_la_constant_decay_closed_form():
    """Constant decay (Lightning Attention-2, eq. 4 unrolled):
    o_t = q_t sum_{s<=t} lambda^{t-s} k_s^T v_s."""
    rng = _rng(11)
    T, d = 20, 4
    q, k, v, _, _ = _la_inputs(rng, 1, 1, T, d, d)
    lam = 0.9
    o, _ = oracle.la_fwd(q, k, v, np.full((1, 1, T), math.log(lam)))
    Q, K, V = q[0, 0], k[0, 0], v[0, 0]
    for t in range(T):
        ref = sum(lam ** (t - s) * (Q[t] @ K[s]) * V[s] for s in range(t + 1))
        np.testing.assert_allclose(o[0, 0, t], ref, rtol=1e-12, atol=1e-12)


def test_la_backward_finite_differences():
    rng = _rng(12)
    B, H, T, dk, dv = 1, 2, 9, 3, 2
    q, k, v, log_a, S0 = _la_inputs(rng, B, H, T, dk, dv)
    dO = rng.standard_normal((B, H, T, dv))
    dST = rng.standard_normal((B, H, dk, dv))

    def loss():
        o, ST = oracle.la_fwd(q, k, v, log_a, S0)
        return float(np.sum(dO * o) + np.sum(dST * ST))

    dq, dk_, dv_, dl, dS0 = oracle.la_bwd(q, k, v, log_a, S0, dO, dST)
    _fd_check(loss, dict(q=q, k=k, v=v, log_a=log_a, S0=S0),
              dict(q=dq, k=dk_, v=dv_, log_a=dl, S0=dS0), sample=30, tol=2e-7)


def test_la_backward_spans_checkpoint_blocks():
    """T larger than the oracle's internal checkpoint interval: gradients by
    finite differences at sampled points."""
    rng = _rng(13)
    B, H, T, dk, dv = 1, 1, 150, 2, 2
    q, k, v, log_a, S0 = _la_inputs(rng, B, H, T, dk, dv, decay=(0.9, 1.0))
    dO = rng.standard_normal((B, H, T, dv))

    def loss():
        o, _ = oracle.la_fwd(q, k, v, log_a, S0)
        return float(np.sum(dO * o))

    dq, dk_, dv_, dl, dS0 = oracle.la_bwd(q, k, v, log_a, S0, dO)
    _fd_check(loss, dict(k=k, log_a=log_a, S0=S0), dict(k=dk_, log_a=dl, S0=dS0), sample=12, tol=1e-6)


def test_la_closed_form_decay_gradient_equals_definition():
    """dL/dlog a_u = sum_{t>=u} q_t.dq_t - sum_{s>=u} k_s.dk_s (+ <dS_T, S_T>)
    equals a_u <Sbar_u, S_{u-1}> (states never needed)."""
    rng = _rng(14)
    B, H, T, dk, dv = 2, 2, 70, 4, 3
    q, k, v, log_a, S0 = _la_inputs(rng, B, H, T, dk, dv, decay=(0.8, 1.0))
    dO = rng.standard_normal((B, H, T, dv))
    dST = rng.standard_normal((B, H, dk, dv))
    _, ST = oracle.la_fwd(q, k, v, log_a, S0)
    dq, dk_, _, dl, _ = oracle.la_bwd(q, k, v, log_a, S0, dO, dST)
    dl_cf = oracle.la_dlog_closed_form(q, k, dq, dk_, dST, ST)
    np.testing.assert_allclose(dl_cf, dl, rtol=1e-10, atol=1e-10)


# ---------------------------------------------------------------- gated linear attention
def _gla_inputs(rng, B, H, T, dk, dv, decay=(0.5, 1.0)):
    q = rng.standard_normal((B, H, T, dk))
    k = rng.standard_normal((B, H, T, dk))
    v = rng.standard_normal((B, H, T, dv))
    log_a = np.log(rng.uniform(*decay, (B, H, T, dk)))
    S0 = rng.standard_normal((B, H, dk, dv))
    return q, k, v, log_a, S0


def test_gla_matches_pathwise_sum():
    """One decay per key dimension, by its paths: o_t[j] = sum_{s<=t} sum_i q_t[i] k_s[i]
    v_s[j] prod_{u=s+1..t} a_u[i] + sum_i q_t[i] prod_{u<=t} a_u[i] S0[i][j], every product
    from its own terms (dk != dv, so a decay on the wrong axis cannot pass)."""
    rng = _rng(21)
    B, H, T, dk, dv = 1, 2, 9, 3, 4
    q, k, v, log_a, S0 = _gla_inputs(rng, B, H, T, dk, dv)
    o, ST = oracle.gla_fwd(q, k, v, log_a, S0)
    a = np.exp(log_a)
    for bi in range(B):
        for h in range(H):
            for t in range(T):
                ref = np.zeros(dv)
                for i in range(dk):
                    ref += q[bi, h, t, i] * np.prod(a[bi, h, : t + 1, i]) * S0[bi, h, i]
                    for s in range(t + 1):
                        ref += q[bi, h, t, i] * k[bi, h, s, i] * np.prod(a[bi, h, s + 1 : t + 1, i]) * v[bi, h, s]
                np.testing.assert_allclose(o[bi, h, t], ref, rtol=1e-12, atol=1e-12)
            ST_ref = np.zeros((dk, dv))
            for i in range(dk):
                ST_ref[i] = np.prod(a[bi, h, :, i]) * S0[bi, h, i]
                for s in range(T):
                    ST_ref[i] += k[bi, h, s, i] * np.prod(a[bi, h, s + 1 :, i]) * v[bi, h, s]
            np.testing.assert_allclose(ST[bi, h], ST_ref, rtol=1e-12, atol=1e-12)


def test_gla_with_one_decay_for_all_dims_is_linear_attention():
    """Every key dimension sharing the step's decay gives the scalar-decay layer; the
    per-dimension decay gradients then sum to the scalar one."""
    rng = _rng(22)
    B, H, T, dk, dv = 2, 1, 13, 4, 3
    q, k, v, _, S0 = _gla_inputs(rng, B, H, T, dk, dv)
    la = np.log(rng.uniform(0.6, 1.0, (B, H, T)))
    lg = np.repeat(la[..., None], dk, axis=-1)
    dO = rng.standard_normal((B, H, T, dv))
    dST = rng.standard_normal((B, H, dk, dv))
    o1, s1 = oracle.gla_fwd(q, k, v, lg, S0)
    o2, s2 = oracle.la_fwd(q, k, v, la, S0)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s1, s2, rtol=1e-12, atol=1e-12)
    g1 = oracle.gla_bwd(q, k, v, lg, S0, dO, dST)
    g2 = oracle.la_bwd(q, k, v, la, S0, dO, dST)
    for x, y in zip((g1[0], g1[1], g1[2], g1[4]), (g2[0], g2[1], g2[2], g2[4])):
        np.testing.assert_allclose(x, y, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(g1[3].sum(-1), g2[3], rtol=1e-11, atol=1e-11)


def test_gla_backward_finite_differences():
    rng = _rng(23)
    B, H, T, dk, dv = 1, 2, 8, 3, 2
    q, k, v, log_a, S0 = _gla_inputs(rng, B, H, T, dk, dv)
    dO = rng.standard_normal((B, H, T, dv))
    dST = rng.standard_normal((B, H, dk, dv))

    def loss():
        o, ST = oracle.gla_fwd(q, k, v, log_a, S0)
        return float(np.sum(dO * o) + np.sum(dST * ST))

    dq, dk_, dv_, dl, dS0 = oracle.gla_bwd(q, k, v, log_a, S0, dO, dST)
    _fd_check(loss, dict(q=q, k=k, v=v, log_a=log_a, S0=S0),
              dict(q=dq, k=dk_, v=dv_, log_a=dl, S0=dS0), sample=40, tol=2e-7)


def test_gla_closed_form_decay_gradient_equals_definition():
    """Per key dimension: sum_{t>=u} q_t[i] dq_t[i] - sum_{s>=u} k_s[i] dk_s[i]
    (+ sum_j dS_T[i][j] S_T[i][j]) equals a_u[i] sum_j Sbar_u[i][j] S_{u-1}[i][j]."""
    rng = _rng(24)
    B, H, T, dk, dv = 2, 2, 40, 4, 3
    q, k, v, log_a, S0 = _gla_inputs(rng, B, H, T, dk, dv, decay=(0.8, 1.0))
    dO = rng.standard_normal((B, H, T, dv))
    dST = rng.standard_normal((B, H, dk, dv))
    _, ST = oracle.gla_fwd(q, k, v, log_a, S0)
    dq, dk_, _, dl, _ = oracle.gla_bwd(q, k, v, log_a, S0, dO, dST)
    dl_cf = oracle.gla_dlog_closed_form(q, k, dq, dk_, dST, ST)
    np.testing.assert_allclose(dl_cf, dl, rtol=1e-10, atol=1e-10)


# ---------------------------------------------------------------- state passing between slices
def test_state_compose_worked_composition():
    """The fold of the pairs (0.5, 1) then (0.5, 0) onto h0 is the single pair (0.25, 0.5)
    applied to h0 ("The scan for one number of state", golden), for several h0 and both
    directions of traversal of the pair list."""
    (a1, b1, a2, b2, A, Bc), = [list(map(float, r)) for r in _golden_rows("composition_example.txt")]
    alphas = np.array([[[a1]], [[a2]]])
    dS = np.array([[[b1]], [[b2]]])
    for h0 in (0.0, 2.0, -3.5):
        out = oracle.state_compose(alphas, dS, np.array([[h0]]), 0, 2, 1)
        assert out[0, 0] == A * h0 + Bc
        # the same list stored in the other order, read from its end
        out_r = oracle.state_compose(alphas[::-1].copy(), dS[::-1].copy(), np.array([[h0]]), 1, 2, -1)
        assert out_r[0, 0] == A * h0 + Bc
    (h0, a1, b1, h1), = [list(map(float, r)) for r in _golden_rows("fold_example.txt")]
    assert oracle.state_compose(np.array([[[a1]]]), np.array([[[b1]]]), np.array([[h0]]), 0, 1, 1)[0, 0] == h1


def test_state_compose_of_slice_pairs_equals_the_sequential_scan():
    """Split a diagonal recurrence into slices; each slice's pair (product of its decays, its
    final state from 0) composed in order onto h0 gives the state entering every later slice --
    the sequential scan's state there ("Splitting one sequence across devices")."""
    rng = np.random.default_rng(11)
    T, D = 57, 5
    a = rng.uniform(0.6, 1.0, (1, T, D))
    b = rng.normal(size=(1, T, D))
    h0 = rng.normal(size=(1, D))
    h, _ = oracle.scan_diag_fwd(a, b, h0)
    bounds = [0, 9, 10, 31, 57]
    alphas, dS = [], []
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        _, hT = oracle.scan_diag_fwd(a[:, lo:hi], b[:, lo:hi])
        alphas.append(np.prod(a[0, lo:hi], axis=0)[:, None])  # one decay per channel (row)
        dS.append(hT[0][:, None])
    alphas = np.stack(alphas)[:, None, :, 0]  # [P, BH=1, A=D]
    dS = np.stack(dS)[:, None, :, 0]          # [P, BH=1, n=D]
    for p in range(1, len(bounds) - 1):
        s_in = oracle.state_compose(alphas, dS, h0, 0, p, 1)
        np.testing.assert_allclose(s_in[0], h[0, bounds[p] - 1], rtol=1e-12, atol=1e-12)


def test_decay_total_closed_forms():
    """exp of the summed log decays: lambda^T for a constant decay, 0 across a reset."""
    T = 37
    lam = np.array([0.9, 0.5, 0.999])
    ld = np.broadcast_to(np.log(lam)[None, None, :], (2, T, 3)).copy()
    np.testing.assert_allclose(oracle.decay_total(ld), np.broadcast_to(lam ** T, (2, 3)), rtol=1e-12)
    ld[1, 20, 1] = -np.inf
    out = oracle.decay_total(ld)
    assert out[1, 1] == 0.0 and out[0, 1] > 0.0
