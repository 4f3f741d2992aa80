"""Pins for the fp64 oracle: each test checks the oracle against something the
pages or the mathematics fix, not against a retyped copy of its own formula.

Passages (page title, section):
  FW  = "Fast Weight Attention for Continual Learning" paper reading
        §3.2 (ridge loss and its normalised step), §4.1 (shifted pair and the
        first-token boundary), §4.2 (Falcon-1, Lemma 3.1, NLMS reduction).
  BLOG = "Attention is also an FFN" blog, §2.1 (linear attention), §4.1
        (elu+1 feature map), §5.2 (check tiny cases by hand).
  MEM = "You could have invented transformers from memory", outer-product
        store: orthonormal keys give interference-free recall.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.golden_io import load

RNG = np.random.default_rng(12345)


def rand(*shape):
    return RNG.standard_normal(shape)


def unit_rows(a):
    return a / np.linalg.norm(a, axis=-1, keepdims=True)


# --------------------------------------------------------------------------
# hand-worked golden cases (BLOG §5.2 practice; rule from FW §3.2/§4.1)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["falcon1_tiny_dk2_dv1.txt", "falcon1_tiny_dk2_dv2.txt"])
def test_golden_falcon1(name):
    g = load(name)
    o, S = oracle.falcon1(g["q"], g["k"], g["v"], g["beta"][0], g["lam"][0], S0=g["S0"],
                          eps=float(g["eps"][0, 0]))
    np.testing.assert_allclose(o, g["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(S, g["S_T"], rtol=0, atol=1e-12)


def test_golden_linattn():
    g = load("linattn_tiny.txt")
    for phi in ("identity", "elu1"):
        o, S = oracle.linattn(g["q"], g["k"], g["v"], phi=phi)
        np.testing.assert_allclose(o, g["o_" + phi], rtol=0, atol=1e-12)
        np.testing.assert_allclose(S, g["S_T_" + phi], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Falcon-1 single-write properties
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dk,dv", [(4, 3), (8, 8), (5, 9)])
def test_exact_recall(dk, dv):
    """lambda = eps = 0, beta = 1: after the write at t, S_t^T x_t = y_t
    exactly (FW §4.2: the normalised step with beta = 1 solves the pair)."""
    T = 7
    q, k, v = rand(T, dk), rand(T, dk), rand(T, dv)
    S0 = rand(dk, dv)
    beta = np.ones(T)
    lam = np.zeros(T)
    for Tp in range(2, T + 1):
        _, S = oracle.falcon1(q[:Tp], k[:Tp], v[:Tp], beta[:Tp], lam[:Tp], S0=S0, eps=0.0)
        x = k[Tp - 2]                         # x_t = k_{t-1} (FW §4.1)
        np.testing.assert_allclose(S.T @ x, v[Tp - 1], rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("dk,dv", [(6, 4), (16, 16)])
def test_textbook_nlms(dk, dv):
    """lambda = eps = 0: every value column is a textbook NLMS filter
    w <- w + mu e x / |x|^2, e = d - w.x, on the shifted pairs (FW §4.2)."""
    T = 40
    q, k, v = rand(T, dk), rand(T, dk), rand(T, dv)
    S0 = rand(dk, dv)
    mu = RNG.uniform(0.1, 1.9, T)
    o, S = oracle.falcon1(q, k, v, mu, np.zeros(T), S0=S0, eps=0.0)
    W = S0.copy()                            # column j = filter j
    o_ref = np.zeros((T, dv))
    for t in range(T):
        if t > 0:
            xin = k[t - 1]
            for j in range(dv):
                e = v[t, j] - np.dot(W[:, j], xin)
                W[:, j] = W[:, j] + mu[t] * e * xin / np.dot(xin, xin)
        for j in range(dv):
            o_ref[t, j] = np.dot(W[:, j], q[t])
    np.testing.assert_allclose(S, W, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("lam_val,beta_val", [(0.5, 1.0), (2.0, 0.7), (0.05, 1.5)])
def test_ridge_fixed_point(lam_val, beta_val):
    """Repeating one pair (x, y) drives S to the minimiser of the ridge loss
    1/2|S^T x - y|^2 + lambda/2 |S|_F^2 of FW §3.2, i.e. x y^T / (|x|^2 + lambda),
    from any start state (the loss is strongly convex for lambda > 0)."""
    dk, dv, T = 5, 3, 4000
    x = rand(dk) * 0.8
    y = rand(dv)
    k = np.tile(x, (T, 1))
    v = np.tile(y, (T, 1))
    S0 = rand(dk, dv)
    _, S = oracle.falcon1(rand(T, dk), k, v, np.full(T, beta_val), np.full(T, lam_val),
                          S0=S0, eps=0.0)
    S_star = np.outer(x, y) / (x @ x + lam_val)
    np.testing.assert_allclose(S, S_star, rtol=0, atol=1e-10)


def test_boundary_first_token_is_noop():
    """x_1 := 0, eta_1 := 0 (FW §4.1): the first write leaves S0 unchanged even
    with a large beta/lambda, and o_1 = S0^T q_1."""
    dk, dv = 6, 5
    q, k, v = rand(1, dk), rand(1, dk), rand(1, dv)
    S0 = rand(dk, dv)
    o, S = oracle.falcon1(q, k, v, np.array([1.9]), np.array([3.0]), S0=S0)
    np.testing.assert_array_equal(S, S0)
    np.testing.assert_allclose(o[0], S0.T @ q[0], rtol=1e-14, atol=1e-14)


def test_k_init_continues_a_prefill():
    """Splitting a sequence in two prefills, the second started with
    k_init = last key of the first, reproduces the single prefill."""
    dk, dv, T, cut = 7, 4, 30, 13
    q, k, v = rand(T, dk), rand(T, dk), rand(T, dv)
    beta, lam = RNG.uniform(0.1, 1.5, T), RNG.uniform(0, 0.1, T)
    S0 = rand(dk, dv) * 0.1
    o, S = oracle.falcon1(q, k, v, beta, lam, S0=S0)
    o1, S1 = oracle.falcon1(q[:cut], k[:cut], v[:cut], beta[:cut], lam[:cut], S0=S0)
    o2, S2 = oracle.falcon1(q[cut:], k[cut:], v[cut:], beta[cut:], lam[cut:], S0=S1,
                            k_init=k[cut - 1])
    np.testing.assert_allclose(np.concatenate([o1, o2]), o, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S2, S, rtol=1e-12, atol=1e-12)


def test_orthonormal_keys_interference_free():
    """MEM: orthonormal keys give zero interference.  With lambda = 0, later
    writes along orthogonal keys do not disturb earlier ones, so for every
    stored key S_T^T x_j = (1 - b_j) S0^T x_j + b_j y_j, b_j = beta_j n/(n+eps);
    with eps = 0 and beta = 1 that is exactly y_j."""
    dk, dv = 12, 7
    m = dk                                   # store a full basis
    Qb, _ = np.linalg.qr(rand(dk, dk))
    keys = Qb.T[:m]                          # orthonormal rows
    T = m + 1
    k = np.vstack([keys, rand(1, dk)])       # k_1..k_m feed x_2..x_{m+1}
    v = rand(T, dv)
    S0 = rand(dk, dv)
    for beta_vals, eps in ((np.ones(T), 0.0), (RNG.uniform(0.2, 1.8, T), 1e-3)):
        _, S = oracle.falcon1(rand(T, dk), k, v, beta_vals, np.zeros(T), S0=S0, eps=eps)
        for j in range(m):
            x = keys[j]
            n = x @ x
            b = beta_vals[j + 1] * n / (n + eps)
            want = (1 - b) * (S0.T @ x) + b * v[j + 1]
            np.testing.assert_allclose(S.T @ x, want, rtol=1e-11, atol=1e-11)


# --------------------------------------------------------------------------
# per-step properties through the decode-step oracle
# --------------------------------------------------------------------------

def _ridge_loss(S, x, y, lam):
    return 0.5 * np.sum((S.T @ x - y) ** 2) + 0.5 * lam * np.sum(S * S)


def test_lemma31_each_write_decreases_its_loss():
    """FW §4.2, Lemma 3.1: with beta in (0,2) the normalised step strictly
    decreases the instantaneous ridge loss (it is one gradient step on an
    (|x|^2 + lambda)-smooth quadratic with step below 2/(|x|^2 + lambda))."""
    dk, dv = 16, 8
    S = rand(dk, dv)
    for _ in range(300):
        x = rand(dk) * np.exp(RNG.standard_normal())
        y = rand(dv)
        beta = RNG.uniform(0.01, 1.99)
        lam = RNG.uniform(0, 0.5)
        before = _ridge_loss(S, x, y, lam)
        _, S_new = oracle.step(rand(dk), x, y, beta, lam, S, eps=1e-6)
        after = _ridge_loss(S_new, x, y, lam)
        assert after < before
        S = S_new


def test_step_norm_bound():
    """|S_t|_F <= |S_{t-1}|_F + eta |x| |y|: the homogeneous part
    gamma I - eta x x^T has spectral norm <= 1 for beta in [0,2)
    (eigenvalues gamma and gamma - eta|x|^2 = 1 - eta(lambda + |x|^2))."""
    dk, dv = 32, 16
    S = np.zeros((dk, dv))
    for _ in range(500):
        x = unit_rows(rand(dk)) * np.exp(RNG.standard_normal())
        y = rand(dv)
        beta = RNG.uniform(1.5, 1.99)
        lam = RNG.uniform(0, 0.01)
        eta = beta / (x @ x + lam + 1e-6)
        _, S_new = oracle.step(rand(dk), x, y, beta, lam, S, eps=1e-6)
        assert (np.linalg.norm(S_new) <= np.linalg.norm(S) + eta * np.linalg.norm(x)
                * np.linalg.norm(y) * (1 + 1e-12) + 1e-12)
        S = S_new


def test_step_read_is_read_after_write():
    """A step returns o = S_new^T q (FW §1.4 read after write) with S_new the
    state the same call returns."""
    dk, dv = 9, 6
    S = rand(dk, dv)
    q, x, y = rand(dk), rand(dk), rand(dv)
    o, S_new = oracle.step(q, x, y, 0.8, 0.03, S)
    np.testing.assert_allclose(o, S_new.T @ q, rtol=1e-13, atol=1e-13)


def test_prefill_equals_steps():
    """A prefill equals T decode steps when step 1 gets beta = 0 (an empty
    first write, FW §4.1) and step t gets k_prev = k_{t-1}."""
    dk, dv, T = 8, 5, 25
    q, k, v = rand(T, dk), rand(T, dk), rand(T, dv)
    beta, lam = RNG.uniform(0.1, 1.9, T), RNG.uniform(0, 0.2, T)
    S0 = rand(dk, dv)
    o, S = oracle.falcon1(q, k, v, beta, lam, S0=S0)
    St = S0
    for t in range(T):
        kp = k[t - 1] if t > 0 else np.zeros(dk)
        b = beta[t] if t > 0 else 0.0
        ot, St = oracle.step(q[t], kp, v[t], b, lam[t], St)
        np.testing.assert_allclose(ot, o[t], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(St, S, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# linear attention
# --------------------------------------------------------------------------

@pytest.mark.parametrize("phi", ["identity", "elu1"])
def test_linattn_masked_quadratic_form(phi):
    """BLOG §2.1/§3.1: O = tril(phi(Q) phi(K)^T) V (+ phi(Q) S0) and
    S_T = S0 + phi(K)^T V, the parallel form of the recurrence."""
    B, H, T, dk, dv = 2, 3, 50, 8, 6
    q, k, v = rand(B, H, T, dk), rand(B, H, T, dk), rand(B, H, T, dv)
    S0 = rand(B, H, dk, dv)
    fq = torch.nn.functional.elu(torch.from_numpy(q)).numpy() + 1 if phi == "elu1" else q
    fk = torch.nn.functional.elu(torch.from_numpy(k)).numpy() + 1 if phi == "elu1" else k
    o, S = oracle.linattn(q, k, v, S0=S0, phi=phi)
    mask = np.tril(np.ones((T, T)))
    o_ref = (fq @ np.swapaxes(fk, -1, -2) * mask) @ v + fq @ S0
    S_ref = S0 + np.swapaxes(fk, -1, -2) @ v
    np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(S, S_ref, rtol=1e-11, atol=1e-11)


def test_linattn_step_matches_quadratic_form():
    """Decode steps in linear-attention mode accumulate S += phi(k) v^T and
    read phi(q)^T S (BLOG §4.1 forward_step), matching the masked form."""
    dk, dv, T = 6, 4, 12
    q, k, v = rand(T, dk), rand(T, dk), rand(T, dv)
    fq = torch.nn.functional.elu(torch.from_numpy(q)).numpy() + 1
    fk = torch.nn.functional.elu(torch.from_numpy(k)).numpy() + 1
    o_ref = (fq @ fk.T * np.tril(np.ones((T, T)))) @ v
    S = np.zeros((dk, dv))
    for t in range(T):
        ot, S = oracle.step(q[t], k[t], v[t], None, None, S, mode="linattn", phi="elu1")
        np.testing.assert_allclose(ot, o_ref[t], rtol=1e-12, atol=1e-12)


def test_elu1_feature_map_on_falcon_keys():
    """phi = elu+1 enters Falcon-1 through the key only: a prefill with phi
    equals an identity-phi prefill on keys mapped by torch's elu + 1."""
    dk, dv, T = 6, 5, 20
    q, k, v = rand(T, dk), rand(T, dk), rand(T, dv)
    beta, lam = RNG.uniform(0.1, 1.5, T), RNG.uniform(0, 0.1, T)
    fk = torch.nn.functional.elu(torch.from_numpy(k)).numpy() + 1
    o1, S1 = oracle.falcon1(q, k, v, beta, lam, phi="elu1")
    o2, S2 = oracle.falcon1(q, fk, v, beta, lam, phi="identity")
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S1, S2, rtol=1e-12, atol=1e-12)


def test_falcon1_beta0_is_identity_map():
    """beta = 0 everywhere means eta = 0, gamma = 1: the state never moves and
    o_t = S0^T q_t for all t."""
    dk, dv, T = 5, 4, 9
    q, k, v = rand(T, dk), rand(T, dk), rand(T, dv)
    S0 = rand(dk, dv)
    o, S = oracle.falcon1(q, k, v, np.zeros(T), RNG.uniform(0, 1, T), S0=S0)
    np.testing.assert_array_equal(S, S0)
    np.testing.assert_allclose(o, q @ S0, rtol=1e-13, atol=1e-13)


def test_threads_do_not_change_results():
    B, H, T, d = 3, 2, 40, 8
    q, k, v = rand(B, H, T, d), rand(B, H, T, d), rand(B, H, T, d)
    beta, lam = RNG.uniform(0.1, 1.5, (B, H, T)), RNG.uniform(0, 0.1, (B, H, T))
    a = oracle.falcon1(q, k, v, beta, lam, nthreads=1)
    b = oracle.falcon1(q, k, v, beta, lam, nthreads=4)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
