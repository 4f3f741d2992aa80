"""Pins of the oracle's Falcon-3 / 3A window, each against something other
than the oracle's own token loop.

Page "Fast Weight Attention for Continual Learning", §4.2: Falcon-3 takes one
gradient step on the average loss of the last W causal pairs, with the step
eta_t = beta_t / (mu_t + lambda_t + eps) set by mu_t, the largest eigenvalue
of the window-average key covariance; §4.3: Falcon-3A writes the targets
instead of the residuals.  The readings pinned here: the window holds the
pairs that exist (the first token's shifted pair does not), B_t counts them,
eta_t = 0 when there are none, and a carried window continues a sequence.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(20261210)


def rand_inputs(nc=2, T=11, dk=6, dv=5, s0=True, beta=(0.1, 1.5), lam_hi=0.1):
    q = RNG.standard_normal((nc, T, dk))
    k = RNG.standard_normal((nc, T, dk))
    v = RNG.standard_normal((nc, T, dv))
    b = RNG.uniform(*beta, (nc, T))
    lam = RNG.uniform(0.0, lam_hi, (nc, T))
    S0 = 0.3 * RNG.standard_normal((nc, dk, dv)) if s0 else None
    return q, k, v, b, lam, S0


def window_keys(k, t, W, same_pair=False, k_init=None):
    """Keys of the pairs that exist in token t's window, for one chain."""
    xs = []
    for m in range(t - W + 1, t + 1):
        if m < 0:
            continue
        if same_pair:
            xs.append(k[m])
        elif m > 0:
            xs.append(k[m - 1])
        elif k_init is not None:
            xs.append(k_init)
    return np.array(xs)


# ------------------------------------------------------------ reductions

@pytest.mark.parametrize("rbw,same_pair", [(False, False), (True, False), (False, True)])
@pytest.mark.parametrize("inner", [False, True])
def test_window_of_one_is_falcon1(inner, rbw, same_pair):
    # W = 1: the window average is the instantaneous loss and lambda_max of
    # x x^T is |x|^2, so Falcon-3 (3A) is Falcon-1 (1A) (pinned on its own)
    q, k, v, beta, lam, S0 = rand_inputs()
    ki = RNG.standard_normal(k[:, 0].shape)
    o1, S1 = oracle.falcon1(q, k, v, beta, lam, S0, k_init=ki, inner=inner, rbw=rbw,
                            same_pair=same_pair)
    o3, S3, _ = oracle.falcon3(q, k, v, beta, lam, 1, S0, k_init=ki, inner=inner, rbw=rbw,
                               same_pair=same_pair)
    np.testing.assert_allclose(o3, o1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S3, S1, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("W", [2, 3, 5, 8])
def test_mu_is_lambda_max_of_the_window_covariance(W):
    # mu_t against numpy's symmetric eigensolver on the d_k x d_k covariance
    # (1/B_t) sum x_j x_j^T built from the definition (not the Gram form)
    q, k, v, beta, lam, S0 = rand_inputs(nc=1, T=13, dk=7)
    _, _, _, mu = oracle.falcon3(q, k, v, beta, lam, W, S0, want_mu=True)
    for t in range(13):
        X = window_keys(k[0], t, W)
        if len(X) == 0:
            assert mu[0, t] == 0.0
            continue
        C = X.T @ X / len(X)
        assert mu[0, t] == pytest.approx(np.linalg.eigvalsh(C)[-1], rel=1e-12, abs=1e-12)


def test_mu_of_orthogonal_keys_is_the_largest_mean_energy():
    # mutually orthogonal window keys: the covariance is diagonal in their
    # directions, so mu_t = max_j |x_j|^2 / B_t
    dk, W, T = 8, 4, 9
    basis = np.linalg.qr(RNG.standard_normal((dk, dk)))[0]
    scale = RNG.uniform(0.5, 3.0, T)
    k = np.stack([scale[t] * basis[:, t % dk] for t in range(T)])[None]   # k_t along e_{t mod 8}
    q = RNG.standard_normal((1, T, dk))
    v = RNG.standard_normal((1, T, 3))
    beta, lam = np.full((1, T), 0.5), np.zeros((1, T))
    _, _, _, mu = oracle.falcon3(q, k, v, beta, lam, W, want_mu=True)
    for t in range(1, T):
        js = [m - 1 for m in range(max(1, t - W + 1), t + 1)]
        assert mu[0, t] == pytest.approx(max(scale[j] ** 2 for j in js) / len(js), rel=1e-13)


def test_mu_with_repeated_keys():
    # a window of identical keys is rank one: mu_t = |x|^2 exactly
    dk, T, W = 5, 7, 4
    x = RNG.standard_normal(dk)
    k = np.tile(x, (1, T, 1))
    _, _, _, mu = oracle.falcon3(RNG.standard_normal((1, T, dk)), k,
                                 RNG.standard_normal((1, T, 2)), np.ones((1, T)),
                                 np.zeros((1, T)), W, want_mu=True)
    np.testing.assert_allclose(mu[0, 1:], np.dot(x, x), rtol=1e-13)


# ------------------------------------------------------------ closed forms

@pytest.mark.parametrize("W", [2, 3, 6])
def test_collinear_keys_give_the_window_least_squares_fit(W):
    # keys c_j u along one unit direction, beta = 1, lambda = eps = 0: the step
    # lands on the least-squares fit of the window along u,
    #   S_t^T u = sum_j c_j y_j / sum_j c_j^2,
    # and leaves S^T w unchanged for every w orthogonal to u
    dk, dv, T = 6, 4, 10
    u = RNG.standard_normal(dk)
    u /= np.linalg.norm(u)
    c = RNG.uniform(0.5, 2.0, T) * RNG.choice([-1.0, 1.0], T)
    k = (c[:, None] * u[None, :])[None]
    v = RNG.standard_normal((1, T, dv))
    S0 = RNG.standard_normal((1, dk, dv))
    w = RNG.standard_normal(dk)
    w -= np.dot(w, u) * u
    S = S0[0]
    for t in range(T):
        _, St, _ = oracle.falcon3(RNG.standard_normal((1, t + 1, dk)), k[:, :t + 1],
                                  v[:, :t + 1], np.ones((1, t + 1)), np.zeros((1, t + 1)), W,
                                  S0, eps=0.0)
        js = [m for m in range(max(1, t - W + 1), t + 1)]   # pairs (c_{m-1} u, v_m)
        if not js:
            np.testing.assert_allclose(St[0], S0[0], rtol=0, atol=0)
            continue
        fit = sum(c[m - 1] * v[0, m] for m in js) / sum(c[m - 1] ** 2 for m in js)
        np.testing.assert_allclose(St[0].T @ u, fit, rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(St[0].T @ w, S0[0].T @ w, rtol=1e-11, atol=1e-11)


def test_inner_product_collinear_keys_add_the_scaled_window_correlation():
    # Falcon-3A with keys c_j u, lambda = 0: mu = mean c_j^2, so one write adds
    # beta u (sum_j c_j y_j / sum_j c_j^2)^T to S
    dk, dv, T, W = 5, 3, 6, 3
    u = RNG.standard_normal(dk)
    u /= np.linalg.norm(u)
    c = RNG.uniform(0.5, 2.0, T)
    k = (c[:, None] * u[None, :])[None]
    v = RNG.standard_normal((1, T, dv))
    beta = RNG.uniform(0.2, 1.0, (1, T))
    S0 = RNG.standard_normal((1, dk, dv))
    _, S5, _ = oracle.falcon3(RNG.standard_normal((1, 5, dk)), k[:, :5], v[:, :5],
                              beta[:, :5], np.zeros((1, 5)), W, S0, eps=0.0, inner=True)
    _, S6, _ = oracle.falcon3(RNG.standard_normal((1, 6, dk)), k, v, beta, np.zeros((1, 6)),
                              W, S0, eps=0.0, inner=True)
    js = [3, 4, 5]
    add = beta[0, 5] * np.outer(u, sum(c[m - 1] * v[0, m] for m in js)
                                / sum(c[m - 1] ** 2 for m in js))
    np.testing.assert_allclose(S6[0], S5[0] + add, rtol=1e-11, atol=1e-11)


def test_fixed_point_when_the_window_is_fitted():
    # lambda = 0 and every window target equals S^T x_j: zero gradient, no change
    dk, dv, T, W = 6, 4, 8, 4
    S0 = RNG.standard_normal((1, dk, dv))
    k = RNG.standard_normal((1, T, dk))
    v = np.zeros((1, T, dv))
    v[0, 1:] = k[0, :-1] @ S0[0]                  # y_t = S0^T x_t with x_t = k_{t-1}
    _, S, _ = oracle.falcon3(RNG.standard_normal((1, T, dk)), k, v,
                             RNG.uniform(0.1, 1.9, (1, T)), np.zeros((1, T)), W, S0)
    np.testing.assert_allclose(S, S0, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ descent

@pytest.mark.parametrize("W", [2, 4, 8])
def test_each_write_decreases_the_window_loss(W):
    # the write is a gradient step on
    #   L(S) = 1/(2 B_t) sum_j |S^T x_j - y_j|^2 + lambda_t/2 |S|_F^2,
    # whose smoothness constant is mu_t + lambda_t; with beta < 2 the step is
    # below 2/(mu_t + lambda_t), so L strictly decreases (the window analogue
    # of the single-pair descent lemma).  beta near 2 makes an underestimated
    # mu overshoot.
    dk, dv, T = 6, 4, 16
    q, k, v, beta, lam, S0 = rand_inputs(nc=1, T=T, dk=dk, dv=dv, beta=(1.7, 1.99),
                                         lam_hi=0.3)
    k *= np.exp(RNG.standard_normal((1, T, 1)))    # keys of mixed norms
    S = S0[0]
    for t in range(T):
        _, St, _ = oracle.falcon3(q[:, :t + 1], k[:, :t + 1], v[:, :t + 1], beta[:, :t + 1],
                                  lam[:, :t + 1], W, S0)
        X = window_keys(k[0], t, W)
        if len(X) == 0:
            continue
        Y = np.array([v[0, m] for m in range(max(1, t - W + 1), t + 1)])

        def loss(M):
            return (0.5 / len(X)) * np.sum((X @ M - Y) ** 2) + 0.5 * lam[0, t] * np.sum(M * M)

        _, Sp, _ = oracle.falcon3(q[:, :t], k[:, :t], v[:, :t], beta[:, :t], lam[:, :t], W,
                                  S0) if t > 0 else (None, S0, None)
        assert loss(St[0]) < loss(Sp[0])


# ------------------------------------------------------------ boundary and carry

def test_first_token_is_no_write_and_second_is_a_single_pair():
    # x_1 = 0 is no pair: token 1 leaves S0; token 2's window holds one pair,
    # so it is the Falcon-1 write of that pair
    q, k, v, beta, lam, S0 = rand_inputs(T=2)
    o3, S3, win = oracle.falcon3(q[:, :1], k[:, :1], v[:, :1], beta[:, :1], lam[:, :1], 4, S0)
    np.testing.assert_array_equal(S3, S0)
    np.testing.assert_allclose(o3[:, 0], np.einsum("cij,ci->cj", S0, q[:, 0]), rtol=1e-13)
    assert list(win[2]) == [0, 0]
    o3, S3, _ = oracle.falcon3(q, k, v, beta, lam, 4, S0)
    o1, S1 = oracle.falcon1(q, k, v, beta, lam, S0)
    np.testing.assert_allclose(S3, S1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o3, o1, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("W", [2, 4, 7])
@pytest.mark.parametrize("inner,same_pair,rbw", [(False, False, False), (True, False, False),
                                                 (False, True, False), (False, False, True)])
def test_carried_window_continues_a_prefill(W, inner, same_pair, rbw):
    # prefill of T tokens == prefill of T1 tokens, then of the rest with the
    # state, the last key and the window carried over (T1 < W included)
    T = 12
    q, k, v, beta, lam, S0 = rand_inputs(T=T)
    full = oracle.falcon3(q, k, v, beta, lam, W, S0, inner=inner, same_pair=same_pair,
                          rbw=rbw)
    for T1 in (1, 2, W - 1, 7):
        a = oracle.falcon3(q[:, :T1], k[:, :T1], v[:, :T1], beta[:, :T1], lam[:, :T1], W, S0,
                           inner=inner, same_pair=same_pair, rbw=rbw)
        b = oracle.falcon3(q[:, T1:], k[:, T1:], v[:, T1:], beta[:, T1:], lam[:, T1:], W,
                           a[1], k_init=k[:, T1 - 1], win=a[2], inner=inner,
                           same_pair=same_pair, rbw=rbw)
        np.testing.assert_allclose(np.concatenate([a[0], b[0]], axis=1), full[0], rtol=1e-12,
                                   atol=1e-12)
        np.testing.assert_allclose(b[1], full[1], rtol=1e-12, atol=1e-12)
        for x, y in zip(b[2], full[2]):
            np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("inner,rbw", [(False, False), (True, False), (False, True)])
def test_steps_continue_a_prefill(inner, rbw):
    # a prefill of T1 tokens followed by one step per further token, each with
    # the previous token's key and the window carried, equals the whole prefill
    T, T1, W = 10, 3, 4
    q, k, v, beta, lam, S0 = rand_inputs(T=T)
    o_full, S_full, win_full = oracle.falcon3(q, k, v, beta, lam, W, S0, inner=inner, rbw=rbw)
    o, S, win = oracle.falcon3(q[:, :T1], k[:, :T1], v[:, :T1], beta[:, :T1], lam[:, :T1], W,
                               S0, inner=inner, rbw=rbw)
    outs = [o]
    for t in range(T1, T):
        ot, S, win = oracle.step3(q[:, t], k[:, t - 1], v[:, t], beta[:, t], lam[:, t], S, W,
                                  win=win, inner=inner, rbw=rbw)
        outs.append(ot[:, None])
    np.testing.assert_allclose(np.concatenate(outs, axis=1), o_full, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S, S_full, rtol=1e-12, atol=1e-12)
    for x, y in zip(win, win_full):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-12)


def test_window_carry_layout():
    # the carry holds the newest W-1 pairs oldest first, phi applied to the
    # key, and counts only pairs that exist
    q, k, v, beta, lam, S0 = rand_inputs(nc=1, T=6)
    _, _, (x, y, n) = oracle.falcon3(q, k, v, beta, lam, 4, S0, phi="elu1")
    assert n[0] == 3
    phi = np.where(k[0] > 0, k[0] + 1.0, np.exp(k[0]))
    np.testing.assert_array_equal(x[0], phi[2:5])     # pairs 3..5 hold keys 2..4
    np.testing.assert_array_equal(y[0], v[0, 3:6])
    _, _, (x, y, n) = oracle.falcon3(q[:, :2], k[:, :2], v[:, :2], beta[:, :2], lam[:, :2], 4)
    assert n[0] == 1                                   # pair 0 does not exist
    np.testing.assert_array_equal(x[0, :2], 0.0)
    np.testing.assert_array_equal(x[0, 2], k[0, 0])
