"""The chunk form of the per-channel step (Falcon-2 / 2A) that the CUDA
kernel evaluates, written densely in fp64 numpy and checked against the
sequential oracle.

A check of the derivation the kernel is built on, not an oracle.  The "Fast
Weight Attention for Continual Learning" paper reading, §4.2 and §4.4: the
squared error is separable by value dimension, so each value channel j takes
its own step eta_{t,j} = beta_{t,j} / (|x_t|^2 + lambda_t + eps) with a shared
residual and feature; the chunk Gram matrix is shared by every channel and
only the triangular system is modulated per channel.  Our derivation, for one
chunk starting from state S0 and one channel j (chunk-local t, s; gamma_t =
1 - eta_t lambda_t, D[t,s] = prod_{i=s+1..t} gamma_i, G_t = prod_{i<=t}
gamma_i, Gm_t = G_{t-1}, A = X X^T, B = Q X^T, U = X S0[:, j], V = Q S0[:, j]):

  r_t = y_t - Gm_t U_t - sum_{s<t} D[t-1,s] eta_s A[t,s] r_s      (residuals;
        Falcon-2A writes y: r_t = y_t)
  o_t = G_t V_t + sum_{s<=t} D[t,s] eta_s B[t,s] r_s               (read after
        the write; read before: Gm_t V_t + sum_{s<t} D[t-1,s] eta_s B[t,s] r_s)
  S_C[:, j] = G_{C-1} S0[:, j] + X^T (D[C-1, .] eta r)

The sums over earlier tokens are evaluated block-factored, as the kernel does:
in blocks of NB tokens, D[t-1, s] for s in an earlier block a is P[t-1] (the
in-block prefix product of t-1's block) times the totals of the blocks in
between times the exclusive in-block suffix product of s.  A running vector
zhat (rescaled by each finished block's total) makes every cross-block sum a
plain dot product with A's or B's row; the last zhat is D[C-1, s] eta_s r_s,
the state update's weights.  No decay product is ever divided.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(2026)


def chunked_falcon2(q, k, v, beta, lam, S0, eps, C, NB, inner=False, rbw=False,
                    same_pair=False, k_init=None):
    T, dk = q.shape
    dv = v.shape[1]
    if same_pair:
        X = k.copy()
    else:
        first = np.zeros((1, dk)) if k_init is None else k_init[None, :]
        X = np.vstack([first, k[:-1]])
    n = np.sum(X * X, axis=1)
    eta = beta / (n + lam + eps)[:, None]            # [T, dv]
    if not same_pair and k_init is None:
        eta[0, :] = 0.0
    gam = 1.0 - eta * lam[:, None]
    S = S0.copy()
    O = np.zeros((T, dv))
    for c0 in range(0, T, C):
        m = min(C, T - c0)
        Xc, Qc, Yc = X[c0:c0 + m], q[c0:c0 + m], v[c0:c0 + m]
        ec, gc = eta[c0:c0 + m], gam[c0:c0 + m]
        A, B = Xc @ Xc.T, Qc @ Xc.T
        U, V = Xc @ S, Qc @ S
        G = np.cumprod(gc, axis=0)
        Gm = np.vstack([np.ones((1, dv)), G[:-1]])
        zhat = np.zeros((m, dv))
        r = np.zeros((m, dv))
        for b0 in range(0, m, NB):
            b1 = min(b0 + NB, m)
            P = np.cumprod(gc[b0:b1], axis=0)          # in-block inclusive prefix
            for t in range(b0, b1):
                tl = t - b0
                ct = P[tl - 1] if tl >= 1 else np.ones(dv)
                HA = A[t, :b0] @ zhat[:b0]
                HB = B[t, :b0] @ zhat[:b0]
                d = np.ones(dv)
                inA = np.zeros(dv)
                inB = np.zeros(dv)
                for s in range(t - 1, b0 - 1, -1):
                    zs = ec[s] * r[s]
                    inA += d * A[t, s] * zs
                    inB += d * B[t, s] * zs
                    d = d * gc[s]
                r[t] = Yc[t] if inner else Yc[t] - Gm[t] * U[t] - ct * HA - inA
                if rbw:
                    O[c0 + t] = Gm[t] * V[t] + ct * HB + inB
                else:
                    O[c0 + t] = G[t] * V[t] + gc[t] * (ct * HB + inB) + ec[t] * B[t, t] * r[t]
            # the block is done: earlier weights take its total decay, its own
            # tokens their suffix products to the block's end
            zhat[:b0] *= np.prod(gc[b0:b1], axis=0)
            suf = np.ones((b1 - b0, dv))
            for s in range(b1 - 2, b0 - 1, -1):
                suf[s - b0] = suf[s - b0 + 1] * gc[s + 1]
            zhat[b0:b1] = suf * ec[b0:b1] * r[b0:b1]
        S = G[m - 1] * S + Xc.T @ zhat
    return O, S


def _case(T, dk, dv, unit=False, beta_hi=1.99):
    q = RNG.standard_normal((T, dk))
    v = RNG.standard_normal((T, dv))
    k = RNG.standard_normal((T, dk))
    k = k / np.linalg.norm(k, axis=1, keepdims=True) if unit else k * np.exp(RNG.standard_normal((T, 1)))
    beta = RNG.uniform(0.1, beta_hi, (T, dv))
    lam = RNG.uniform(0, 0.5, T)
    S0 = RNG.standard_normal((dk, dv))
    return q, k, v, beta, lam, S0


def _check(o, S, o_ref, S_ref):
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-9 * max(1.0, np.abs(o_ref).max()))
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-9 * max(1.0, np.abs(S_ref).max()))


@pytest.mark.parametrize("C,NB", [(1, 1), (8, 4), (16, 8), (64, 8), (64, 16), (20, 8)])
@pytest.mark.parametrize("T", [1, 2, 37, 64, 130])
def test_chan_chunk_form_matches_oracle(C, NB, T):
    q, k, v, beta, lam, S0 = _case(T, 8, 6)
    o_ref, S_ref = oracle.falcon2(q, k, v, beta, lam, S0, eps=1e-6)
    o, S = chunked_falcon2(q, k, v, beta, lam, S0, 1e-6, C, NB)
    _check(o, S, o_ref, S_ref)


@pytest.mark.parametrize("inner,rbw,same_pair,kinit", [(True, False, False, False),
                                                       (False, True, False, False),
                                                       (True, True, True, False),
                                                       (False, False, True, False),
                                                       (False, False, False, True),
                                                       (True, True, False, True)])
def test_chan_chunk_form_variants(inner, rbw, same_pair, kinit):
    T = 75
    q, k, v, beta, lam, S0 = _case(T, 8, 5)
    ki = RNG.standard_normal(8) if kinit else None
    o_ref, S_ref = oracle.falcon2(q, k, v, beta, lam, S0, k_init=ki, eps=1e-6, inner=inner,
                                  rbw=rbw, same_pair=same_pair)
    o, S = chunked_falcon2(q, k, v, beta, lam, S0, 1e-6, 64, 8, inner=inner, rbw=rbw,
                           same_pair=same_pair, k_init=ki)
    _check(o, S, o_ref, S_ref)


def test_chan_chunk_form_with_nonpositive_decay():
    """gamma <= 0 on some (token, channel) pairs: the block factorisation uses
    only products, so the form stays exact."""
    T, dk, dv = 50, 8, 4
    q, k, v, beta, lam, S0 = _case(T, dk, dv)
    k[7] *= 1e-3
    k[30] *= 1e-3
    lam[8] = lam[31] = 0.4
    beta[8] = beta[31] = 1.95
    X = np.vstack([np.zeros((1, dk)), k[:-1]])
    eta = beta / (np.sum(X * X, 1) + lam + 1e-6)[:, None]
    assert (1 - eta[1:] * lam[1:, None]).min() <= 0.0
    o_ref, S_ref = oracle.falcon2(q, k, v, beta, lam, S0, eps=1e-6)
    o, S = chunked_falcon2(q, k, v, beta, lam, S0, 1e-6, 16, 8)
    _check(o, S, o_ref, S_ref)
