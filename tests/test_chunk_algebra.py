"""The chunk-parallel (UT / WY) form that the CUDA prefill kernel evaluates,
written densely in fp64 numpy and checked against the sequential oracle.

This is a check of the derivation the kernel is built on, not an oracle: the
"Fast Weight Attention for Continual Learning" paper reading, §4.4, says that
Falcon-1's chain of rank-one edits inside a chunk collapses (WY representation)
into one triangular system -- intra-chunk parallel solve, short inter-chunk
recurrence, parallel outputs -- but prints no equations.  Our own derivation,
for one chunk of C tokens starting from state S0 (chunk-local, 1-based t, s):

  gamma_t = 1 - eta_t lambda_t,   D[t,s] = prod_{i=s+1..t} gamma_i (D[t,t]=1),
  g_t = D[t,0],  L[t,s] = D[t-1,s] eta_s (x_t . x_s)         (s < t),
  T = (I + L)^{-1},  W = T diag(g_{t-1}) X,  U = T Y,
  R = U - W S0                         (the true residuals r_t),
  P[t,s] = D[t,s] eta_s (q_t . x_s)    (s <= t),
  O = diag(g) Q S0 + P R,
  S_C = g_C S0 + X^T diag(D[C,s] eta_s) R.

D is formed from direct products, never by dividing prefix products, because
gamma can be zero or negative.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(777)


def chunked_falcon1(q, k, v, beta, lam, S0, eps, C):
    T, dk = q.shape
    dv = v.shape[1]
    # shifted pairs: x_t = k_{t-1}, x_1 = 0 with eta_1 = 0
    X = np.vstack([np.zeros((1, dk)), k[:-1]])
    n = np.sum(X * X, axis=1)
    eta = beta / (n + lam + eps)
    eta[0] = 0.0
    gam = 1.0 - eta * lam
    S = S0.copy()
    O = np.zeros((T, dv))
    for c0 in range(0, T, C):
        sl = slice(c0, min(c0 + C, T))
        Xc, Qc, Yc = X[sl], q[sl], v[sl]
        ec, gc = eta[sl], gam[sl]
        m = Xc.shape[0]
        D = np.zeros((m + 1, m + 1))       # index 0 = chunk start
        for t in range(m + 1):
            D[t, t] = 1.0
            for s in range(t - 1, -1, -1):
                D[t, s] = D[t, s + 1] * gc[s]   # gamma of token s+1 (1-based)
        g = D[1:, 0]
        gm = D[:-1, 0]
        A = Xc @ Xc.T
        Lm = np.zeros((m, m))
        for t in range(m):
            for s in range(t):
                Lm[t, s] = D[t, s + 1] * ec[s] * A[t, s]
        Tm = np.linalg.inv(np.eye(m) + Lm)
        W = Tm @ (gm[:, None] * Xc)
        U = Tm @ Yc
        R = U - W @ S
        P = np.zeros((m, m))
        QX = Qc @ Xc.T
        for t in range(m):
            for s in range(t + 1):
                P[t, s] = D[t + 1, s + 1] * ec[s] * QX[t, s]
        O[sl] = g[:, None] * (Qc @ S) + P @ R
        wC = D[m, 1:] * ec
        S = g[-1] * S + Xc.T @ (wC[:, None] * R)
    return O, S


@pytest.mark.parametrize("C", [1, 3, 8, 16, 64])
@pytest.mark.parametrize("T", [1, 2, 37, 64, 100])
def test_chunked_form_matches_oracle(C, T):
    dk, dv = 8, 6
    q, v = RNG.standard_normal((T, dk)), RNG.standard_normal((T, dv))
    k = RNG.standard_normal((T, dk)) * np.exp(RNG.standard_normal((T, 1)))
    beta = RNG.uniform(1.5, 1.99, T)
    lam = RNG.uniform(0, 0.5, T)
    S0 = RNG.standard_normal((dk, dv))
    o_ref, S_ref = oracle.falcon1(q, k, v, beta, lam, S0=S0, eps=1e-6)
    o, S = chunked_falcon1(q, k, v, beta, lam, S0, 1e-6, C)
    scale = max(1.0, np.abs(o_ref).max())
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-9 * scale)
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-9 * max(1.0, np.abs(S_ref).max()))


def test_chunked_form_with_nonpositive_decay():
    """Force gamma <= 0 tokens (tiny keys, large lambda): the division-free
    products keep the chunk form exact."""
    T, dk, dv, C = 40, 8, 5, 16
    q, v = RNG.standard_normal((T, dk)), RNG.standard_normal((T, dv))
    k = RNG.standard_normal((T, dk))
    k[5] *= 1e-3
    k[20] *= 1e-3
    beta = np.full(T, 1.9)
    lam = np.full(T, 0.3)
    S0 = RNG.standard_normal((dk, dv))
    X = np.vstack([np.zeros((1, dk)), k[:-1]])
    eta = beta / (np.sum(X * X, 1) + lam + 1e-6)
    assert (1 - eta[1:] * lam[1:]).min() <= 0.0
    o_ref, S_ref = oracle.falcon1(q, k, v, beta, lam, S0=S0, eps=1e-6)
    o, S = chunked_falcon1(q, k, v, beta, lam, S0, 1e-6, C)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-9 * np.abs(o_ref).max())
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-9 * np.abs(S_ref).max())


# ---------------------------------------------------------------- two segments

def _run_mode(mode, q, k, v, beta, lam, S0, k_init, rbw, same_pair):
    if mode == "linattn":
        return oracle.linattn(q, k, v, S0=S0, phi="elu1", rbw=rbw)
    return oracle.falcon1(q, k, v, beta, lam, S0=S0, k_init=k_init, eps=1e-6,
                          inner=(mode == "falcon1a"), rbw=rbw, same_pair=same_pair)


@pytest.mark.parametrize("mode,rbw,same_pair", [("falcon1", False, False), ("falcon1", True, False),
                                                ("falcon1", False, True), ("falcon1a", False, False),
                                                ("linattn", False, False), ("linattn", True, False)])
def test_two_segment_affine_composition(mode, rbw, same_pair):
    """The state map of a run of tokens is affine in its initial state
    (S_t = Phi_t S_mid + S_t^0), which the chunked prefill's two-segment form
    uses: split the chain at t0, run the second segment from a zero state and
    again from S = I with zero targets (its outputs are Phi_t^T q_t, its final
    state Phi_T); then o_t = o_t^0 + S_mid^T Phi_t^T q_t and
    S_T = Phi_T S_mid + S_T^0 reproduce the whole run (the Falcon page §3.2
    write and §4.3's additive write, the blog's linear-attention sum)."""
    T, dk, dv, t0 = 57, 6, 5, 23
    q = RNG.standard_normal((T, dk))
    k = RNG.standard_normal((T, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = RNG.standard_normal((T, dv))
    beta = RNG.uniform(0.1, 1.95, T)   # gamma <= 0 on some tokens
    lam = RNG.uniform(0.0, 0.6, T)
    S0 = RNG.standard_normal((dk, dv)) * 0.3
    o_full, S_full = _run_mode(mode, q, k, v, beta, lam, S0, None, rbw, same_pair)
    o0, S_mid = _run_mode(mode, q[:t0], k[:t0], v[:t0], beta[:t0], lam[:t0], S0, None, rbw, same_pair)
    # the second segment's first pair is (k_{t0-1}, v_t0) when keys are shifted
    kin = k[t0 - 1] if (mode != "linattn" and not same_pair) else None
    sl = slice(t0, T)
    oz, Sz = _run_mode(mode, q[sl], k[sl], v[sl], beta[sl], lam[sl], None, kin, rbw, same_pair)
    oi, Phi = _run_mode(mode, q[sl], k[sl], np.zeros((T - t0, dk)), beta[sl], lam[sl], np.eye(dk),
                        kin, rbw, same_pair)
    o = np.concatenate([o0, oz + oi @ S_mid])
    S = Phi @ S_mid + Sz
    np.testing.assert_allclose(o, o_full, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(S, S_full, rtol=1e-10, atol=1e-10)
