"""Pins of the oracle's variants, each against something other than the
oracle's own token loop.

Variants (page "Fast Weight Attention for Continual Learning"): the
inner-product family Falcon-1A (§4.3: additive write, no residual, the same
normalised step), Falcon-2 and 2A (§4.2: a step size per value channel, the
residual and feature shared), and the read-before-write / same-step-pair
arms of the 2 x 2 pairing design (§3.3, §4.1).  The pages print no formula for the two
arms; the readings pinned here are o_t = S_{t-1}^T q_t and x_t = phi(k_t).
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(20261207)


def gates(shape_t, lo=0.1, hi=1.5, lam_hi=0.1):
    return RNG.uniform(lo, hi, shape_t), RNG.uniform(0.0, lam_hi, shape_t)


def rand_inputs(nc=2, T=9, dk=5, dv=4, s0=True):
    q = RNG.standard_normal((nc, T, dk))
    k = RNG.standard_normal((nc, T, dk))
    v = RNG.standard_normal((nc, T, dv))
    beta, lam = gates((nc, T))
    S0 = 0.3 * RNG.standard_normal((nc, dk, dv)) if s0 else None
    return q, k, v, beta, lam, S0


# ---------------------------------------------------------------- same-step pair

def test_same_pair_is_the_shifted_form_on_rolled_keys():
    # x_t = k_t for every t  ==  shifted pairing (x_t = k'_{t-1}) on k'_s = k_{s+1}
    # with the first key supplied as k_init.
    q, k, v, beta, lam, S0 = rand_inputs()
    o1, S1 = oracle.falcon1(q, k, v, beta, lam, S0, same_pair=True)
    k_roll = np.concatenate([k[:, 1:], np.zeros_like(k[:, :1])], axis=1)
    o2, S2 = oracle.falcon1(q, k_roll, v, beta, lam, S0, k_init=k[:, 0])
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(S1, S2, rtol=1e-13, atol=1e-13)


def test_same_pair_first_token_writes():
    # with the same-step pair the first token is a real write: exact recall of
    # (k_1, v_1) when lambda = eps = 0 and beta = 1
    q, k, v, beta, lam, S0 = rand_inputs(T=1)
    o, S = oracle.falcon1(q, k, v, np.ones_like(beta), np.zeros_like(lam), S0, eps=0.0,
                          same_pair=True)
    recall = np.einsum("cij,ci->cj", S, k[:, 0])
    np.testing.assert_allclose(recall, v[:, 0], rtol=1e-12, atol=1e-12)


def test_same_pair_ignores_k_init():
    q, k, v, beta, lam, S0 = rand_inputs()
    a = oracle.falcon1(q, k, v, beta, lam, S0, same_pair=True)
    b = oracle.falcon1(q, k, v, beta, lam, S0, k_init=RNG.standard_normal(k[:, 0].shape),
                       same_pair=True)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ------------------------------------------------------------ read before write

@pytest.mark.parametrize("inner", [False, True])
@pytest.mark.parametrize("same_pair", [False, True])
def test_rbw_reads_the_previous_state(inner, same_pair):
    # o_t(RBW) = S_{t-1}^T q_t, with S_{t-1} from a read-after-write run over the
    # first t-1 tokens; the state after T tokens is the same for both reads.
    q, k, v, beta, lam, S0 = rand_inputs(T=7)
    o_rbw, S_rbw = oracle.falcon1(q, k, v, beta, lam, S0, inner=inner, rbw=True,
                                  same_pair=same_pair)
    _, S_raw = oracle.falcon1(q, k, v, beta, lam, S0, inner=inner, same_pair=same_pair)
    np.testing.assert_allclose(S_rbw, S_raw, rtol=1e-13, atol=1e-13)
    for t in range(q.shape[1]):
        if t == 0:
            S_prev = S0
        else:
            _, S_prev = oracle.falcon1(q[:, :t], k[:, :t], v[:, :t], beta[:, :t], lam[:, :t],
                                       S0, inner=inner, same_pair=same_pair)
        want = np.einsum("cij,ci->cj", S_prev, q[:, t])
        np.testing.assert_allclose(o_rbw[:, t], want, rtol=1e-12, atol=1e-12)


def test_rbw_linear_attention_is_the_strict_quadratic_form():
    # o = tril(phi(Q) phi(K)^T, -1) V + phi(Q) S0   (the diagonal excluded)
    q, k, v, _, _, S0 = rand_inputs(T=8)
    o, S = oracle.linattn(q, k, v, S0, phi="elu1", rbw=True)
    phi = lambda z: np.where(z > 0, z + 1.0, np.exp(np.minimum(z, 0.0)))
    fq, fk = phi(q), phi(k)
    A = np.tril(np.einsum("cti,csi->cts", fq, fk), -1)
    want = np.einsum("cts,csj->ctj", A, v) + np.einsum("cti,cij->ctj", fq, S0)
    np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S, S0 + np.einsum("csi,csj->cij", fk, v), rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------- inner-product 1A

def closed_form_1a(q, k, v, beta, lam, S0, eps, same_pair=False):
    """Falcon-1A written as decayed sums of outer products:
    S_t = (prod_{i<=t} g_i) S0 + sum_{s<=t} (prod_{s<i<=t} g_i) eta_s x_s y_s^T."""
    nc, T, dk = k.shape
    if same_pair:
        x = k.copy()
        has = np.ones((nc, T), bool)
    else:
        x = np.concatenate([np.zeros_like(k[:, :1]), k[:, :-1]], axis=1)
        has = np.ones((nc, T), bool)
        has[:, 0] = False
    n = np.einsum("cti,cti->ct", x, x)
    eta = np.where(has, beta / (n + lam + eps), 0.0)
    g = 1.0 - eta * lam
    o = np.zeros(v.shape)
    S_T = None
    for t in range(T):
        # D[t, s] = prod_{s < i <= t} g_i ; G_t = prod_{i <= t} g_i
        D = np.array([[np.prod(g[c, s + 1:t + 1]) for s in range(t + 1)] for c in range(nc)])
        Gt = np.prod(g[:, :t + 1], axis=1)
        St = Gt[:, None, None] * (S0 if S0 is not None else 0.0) + np.einsum(
            "cs,csi,csj->cij", D * eta[:, :t + 1], x[:, :t + 1], v[:, :t + 1])
        o[:, t] = np.einsum("cij,ci->cj", St, q[:, t])
        S_T = St
    return o, S_T


@pytest.mark.parametrize("same_pair", [False, True])
def test_falcon1a_matches_its_closed_form(same_pair):
    q, k, v, beta, lam, S0 = rand_inputs(T=10)
    o, S = oracle.falcon1(q, k, v, beta, lam, S0, eps=1e-6, inner=True, same_pair=same_pair)
    o2, S2 = closed_form_1a(q, k, v, beta, lam, S0, 1e-6, same_pair=same_pair)
    np.testing.assert_allclose(o, o2, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(S, S2, rtol=1e-11, atol=1e-12)


def test_falcon1a_without_decay_and_unit_step_is_shifted_linear_attention():
    # lambda = 0 and beta_t = |x_t|^2 + eps give eta_t = 1, gamma_t = 1: the write
    # is S += x_t v_t^T with x_t = k_{t-1} (x_1 = 0) -- linear attention (phi =
    # identity) on the keys shifted by one token.
    q, k, v, _, _, S0 = rand_inputs(T=8)
    eps = 1e-3
    x = np.concatenate([np.zeros_like(k[:, :1]), k[:, :-1]], axis=1)
    beta = np.einsum("cti,cti->ct", x, x) + eps
    lam = np.zeros_like(beta)
    o, S = oracle.falcon1(q, k, v, beta, lam, S0, eps=eps, inner=True)
    o2, S2 = oracle.linattn(q, x, v, S0, phi="identity")
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S, S2, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- decode steps

@pytest.mark.parametrize("mode", ["falcon1", "falcon1a"])
def test_step_variants_direct_formula(mode):
    ns, dk, dv = 3, 6, 5
    q = RNG.standard_normal((ns, dk))
    kp = RNG.standard_normal((ns, dk))
    v = RNG.standard_normal((ns, dv))
    beta, lam = gates((ns,))
    S = RNG.standard_normal((ns, dk, dv))
    n = np.einsum("ci,ci->c", kp, kp)
    eta = beta / (n + lam + 1e-6)
    g = 1.0 - eta * lam
    r = v - (np.einsum("cij,ci->cj", S, kp) if mode == "falcon1" else 0.0)
    S_new = g[:, None, None] * S + eta[:, None, None] * np.einsum("ci,cj->cij", kp, r)
    for rbw in (False, True):
        o, S2 = oracle.step(q, kp, v, beta, lam, S, mode=mode, rbw=rbw)
        np.testing.assert_allclose(S2, S_new, rtol=1e-12, atol=1e-12)
        want = np.einsum("cij,ci->cj", S if rbw else S_new, q)
        np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("inner", [False, True])
@pytest.mark.parametrize("rbw", [False, True])
def test_prefill_equals_steps_for_the_variants(inner, rbw):
    q, k, v, beta, lam, S0 = rand_inputs(T=6)
    o, S = oracle.falcon1(q, k, v, beta, lam, S0, inner=inner, rbw=rbw)
    Sc = S0.copy()
    mode = "falcon1a" if inner else "falcon1"
    for t in range(q.shape[1]):
        kp = k[:, t - 1] if t > 0 else np.zeros_like(k[:, 0])
        b = beta[:, t] if t > 0 else np.zeros_like(beta[:, 0])   # empty first write
        ot, Sc = oracle.step(q[:, t], kp, v[:, t], b, lam[:, t], Sc, mode=mode, rbw=rbw)
        np.testing.assert_allclose(ot, o[:, t], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Sc, S, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ Falcon-2 (per channel)

@pytest.mark.parametrize("inner", [False, True])
def test_falcon2_with_equal_channel_steps_is_falcon1(inner):
    q, k, v, beta, lam, S0 = rand_inputs()
    beta_c = np.repeat(beta[..., None], v.shape[-1], axis=-1)
    o2, S2 = oracle.falcon2(q, k, v, beta_c, lam, S0, inner=inner)
    o1, S1 = oracle.falcon1(q, k, v, beta, lam, S0, inner=inner)
    np.testing.assert_allclose(o2, o1, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(S2, S1, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("inner", [False, True])
@pytest.mark.parametrize("rbw,same_pair", [(False, False), (True, True)])
def test_falcon2_channels_are_independent_scalar_writes(inner, rbw, same_pair):
    # the page's "d_v independent scalar updates sharing one separable
    # objective": column j of Falcon-2 is Falcon-1 on value column j alone,
    # with that column's step sizes
    q, k, v, _, lam, S0 = rand_inputs(T=11)
    beta_c = RNG.uniform(0.1, 1.9, v.shape)
    o2, S2 = oracle.falcon2(q, k, v, beta_c, lam, S0, inner=inner, rbw=rbw, same_pair=same_pair)
    for j in range(v.shape[-1]):
        o1, S1 = oracle.falcon1(q, k, v[..., j:j + 1], beta_c[..., j], lam, S0[..., j:j + 1],
                                inner=inner, rbw=rbw, same_pair=same_pair)
        np.testing.assert_allclose(o2[..., j:j + 1], o1, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(S2[..., j:j + 1], S1, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("mode", ["falcon2", "falcon2a"])
def test_falcon2_step_direct_formula(mode):
    ns, dk, dv = 3, 6, 5
    q = RNG.standard_normal((ns, dk))
    kp = RNG.standard_normal((ns, dk))
    v = RNG.standard_normal((ns, dv))
    beta = RNG.uniform(0.1, 1.5, (ns, dv))
    lam = RNG.uniform(0.0, 0.1, (ns,))
    S = RNG.standard_normal((ns, dk, dv))
    n = np.einsum("ci,ci->c", kp, kp)
    eta = beta / (n + lam + 1e-6)[:, None]           # [ns, dv]
    g = 1.0 - eta * lam[:, None]
    r = v - (np.einsum("cij,ci->cj", S, kp) if mode == "falcon2" else 0.0)
    S_new = g[:, None, :] * S + eta[:, None, :] * np.einsum("ci,cj->cij", kp, r)
    for rbw in (False, True):
        o, S2 = oracle.step(q, kp, v, beta, lam, S, mode=mode, rbw=rbw)
        np.testing.assert_allclose(S2, S_new, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(o, np.einsum("cij,ci->cj", S if rbw else S_new, q),
                                   rtol=1e-12, atol=1e-12)


def test_falcon2_prefill_equals_steps():
    q, k, v, _, lam, S0 = rand_inputs(T=6)
    beta_c = RNG.uniform(0.1, 1.5, v.shape)
    o, S = oracle.falcon2(q, k, v, beta_c, lam, S0)
    Sc = S0.copy()
    for t in range(q.shape[1]):
        kp = k[:, t - 1] if t > 0 else np.zeros_like(k[:, 0])
        b = beta_c[:, t] if t > 0 else np.zeros_like(beta_c[:, 0])
        ot, Sc = oracle.step(q[:, t], kp, v[:, t], b, lam[:, t], Sc, mode="falcon2")
        np.testing.assert_allclose(ot, o[:, t], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Sc, S, rtol=1e-12, atol=1e-12)
