"""GPU parity of the Falcon-3 / 3A window kernels against the fp64 oracle,
through the C ABI (fw_window_prefill, fw_window_step).

Gates as for the other paths: relative L2 over the whole tensor, o, S_T and
the carried window separately, 1e-4 for fp32 inputs and 2e-2 for bf16 inputs
(fp32 state).  Sizes span several staged token blocks (32 tokens for windows
up to 4 pairs, 16 above) with a ragged tail.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_token_mixer_gb300 import fw
from linear_token_mixer_gb300 import inputs as I
from tests.parity_util import TOL, gate_prefill, rel_l2, select_chains, to64

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from linear_token_mixer_gb300 import build as B
    B.build()
    fw.lib()
    torch.cuda.init()


def _inputs(mode, dtype, d, T, W, B=2, H=2, seed=31, s0=True, key_norm="unit"):
    base = I.WORKLOADS["falcon3_bf16"]
    w = base.with_shape(B=B, H=H, T=T, d=d, dtype=dtype, s0_std=0.1 if s0 else 0.0,
                        mode=mode, window=W, key_norm=key_norm)
    return w, I.prefill_inputs(w, seed=seed)


def _dev(x):
    return {k: (t.to(DEV) if t is not None else None) for k, t in x.items()}


def _oracle(w, x, k_init=None, win=None, rbw=False, same_pair=False):
    c = {k: (t.cpu() if t is not None else None) for k, t in x.items()}
    return oracle.falcon3(c["q"], c["k"], c["v"], c["beta"], c["lam"], w.window, S0=c["S0"],
                          k_init=None if k_init is None else k_init.cpu(),
                          win=None if win is None else (to64(win[0]), to64(win[1]),
                                                        win[2].cpu().numpy()),
                          phi=w.phi, eps=w.eps, inner=(w.mode == "falcon3a"), rbw=rbw,
                          same_pair=same_pair)


def _gpu(w, x, k_init=None, win_in=None, rbw=False, same_pair=False):
    g = _dev(x)
    o, S, win = fw.window_prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], w.window,
                                  g["S0"], mode=w.mode, phi=w.phi, eps=w.eps,
                                  k_init=None if k_init is None else k_init.to(DEV),
                                  win_in=win_in, rbw=rbw, same_pair=same_pair)
    fw.check()
    return o, S, win


def _assert_close(w, got, ref):
    tol = TOL[w.dtype]
    o, S, win = got
    o_ref, S_ref, win_ref = ref
    eo, es = gate_prefill(to64(o), o_ref, to64(S), S_ref, tol)
    if w.window > 1:
        np.testing.assert_array_equal(win[2].cpu().numpy(), win_ref[2])
        ex, ey = rel_l2(to64(win[0]), win_ref[0]), rel_l2(to64(win[1]), win_ref[1])
        assert ex <= 1e-6 and ey <= 1e-6, (ex, ey)   # copies of (phi of) the inputs
    return eo, es


@pytest.mark.parametrize("W", [1, 2, 4, 5, 8])
@pytest.mark.parametrize("mode", ["falcon3", "falcon3a"])
@pytest.mark.parametrize("dtype,d", [(torch.float32, 64), (torch.float32, 128),
                                     (torch.bfloat16, 128)])
def test_window_prefill_matches_oracle(dtype, d, mode, W):
    w, x = _inputs(mode, dtype, d, T=77, W=W)
    _assert_close(w, _gpu(w, x), _oracle(w, x))


@pytest.mark.parametrize("rbw,same_pair", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("mode", ["falcon3", "falcon3a"])
@pytest.mark.parametrize("W", [3, 8])
def test_window_prefill_flags(W, mode, rbw, same_pair):
    w, x = _inputs(mode, torch.float32, 64, T=45, W=W)
    _assert_close(w, _gpu(w, x, rbw=rbw, same_pair=same_pair),
                  _oracle(w, x, rbw=rbw, same_pair=same_pair))


@pytest.mark.parametrize("W", [1, 4, 7])
def test_window_of_one_and_more_with_lognormal_keys_and_elu(W):
    # unnormalised keys (LogNormal norms) and phi = elu + 1 on the key
    w, x = _inputs("falcon3", torch.float32, 64, T=70, W=W, key_norm="lognormal")
    w = w.with_shape(phi="elu1")
    _assert_close(w, _gpu(w, x), _oracle(w, x))


@pytest.mark.parametrize("T", [1, 2, 3, 16, 32, 33])
@pytest.mark.parametrize("W", [4, 8])
def test_window_prefill_short_and_block_edge_lengths(W, T):
    w, x = _inputs("falcon3", torch.float32, 64, T=T, W=W, s0=False)
    _assert_close(w, _gpu(w, x), _oracle(w, x))


@pytest.mark.parametrize("mode", ["falcon3", "falcon3a"])
@pytest.mark.parametrize("W,T1", [(4, 1), (4, 2), (4, 40), (8, 5), (8, 37)])
def test_carried_window_continues_a_prefill(W, T1, mode):
    # GPU prefill of T1 tokens, then of the rest with the state, the last key
    # and the carried window, against the oracle on the whole sequence
    T = 61
    w, x = _inputs(mode, torch.float32, 64, T=T, W=W)
    first = {k: (t[:, :, :T1].contiguous() if t is not None and k != "S0" else t)
             for k, t in x.items()}
    w1 = w.with_shape(T=T1)
    o1, S1, win1 = _gpu(w1, first)
    rest = {k: (t[:, :, T1:].contiguous() if t is not None and k != "S0" else None)
            for k, t in x.items()}
    rest["S0"] = S1
    o2, S2, win2 = _gpu(w.with_shape(T=T - T1), rest, k_init=x["k"][:, :, T1 - 1].contiguous(),
                        win_in=win1)
    ref = _oracle(w, x)
    _assert_close(w, (torch.cat([o1, o2], dim=2), S2, win2), ref)


@pytest.mark.parametrize("mode", ["falcon3", "falcon3a"])
@pytest.mark.parametrize("W", [1, 2, 4, 8])
@pytest.mark.parametrize("rbw", [False, True])
def test_window_steps_continue_a_prefill(W, mode, rbw):
    # a GPU prefill of T1 tokens, then one fw_window_step per token (the two
    # window buffers alternate), against the oracle's whole prefill
    T, T1 = 24, 5
    for dtype, d in ((torch.float32, 64), (torch.bfloat16, 128)):
        w, x = _inputs(mode, dtype, d, T=T, W=W, B=3, H=2)
        first = {k: (t[:, :, :T1].contiguous() if t is not None and k != "S0" else t)
                 for k, t in x.items()}
        o1, S, win = _gpu(w.with_shape(T=T1), first, rbw=rbw)
        g = _dev(x)
        spare = fw.new_window(w.B, w.H, d, W) if W > 1 else None
        outs = [o1]
        for t in range(T1, T):
            o, out = fw.window_step(g["q"][:, :, t].contiguous(), g["k"][:, :, t - 1].contiguous(),
                                    g["v"][:, :, t].contiguous(), g["beta"][:, :, t].contiguous(),
                                    g["lam"][:, :, t].contiguous(), S, W, win_in=win,
                                    win_out=spare, mode=mode, eps=w.eps, rbw=rbw)
            spare, win = win, out
            outs.append(o[:, :, None])
        fw.check()
        ref = _oracle(w, x, rbw=rbw)
        _assert_close(w, (torch.cat(outs, dim=2), S, win), ref)


def test_window_step_from_an_empty_window_matches_the_oracle_step():
    # a lone step with no carried pairs and with a partly filled window
    W, d = 5, 128
    rng = torch.Generator().manual_seed(5)
    B, H = 4, 3
    q, k, v = (torch.randn(B, H, d, generator=rng).to(torch.bfloat16) for _ in range(3))
    beta = torch.rand(B, H, generator=rng) * 1.4 + 0.1
    lam = torch.rand(B, H, generator=rng) * 0.1
    S0 = torch.randn(B, H, d, d, generator=rng) * 0.1
    cx = torch.randn(B, H, W - 1, d, generator=rng)
    cy = torch.randn(B, H, W - 1, d, generator=rng)
    cn = torch.randint(0, W, (B, H), generator=rng, dtype=torch.int32)
    for win in (None, (cx, cy, cn)):
        S = S0.to(DEV).clone()
        o, out = fw.window_step(q.to(DEV), k.to(DEV), v.to(DEV), beta.to(DEV), lam.to(DEV), S, W,
                                win_in=None if win is None else tuple(t.to(DEV) for t in win))
        fw.check()
        o_ref, S_ref, win_ref = oracle.step3(q, k, v, beta, lam, S0, W,
                                             win=None if win is None else
                                             (to64(cx), to64(cy), cn.numpy()))
        assert rel_l2(to64(o), o_ref) <= TOL[torch.bfloat16]
        assert rel_l2(to64(S), S_ref) <= 1e-5
        np.testing.assert_array_equal(out[2].cpu().numpy(), win_ref[2])
        # held slots are copies; slots that hold no pair are zero
        np.testing.assert_allclose(to64(out[0]), win_ref[0], rtol=0, atol=1e-6)
        np.testing.assert_allclose(to64(out[1]), win_ref[1], rtol=0, atol=1e-6)


@pytest.mark.parametrize("name", ["falcon3_bf16", "falcon3a_bf16"])
def test_full_size_window_prefill_sampled_chains(name):
    # the full workload in the launch configuration the bench times; the
    # oracle recomputes three whole chains (chains are independent)
    w = I.WORKLOADS[name]
    x = _dev(I.prefill_inputs(w, device=DEV))
    o, S, win = fw.window_prefill(x["q"], x["k"], x["v"], x["beta"], x["lam"], w.window,
                                  x["S0"], mode=w.mode, eps=w.eps)
    fw.check()
    idx = [0, 57, w.B * w.H - 1]
    sub = select_chains(x, idx)
    ref = oracle.falcon3(sub["q"], sub["k"], sub["v"], sub["beta"], sub["lam"], w.window,
                         S0=sub["S0"], eps=w.eps, inner=(w.mode == "falcon3a"))
    of = o.reshape(-1, w.T, w.d)[idx].unsqueeze(0)
    Sf = S.reshape(-1, w.d, w.d)[idx].unsqueeze(0)
    gate_prefill(to64(of), ref[0], to64(Sf), ref[1], TOL[w.dtype])
    assert torch.isfinite(o.float()).all() and torch.isfinite(S).all()


@pytest.mark.parametrize("W", [2, 4, 8])
def test_window_prefill_degenerate_and_badly_scaled_windows(W):
    # windows whose Gram matrix is singular (a key repeated over several
    # tokens) or badly conditioned (keys scaled down by 1e-3 next to unit
    # keys): the eigenvalue solve must still give the window's lambda_max
    w, x = _inputs("falcon3", torch.float32, 64, T=90, W=W, key_norm="unit")
    k = x["k"].clone()
    k[:, :, 10:20] = k[:, :, 10:11]          # one key ten times in a row
    k[:, :, 40:60:3] *= 1e-3                 # small keys among unit keys
    k[:, :, 70:75] = 0.0                     # zero keys (pairs that exist, x = 0)
    x["k"] = k
    _assert_close(w, _gpu(w, x), _oracle(w, x))
    # the same windows through the decode step, prefill of 8 tokens first
    first = {kk: (t[:, :, :8].contiguous() if t is not None and kk != "S0" else t)
             for kk, t in x.items()}
    o1, S, win = _gpu(w.with_shape(T=8), first)
    g = _dev(x)
    spare = fw.new_window(w.B, w.H, w.d, W)
    outs = [o1]
    for t in range(8, w.T):
        o, out = fw.window_step(g["q"][:, :, t].contiguous(), g["k"][:, :, t - 1].contiguous(),
                                g["v"][:, :, t].contiguous(), g["beta"][:, :, t].contiguous(),
                                g["lam"][:, :, t].contiguous(), S, W, win_in=win,
                                win_out=spare, eps=w.eps)
        spare, win = win, out
        outs.append(o[:, :, None])
    fw.check()
    _assert_close(w, (torch.cat(outs, dim=2), S, win), _oracle(w, x))


@pytest.mark.parametrize("mode", ["falcon3", "falcon3a"])
def test_window_step_full_size_sampled(mode):
    # the decode configuration the bench times: 256 sequences x H=32 states, d=128,
    # fp32 state (537 MB), bf16 step vectors, W=4, the two window buffers
    # alternating; three steps from a random state, so the carried window holds
    # 0, 1, 2 pairs.  Sampled states against the oracle's step, one by one.
    cfg = I.DECODE
    Bn, H, d, W, K = cfg["batch"], cfg["H"], cfg["d"], 4, 3
    x = I.decode_inputs(K, Bn, H, d)
    g = torch.Generator().manual_seed(41)
    S0 = torch.randn(Bn, H, d, d, generator=g) * 0.05
    S = S0.to(DEV)
    wins = [fw.new_window(Bn, H, d, W, DEV), fw.new_window(Bn, H, d, W, DEV)]
    outs = []
    for s in range(K):
        o, _ = fw.window_step(x["q"][s].to(DEV), x["k_prev"][s].to(DEV), x["v"][s].to(DEV),
                              x["beta"][s].to(DEV), x["lam"][s].to(DEV), S, W,
                              win_in=wins[s & 1] if s > 0 else None, win_out=wins[(s + 1) & 1],
                              mode=mode, eps=cfg["eps"])
        outs.append(o.cpu())
    fw.check()
    bi = torch.tensor([0, 17, 128, 255, 200, 64, 255])
    hi = torch.tensor([0, 5, 31, 31, 3, 16, 0])
    S_ref, win = S0[bi, hi], None
    for s in range(K):
        o_ref, S_ref, win = oracle.step3(x["q"][s][bi, hi], x["k_prev"][s][bi, hi],
                                         x["v"][s][bi, hi], x["beta"][s][bi, hi],
                                         x["lam"][s][bi, hi], S_ref, W, win=win,
                                         eps=cfg["eps"], inner=(mode == "falcon3a"))
        assert rel_l2(to64(outs[s][bi, hi]), o_ref) <= TOL[torch.bfloat16]
    assert rel_l2(to64(S.cpu()[bi, hi]), S_ref) <= 1e-5
    last = wins[K & 1]
    np.testing.assert_array_equal(last[2].cpu()[bi, hi].numpy(), win[2])
    np.testing.assert_allclose(to64(last[0].cpu()[bi, hi]), win[0], rtol=0, atol=1e-6)
    np.testing.assert_allclose(to64(last[1].cpu()[bi, hi]), win[1], rtol=0, atol=1e-6)
