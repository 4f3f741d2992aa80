"""GPU parity of the chunked tensor-core prefill with many chains in one
launch, and of the two plain entry points fw_prefill / fw_step.

The launch picks its state-carry instantiation by the share of SMs the chains
fill, so the edge cases run here with enough chains for the instantiation the
full-size bf16 workloads use (96 chains: B=2, H=48), and at the two chain
counts either side of the switch.  Every chain is gated on its own (relative
L2 of o and S_T against the fp64 oracle, 2e-2 for bf16 inputs).

Passages: "Fast Weight Attention for Continual Learning" paper reading §4.1
(the shifted pair and the first-token boundary), §4.2 (the write), §3.3 / §4.1
(read before write, same-step pair), §4.3 (the inner-product write); the
"Attention is also an FFN" blog §2.1 (linear attention).
"""
import ctypes

import pytest
import torch

import oracle
from linear_token_mixer_gb300 import fw
from linear_token_mixer_gb300 import inputs as I
from tests.parity_util import TOL, gate, gate_prefill, oracle_prefill, to64

pytestmark = pytest.mark.gpu

DEV = "cuda"
MANY = (2, 48)   # B, H: 96 chains


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from linear_token_mixer_gb300 import build as B
    B.build()
    fw.lib()
    torch.cuda.init()


def _inputs(mode, T, B, H, seed, s0=True, phi=None):
    base = I.WORKLOADS["linattn_bf16" if mode == "linattn" else "falcon1_bf16"]
    w = base.with_shape(B=B, H=H, T=T, s0_std=0.1 if s0 else 0.0, mode=mode,
                        phi=phi or base.phi)
    return w, I.prefill_inputs(w, seed=seed)


def _check(w, x, algo="chunked", rbw=False, same_pair=False, k_init=None):
    g = {k: (t.to(DEV) if t is not None else None) for k, t in x.items()}
    o, S = fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], g["S0"], mode=w.mode,
                      phi=w.phi, eps=w.eps, algo=algo, rbw=rbw, same_pair=same_pair,
                      k_init=None if k_init is None else k_init.to(DEV))
    fw.check()
    o_ref, S_ref = oracle_prefill(w.mode, w.phi, w.eps, x, k_init=k_init, rbw=rbw,
                                  same_pair=same_pair)
    return gate_prefill(to64(o), o_ref, to64(S), S_ref, TOL[w.dtype])


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 130, 257])
@pytest.mark.parametrize("mode,phi", [("falcon1", "identity"), ("falcon1a", "identity"),
                                      ("linattn", "elu1"), ("linattn", "identity")])
def test_chunked_many_chains_ragged(mode, phi, T):
    w, x = _inputs(mode, T, *MANY, seed=100 + T, s0=(T % 2 == 0), phi=phi)
    _check(w, x)


@pytest.mark.parametrize("mode", ["falcon1", "falcon1a"])
def test_chunked_many_chains_nonpositive_decay_zero_steps_zero_keys(mode):
    """gamma < 0 tokens (tiny keys with large lambda and beta near 2), beta = 0
    runs across a chunk boundary and an all-zero key, in chains that fill most
    of the SMs."""
    w, x = _inputs(mode, 190, *MANY, seed=7)
    k = x["k"].float()
    k[:, :, 10] *= 1e-3
    k[:, :, 70] *= 1e-3
    k[:, :, 100] = 0.0
    x["k"] = k.to(torch.bfloat16)
    x["lam"][:, :, 11] = 0.5
    x["lam"][:, :, 71] = 0.5
    x["beta"][:, :, 11] = 1.9
    x["beta"][:, :, 71] = 1.9
    x["beta"][:, :, 60:68] = 0.0
    n = (x["k"].double()[:, :, 10] ** 2).sum(-1)
    eta = x["beta"][:, :, 11].double() / (n + 0.5 + 1e-6)
    assert (1 - eta * 0.5).max() < 0.0   # every chain has a negative decay
    _check(w, x)


@pytest.mark.parametrize("T", [5, 64, 200])
@pytest.mark.parametrize("mode", ["falcon1", "falcon1a"])
def test_chunked_many_chains_k_init(mode, T):
    w, x = _inputs(mode, T, *MANY, seed=30 + T)
    kin = torch.randn(*MANY, 128, generator=torch.Generator().manual_seed(T))
    kin = (kin / kin.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    _check(w, x, k_init=kin)


@pytest.mark.parametrize("T", [1, 65, 257])
@pytest.mark.parametrize("mode,rbw,same_pair", [("falcon1", True, False),
                                                ("falcon1", False, True),
                                                ("falcon1", True, True),
                                                ("falcon1a", True, False),
                                                ("falcon1a", False, True),
                                                ("falcon1a", True, True),
                                                ("linattn", True, False)])
def test_chunked_many_chains_variants(mode, rbw, same_pair, T):
    w, x = _inputs(mode, T, *MANY, seed=200 + T)
    _check(w, x, rbw=rbw, same_pair=same_pair)


def _switch_chains():
    """The largest chain count that takes the split state carry (chains on at
    most 11/20 of the SMs), as the launcher computes it."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return (11 * sms) // 20


@pytest.mark.parametrize("side", [0, 1])
@pytest.mark.parametrize("mode", ["falcon1", "falcon1a", "linattn"])
def test_chunked_either_side_of_the_carry_switch(mode, side):
    n = _switch_chains() + side
    w, x = _inputs(mode, 200, 1, n, seed=300 + side, phi="elu1" if mode == "linattn" else None)
    _check(w, x)


# ---------------------------------------------------------------- plain entry points

def _shape(B, H, T, d):
    return fw.fw_shape(B, H, T, d, d)


@pytest.mark.parametrize("T", [70, 200])
@pytest.mark.parametrize("mode", ["falcon1", "linattn"])
def test_fw_prefill_plain_entry_point(mode, T):
    """fw_prefill(q, k, v, beta, lambda, S0) -> (o, S_T) itself, bf16 d = 128,
    against the oracle."""
    phi = "elu1" if mode == "linattn" else "identity"
    w, x = _inputs(mode, T, 2, 3, seed=T, phi=phi)
    g = {k: (t.to(DEV) if t is not None else None) for k, t in x.items()}
    o = torch.empty_like(g["q"])
    S = torch.empty(2, 3, 128, 128, device=DEV)
    shp = _shape(2, 3, T, 128)
    p = lambda t: None if t is None else t.data_ptr()
    st = fw.lib().fw_prefill(p(g["q"]), p(g["k"]), p(g["v"]), p(g["beta"]), p(g["lam"]),
                             p(g["S0"]), p(o), p(S), ctypes.byref(shp), fw.FW_BF16,
                             fw.MODES[mode], fw.PHIS[phi], ctypes.c_float(w.eps),
                             torch.cuda.current_stream().cuda_stream)
    assert st == fw.FW_OK
    fw.check()
    o_ref, S_ref = oracle_prefill(mode, phi, w.eps, x)
    gate_prefill(to64(o), o_ref, to64(S), S_ref, TOL[torch.bfloat16])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fw_step_plain_entry_point(dtype):
    """fw_step(q, k_prev, v, beta, lambda, S) -> (o, S) itself: three steps in
    a row on 6 states, against the oracle's step."""
    steps, Bn, H, d = 3, 2, 3, 128
    x = I.decode_inputs(steps, Bn, H, d, dtype=dtype, seed=21)
    S0 = torch.randn(Bn, H, d, d, generator=torch.Generator().manual_seed(22)) * 0.1
    Sg = S0.to(DEV)
    Sr = S0.double().numpy()
    shp = _shape(Bn, H, 1, d)
    for s in range(steps):
        a = {n: x[n][s].to(DEV).contiguous() for n in ("q", "k_prev", "v", "beta", "lam")}
        og = torch.empty_like(a["q"])
        st = fw.lib().fw_step(a["q"].data_ptr(), a["k_prev"].data_ptr(), a["v"].data_ptr(),
                              a["beta"].data_ptr(), a["lam"].data_ptr(), Sg.data_ptr(),
                              og.data_ptr(), ctypes.byref(shp), fw.DTYPES[dtype],
                              fw.MODES["falcon1"], fw.PHIS["identity"], ctypes.c_float(1e-6),
                              torch.cuda.current_stream().cuda_stream)
        assert st == fw.FW_OK
        o_r, Sr = oracle.step(x["q"][s], x["k_prev"][s], x["v"][s], x["beta"][s], x["lam"][s],
                              Sr, eps=1e-6)
        gate(to64(og), o_r, TOL[dtype], "o")
    fw.check()
    gate(to64(Sg), Sr, TOL[dtype], "S")
