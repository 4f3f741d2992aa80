"""GPU parity of the chunked tensor-core prefill of the per-channel step
(Falcon-2 / 2A: a step size per value channel), through the C ABI, against
the fp64 oracle.

Passages: "Fast Weight Attention for Continual Learning" paper reading §4.2
(eta_{t,j} = beta_{t,j} / (|x_t|^2 + lambda_t + eps), shared residual and
feature), §4.3 (the additive write of 2A), §4.4 (shared Gram matrix, one
triangular system per channel).  Every chain is gated on its own: relative L2
of o and S_T, 2e-2 for bf16 inputs with the fp32 state.
"""
import pytest
import torch

import oracle
from linear_token_mixer_gb300 import fw
from linear_token_mixer_gb300 import inputs as I
from tests.parity_util import TOL, gate_prefill, rel_l2, to64

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from linear_token_mixer_gb300 import build as B
    B.build()
    fw.lib()
    torch.cuda.init()


def _inputs(T, B=2, H=3, seed=1, mode="falcon2"):
    w = I.WORKLOADS["falcon2_bf16"].with_shape(B=B, H=H, T=T, mode=mode)
    return w, I.prefill_inputs(w, seed=seed)


def _run(w, x, algo="chunked", rbw=False, same_pair=False, k_init=None):
    g = {k: (t.to(DEV) if t is not None else None) for k, t in x.items()}
    o, S = fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], g["S0"], mode=w.mode,
                      eps=w.eps, algo=algo, rbw=rbw, same_pair=same_pair,
                      k_init=None if k_init is None else k_init.to(DEV))
    fw.check()
    return o, S


def _check(w, x, algo="chunked", rbw=False, same_pair=False, k_init=None):
    o, S = _run(w, x, algo, rbw, same_pair, k_init)
    c = {k: (t.cpu() if t is not None else None) for k, t in x.items()}
    o_ref, S_ref = oracle.falcon2(c["q"], c["k"], c["v"], c["beta"], c["lam"], c["S0"],
                                  k_init=None if k_init is None else k_init.cpu(), eps=w.eps,
                                  inner=(w.mode == "falcon2a"), rbw=rbw, same_pair=same_pair)
    return gate_prefill(to64(o), o_ref, to64(S), S_ref, TOL[torch.bfloat16])


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 130, 257])
@pytest.mark.parametrize("mode", ["falcon2", "falcon2a"])
def test_chan_chunked_ragged(mode, T):
    w, x = _inputs(T, seed=T, mode=mode)
    _check(w, x)


@pytest.mark.parametrize("mode", ["falcon2", "falcon2a"])
@pytest.mark.parametrize("rbw,same_pair,kinit", [(True, False, False), (False, True, False),
                                                 (True, True, False), (False, False, True),
                                                 (True, False, True)])
def test_chan_chunked_variants(mode, rbw, same_pair, kinit):
    w, x = _inputs(150, seed=5, mode=mode)
    k_init = None
    if kinit:
        k_init = torch.randn(w.B, w.H, w.d, generator=torch.Generator().manual_seed(6))
        k_init = (k_init / k_init.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    _check(w, x, rbw=rbw, same_pair=same_pair, k_init=k_init)


def test_chan_chunked_nonpositive_decay_and_zero_steps():
    """Some (token, channel) pairs with gamma <= 0 (tiny keys, large lambda,
    beta near 2), beta = 0 runs and an all-zero key: the block-factored decay
    products use no division."""
    w, x = _inputs(190, seed=9)
    k = x["k"].float()
    k[:, :, 10] *= 1e-3
    k[:, :, 70] *= 1e-3
    k[:, :, 100] = 0.0
    x["k"] = k.to(torch.bfloat16)
    x["lam"][:, :, 11] = 0.5
    x["lam"][:, :, 71] = 0.5
    x["beta"][:, :, 11, :64] = 1.9
    x["beta"][:, :, 71, 64:] = 1.9
    x["beta"][:, :, 40:44] = 0.0
    n = (x["k"].double()[:, :, 10] ** 2).sum(-1)
    eta = x["beta"][:, :, 11, 0].double() / (n + 0.5 + 1e-6)
    assert (1 - eta * 0.5).max() < 0.0
    _check(w, x)


@pytest.mark.parametrize("T", [65, 257])
def test_chan_chunked_many_chains(T):
    w, x = _inputs(T, B=2, H=48, seed=40 + T)
    _check(w, x)


def test_chan_chunked_matches_per_token_kernel():
    # the chunked kernel and the plain per-token kernel agree far inside the gate
    for mode in ("falcon2", "falcon2a"):
        w, x = _inputs(300, seed=3, mode=mode)
        oc, Sc = _run(w, x, "chunked")
        orr, Sr = _run(w, x, "recurrent")
        assert rel_l2(to64(oc), to64(orr)) <= 1e-2
        assert rel_l2(to64(Sc), to64(Sr)) <= 1e-2


def test_chan_chunked_timeout_path_reports_and_recovers():
    """A bounded wait on a barrier nothing arrives on runs out in the
    per-channel kernel too: FW_ERR_TIMEOUT through fw_check, resources freed,
    and the next call on the same context is correct."""
    L = fw.lib()
    w, x = _inputs(200, seed=7)
    g = {k: (t.to(DEV) if t is not None else None) for k, t in x.items()}
    L.fw_set_wait_limit_us(2000)
    L.fw_debug_force_timeout(1)
    try:
        fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], g["S0"], mode=w.mode,
                   eps=w.eps, algo="chunked")
        with pytest.raises(fw.FwError) as ei:
            fw.check()
        assert ei.value.status == -7
    finally:
        L.fw_debug_force_timeout(0)
        L.fw_set_wait_limit_us(0)
    fw.check()  # the error word was cleared
    _check(w, x)
