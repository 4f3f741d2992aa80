"""GPU parity of the two-segment form of the chunked prefill, through the C ABI,
against the fp64 oracle.

With few chains and a long sequence each chain is split at a chunk boundary: the
first segment runs from S0 while the second runs twice at once, from a zero
state and from S = I with zero targets.  The state map of a segment is affine in
its initial state (the Falcon page §3.2 write, S_t = (1 - eta_t lambda_t) S_{t-1}
+ eta_t x_t (y_t - S_{t-1}^T x_t)^T, and the plain linear-attention sum are both
affine in S_{t-1}), so a second kernel adds S_mid^T (Phi_t^T q_t) to the second
segment's outputs and forms S_T = Phi_T S_mid + S_T^0.  Here the testing hook
forces the split on small ragged cases; the full-size long-context workload
(32 chains, T = 32768) takes it by itself in the full-size sampled test.  Every
chain is gated on its own: relative L2 of o and S_T, 2e-2 for bf16 inputs.
"""
import pytest
import torch

from linear_token_mixer_gb300 import fw
from linear_token_mixer_gb300 import inputs as I
from tests.parity_util import TOL, gate_prefill, oracle_prefill, rel_l2, to64

pytestmark = pytest.mark.gpu

DEV = "cuda"
WL = {"falcon1": "falcon1_bf16", "falcon1a": "falcon1a_bf16", "linattn": "linattn_bf16"}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from linear_token_mixer_gb300 import build as B
    B.build()
    L = fw.lib()
    torch.cuda.init()
    L.fw_debug_segment_split(1)
    yield
    L.fw_debug_segment_split(0)


def _inputs(mode, T, B=2, H=3, seed=1, s0=True, phi=None):
    base = I.WORKLOADS[WL[mode]]
    w = base.with_shape(B=B, H=H, T=T, s0_std=0.1 if s0 else 0.0, phi=phi or base.phi)
    return w, I.prefill_inputs(w, seed=seed)


def _run(w, x, rbw=False, same_pair=False, k_init=None, in_place=False):
    g = {k: (t.to(DEV) if t is not None else None) for k, t in x.items()}
    S_T = g["S0"].clone() if (in_place and g["S0"] is not None) else None
    S0 = S_T if S_T is not None else g["S0"]
    o, S = fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], S0, mode=w.mode, phi=w.phi,
                      eps=w.eps, algo="chunked", rbw=rbw, same_pair=same_pair, S_T=S_T,
                      k_init=None if k_init is None else k_init.to(DEV))
    fw.check()
    return o, S


def _check(w, x, rbw=False, same_pair=False, k_init=None, in_place=False):
    o, S = _run(w, x, rbw, same_pair, k_init, in_place)
    o_ref, S_ref = oracle_prefill(w.mode, w.phi, w.eps, x, k_init=k_init, rbw=rbw,
                                  same_pair=same_pair)
    return gate_prefill(to64(o), o_ref, to64(S), S_ref, TOL[torch.bfloat16])


@pytest.mark.parametrize("T", [65, 128, 130, 257, 700])
@pytest.mark.parametrize("mode", ["falcon1", "falcon1a", "linattn"])
def test_segments_ragged(mode, T):
    w, x = _inputs(mode, T, seed=T, s0=(T % 2 == 0))
    _check(w, x)


@pytest.mark.parametrize("rbw,same_pair,kinit", [(True, False, False), (False, True, False),
                                                 (False, False, True), (True, False, True)])
def test_segments_flags(rbw, same_pair, kinit):
    w, x = _inputs("falcon1", 300, seed=11)
    k_init = None
    if kinit:
        k_init = torch.randn(w.B, w.H, w.d, generator=torch.Generator().manual_seed(12))
        k_init = (k_init / k_init.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    _check(w, x, rbw=rbw, same_pair=same_pair, k_init=k_init)


def test_segments_linattn_identity_map():
    w, x = _inputs("linattn", 333, seed=13, phi="identity")
    _check(w, x)


def test_segments_s0_aliases_s_t():
    w, x = _inputs("falcon1", 257, seed=14)
    _check(w, x, in_place=True)


def test_segments_nonpositive_decay():
    """Long-context distributions (lognormal keys, beta near 2): gamma <= 0 on
    some tokens, so the transition of the second segment is not a plain decay."""
    base = I.WORKLOADS["falcon1_long"]
    w = base.with_shape(B=1, H=4, T=1000)
    x = I.prefill_inputs(w, seed=15)
    _check(w, x)


def test_segments_match_unsplit_kernel():
    """The split and the unsplit chunked kernel agree far inside the gate."""
    L = fw.lib()
    w, x = _inputs("falcon1", 900, seed=16)
    o1, S1 = _run(w, x)
    L.fw_debug_segment_split(-1)
    try:
        o0, S0 = _run(w, x)
    finally:
        L.fw_debug_segment_split(1)
    assert rel_l2(to64(o1), to64(o0)) <= 1e-2
    assert rel_l2(to64(S1), to64(S0)) <= 1e-2


def test_segments_timeout_path_reports_and_recovers():
    """A bounded wait that runs out in the segment launch is reported through
    fw_check (FW_ERR_TIMEOUT; the fix-up then runs on what the aborted launch
    left, in bounds), and the next call on the same context is correct."""
    L = fw.lib()
    w, x = _inputs("falcon1", 300, seed=17)
    g = {k: (t.to(DEV) if t is not None else None) for k, t in x.items()}
    L.fw_set_wait_limit_us(2000)
    L.fw_debug_force_timeout(1)
    try:
        fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], g["S0"], mode=w.mode, phi=w.phi,
                   eps=w.eps, algo="chunked")
        with pytest.raises(fw.FwError) as ei:
            fw.check()
        assert ei.value.status == -7
    finally:
        L.fw_debug_force_timeout(0)
        L.fw_set_wait_limit_us(0)
    fw.check()
    _check(w, x)
