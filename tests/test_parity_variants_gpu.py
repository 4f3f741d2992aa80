"""GPU parity of the variants against the fp64 oracle, through the C ABI:
the inner-product family (Falcon-1A) and the read-before-write / same-step
pair arms, on every kernel that takes them (per-token prefill, chunked
prefill where supported, decode step).

Gates as for the main paths: relative L2 over the whole tensor and over every
chain, o and S_T separately, 1e-4 for fp32 inputs and 2e-2 for bf16 inputs
(fp32 state).
"""
import numpy as np
import pytest
import torch

import oracle
from linear_token_mixer_gb300 import fw
from linear_token_mixer_gb300 import inputs as I
from tests.parity_util import TOL, gate_prefill, oracle_prefill, rel_l2, select_chains, to64

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from linear_token_mixer_gb300 import build as B
    B.build()
    fw.lib()
    torch.cuda.init()


def _inputs(mode, dtype, d, T, B=2, H=2, seed=11, s0=True, phi=None):
    base = I.WORKLOADS["linattn_bf16" if mode == "linattn" else "falcon1_bf16"]
    w = base.with_shape(B=B, H=H, T=T, d=d, dtype=dtype, s0_std=0.1 if s0 else 0.0,
                        mode=mode, phi=phi or base.phi)
    return w, I.prefill_inputs(w, seed=seed)


def _run(w, x, algo, rbw, same_pair, k_init=None):
    g = {k: (t.to(DEV) if t is not None else None) for k, t in x.items()}
    o, S = fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], g["S0"], mode=w.mode,
                      phi=w.phi, eps=w.eps, algo=algo, rbw=rbw, same_pair=same_pair,
                      k_init=None if k_init is None else k_init.to(DEV))
    fw.check()
    return o, S


def _check(w, x, algo, rbw, same_pair, k_init=None):
    o, S = _run(w, x, algo, rbw, same_pair, k_init)
    o_ref, S_ref = oracle_prefill(w.mode, w.phi, w.eps, x, k_init=k_init, rbw=rbw,
                                  same_pair=same_pair)
    return gate_prefill(to64(o), o_ref, to64(S), S_ref, TOL[w.dtype])


@pytest.mark.parametrize("same_pair", [False, True])
@pytest.mark.parametrize("rbw", [False, True])
@pytest.mark.parametrize("mode", ["falcon1", "falcon1a"])
@pytest.mark.parametrize("dtype,d", [(torch.float32, 64), (torch.float32, 128),
                                     (torch.bfloat16, 64), (torch.bfloat16, 128)])
def test_recurrent_variants(dtype, d, mode, rbw, same_pair):
    w, x = _inputs(mode, dtype, d, T=67, s0=rbw)
    _check(w, x, "recurrent", rbw, same_pair)


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 130])
@pytest.mark.parametrize("mode,rbw,same_pair", [("falcon1a", False, False),
                                                ("falcon1a", True, True),
                                                ("falcon1", True, False),
                                                ("falcon1", False, True),
                                                ("linattn", True, False)])
def test_auto_variants_bf16_d128(T, mode, rbw, same_pair):
    # the dispatch AUTO makes for the variants (the chunked kernel where it takes
    # them, the per-token kernel otherwise); chunk boundaries and a ragged tail
    w, x = _inputs(mode, torch.bfloat16, 128, T=T)
    _check(w, x, "auto", rbw, same_pair)


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 130, 257])
@pytest.mark.parametrize("mode,rbw,same_pair", [("falcon1a", False, False),
                                                ("falcon1a", True, False),
                                                ("falcon1a", False, True),
                                                ("falcon1a", True, True),
                                                ("falcon1", True, False),
                                                ("falcon1", False, True),
                                                ("falcon1", True, True),
                                                ("linattn", True, False)])
def test_chunked_variants(T, mode, rbw, same_pair):
    # the tensor-core kernel itself; S0 != 0 so the decayed start state is read
    w, x = _inputs(mode, torch.bfloat16, 128, T=T, B=2, H=2, seed=T)
    _check(w, x, "chunked", rbw, same_pair)


def test_chunked_variants_match_recurrent_kernel():
    # the two kernels on the same bf16 inputs agree far inside the gate
    for mode, rbw, sp in (("falcon1a", True, True), ("falcon1", True, True)):
        w, x = _inputs(mode, torch.bfloat16, 128, T=300, seed=2)
        oc, Sc = _run(w, x, "chunked", rbw, sp)
        orr, Sr = _run(w, x, "recurrent", rbw, sp)
        assert rel_l2(to64(oc), to64(orr)) <= 1e-2
        assert rel_l2(to64(Sc), to64(Sr)) <= 1e-2


def test_chunked_falcon1a_k_init():
    w, x = _inputs("falcon1a", torch.bfloat16, 128, T=150, seed=7)
    k_init = torch.randn(w.B, w.H, w.d, generator=torch.Generator().manual_seed(8))
    k_init = (k_init / k_init.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    _check(w, x, "chunked", False, False, k_init=k_init)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d", [64, 128])
def test_linattn_rbw(dtype, d):
    w, x = _inputs("linattn", dtype, d, T=37)
    _check(w, x, "recurrent", True, False)


def test_falcon1a_k_init_continuation():
    # two calls with k_init equal one call over the whole sequence
    w, x = _inputs("falcon1a", torch.float32, 64, T=40)
    g = {k: (t.to(DEV) if t is not None else None) for k, t in x.items()}
    o_full, S_full = fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], g["S0"],
                                mode="falcon1a", eps=w.eps)
    cut = 17
    sl = lambda t, a, b: t[:, :, a:b].contiguous()
    o1, S1 = fw.prefill(sl(g["q"], 0, cut), sl(g["k"], 0, cut), sl(g["v"], 0, cut),
                        sl(g["beta"], 0, cut), sl(g["lam"], 0, cut), g["S0"], mode="falcon1a",
                        eps=w.eps)
    o2, S2 = fw.prefill(sl(g["q"], cut, 40), sl(g["k"], cut, 40), sl(g["v"], cut, 40),
                        sl(g["beta"], cut, 40), sl(g["lam"], cut, 40), S1, mode="falcon1a",
                        eps=w.eps, k_init=g["k"][:, :, cut - 1].contiguous())
    fw.check()
    assert rel_l2(to64(torch.cat([o1, o2], dim=2)), to64(o_full)) <= 1e-6
    assert rel_l2(to64(S2), to64(S_full)) <= 1e-6


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mode,rbw", [("falcon1a", False), ("falcon1a", True),
                                      ("falcon1", True), ("linattn", True)])
def test_decode_variants(dtype, d, mode, rbw):
    steps, Bn, H = 5, 3, 2
    x = I.decode_inputs(steps, Bn, H, d, dtype=dtype, seed=9)
    phi = "elu1" if mode == "linattn" else "identity"
    gated = mode != "linattn"
    S0 = torch.randn(Bn, H, d, d, generator=torch.Generator().manual_seed(4)) * 0.1
    Sg = S0.to(DEV)
    Sr = S0.double().numpy()
    tol = TOL[dtype]
    for s in range(steps):
        args = [x[n][s] for n in ("q", "k_prev", "v", "beta", "lam")]
        og = fw.step(*[a.to(DEV) for a in args[:3]], args[3].to(DEV) if gated else None,
                     args[4].to(DEV) if gated else None, Sg, mode=mode, phi=phi, rbw=rbw)
        o_r, Sr = oracle.step(*args[:3], args[3] if gated else None, args[4] if gated else None,
                              Sr, mode=mode, phi=phi, rbw=rbw)
        assert rel_l2(to64(og), o_r) <= tol
    fw.check()
    assert rel_l2(to64(Sg), Sr) <= tol


@pytest.mark.parametrize("rbw,same_pair", [(False, False), (True, True)])
def test_falcon1a_workload_full_size_sampled(rbw, same_pair):
    # B8 H16 T4096 d128 bf16: the whole launch on the GPU, 3 chains checked
    w = I.WORKLOADS["falcon1a_bf16"]
    x = I.prefill_inputs(w, device=DEV)
    o, S = _run(w, x, "auto", rbw, same_pair)
    chains = [0, 61, 127]
    xs = select_chains(x, chains)
    o_ref, S_ref = oracle_prefill(w.mode, w.phi, w.eps, xs, rbw=rbw, same_pair=same_pair)
    og = to64(o.reshape(-1, w.T, w.d)[chains])[None]
    Sg = to64(S.reshape(-1, w.d, w.d)[chains])[None]
    gate_prefill(og, o_ref, Sg, S_ref, TOL[w.dtype])


# ------------------------------------------------- Falcon-2 / 2A (a step per channel)

def _channel_betas(x, dv, seed=12):
    g = torch.Generator().manual_seed(seed)
    lead = tuple(x["beta"].shape)
    return torch.rand(lead + (dv,), generator=g) * 1.4 + 0.1   # U(0.1, 1.5) per channel


@pytest.mark.parametrize("algo", ["auto", "recurrent"])
@pytest.mark.parametrize("mode", ["falcon2", "falcon2a"])
@pytest.mark.parametrize("rbw,same_pair,kinit", [(False, False, False), (True, True, False),
                                                 (True, False, True), (False, True, False)])
@pytest.mark.parametrize("dtype,d", [(torch.float32, 64), (torch.float32, 128),
                                     (torch.bfloat16, 128)])
def test_falcon2_prefill(mode, rbw, same_pair, kinit, dtype, d, algo):
    # AUTO takes the per-channel chunked kernel for bf16 with d = 128 and the
    # staged per-token kernel (window of one pair, a step per column) for the
    # other shapes; RECURRENT the plain per-token kernel.  T spans several blocks.
    w, x = _inputs("falcon1", dtype, d, T=70)
    x["beta"] = _channel_betas(x, d)
    k_init = torch.randn(x["k"].shape[:2] + (d,), generator=torch.Generator().manual_seed(3))
    k_init = k_init.to(dtype) if kinit else None
    g = {k: (t.to(DEV) if t is not None else None) for k, t in x.items()}
    o, S = fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], g["S0"], mode=mode,
                      eps=w.eps, rbw=rbw, same_pair=same_pair, algo=algo,
                      k_init=None if k_init is None else k_init.to(DEV))
    fw.check()
    c = {k: t.cpu() for k, t in x.items()}
    o_ref, S_ref = oracle.falcon2(c["q"], c["k"], c["v"], c["beta"], c["lam"], c["S0"],
                                  k_init=k_init, eps=w.eps, inner=(mode == "falcon2a"), rbw=rbw,
                                  same_pair=same_pair)
    gate_prefill(to64(o), o_ref, to64(S), S_ref, TOL[dtype])


@pytest.mark.parametrize("mode", ["falcon2", "falcon2a"])
def test_falcon2_elu1_bf16_takes_the_per_token_kernel(mode):
    # phi = elu+1 with bf16 d = 128: the chunked kernel declines it (its bf16
    # Gram operands would round phi(k) ~ 1 + k), AUTO serves it on the staged
    # per-token kernel within the bf16 gate
    w, x = _inputs("falcon1", torch.bfloat16, 128, T=90, phi="elu1")
    x["beta"] = _channel_betas(x, 128)
    g = {k: (t.to(DEV) if t is not None else None) for k, t in x.items()}
    o, S = fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], g["S0"], mode=mode,
                      phi="elu1", eps=w.eps)
    fw.check()
    with pytest.raises(fw.FwError):
        fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], g["S0"], mode=mode,
                   phi="elu1", eps=w.eps, algo="chunked")
    c = {k: t.cpu() for k, t in x.items()}
    o_ref, S_ref = oracle.falcon2(c["q"], c["k"], c["v"], c["beta"], c["lam"], c["S0"],
                                  phi="elu1", eps=w.eps, inner=(mode == "falcon2a"))
    gate_prefill(to64(o), o_ref, to64(S), S_ref, TOL[torch.bfloat16])


@pytest.mark.parametrize("mode", ["falcon2", "falcon2a"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rbw", [False, True])
def test_falcon2_decode(mode, dtype, rbw):
    steps, Bn, H, d = 4, 3, 2, 128
    x = I.decode_inputs(steps, Bn, H, d, dtype=dtype, seed=13)
    gb = torch.Generator().manual_seed(14)
    beta = torch.rand(steps, Bn, H, d, generator=gb) * 1.4 + 0.1
    S0 = torch.randn(Bn, H, d, d, generator=torch.Generator().manual_seed(15)) * 0.1
    Sg = S0.to(DEV)
    Sr = S0.double().numpy()
    for s in range(steps):
        og = fw.step(x["q"][s].to(DEV), x["k_prev"][s].to(DEV), x["v"][s].to(DEV),
                     beta[s].to(DEV), x["lam"][s].to(DEV), Sg, mode=mode, rbw=rbw)
        o_r, Sr = oracle.step(x["q"][s], x["k_prev"][s], x["v"][s], beta[s], x["lam"][s], Sr,
                              mode=mode, rbw=rbw)
        assert rel_l2(to64(og), o_r) <= TOL[dtype]
    fw.check()
    assert rel_l2(to64(Sg), Sr) <= TOL[dtype]


@pytest.mark.parametrize("mode", ["falcon2", "falcon2a"])
def test_falcon2_workload_full_size_sampled(mode):
    # B8 H16 T4096 d128 bf16 with a step per value channel, the launch the
    # bench times (AUTO: the per-channel chunked kernel); 4 chains checked
    w = I.WORKLOADS["falcon2_bf16"].with_shape(mode=mode)
    x = I.prefill_inputs(w, device=DEV)
    o, S = fw.prefill(x["q"], x["k"], x["v"], x["beta"], x["lam"], x["S0"], mode=w.mode,
                      eps=w.eps)
    fw.check()
    chains = [0, 31, 77, 127]
    xs = select_chains(x, chains)
    o_ref, S_ref = oracle.falcon2(xs["q"], xs["k"], xs["v"], xs["beta"], xs["lam"], xs["S0"],
                                  eps=w.eps, inner=(mode == "falcon2a"))
    og = to64(o.reshape(-1, w.T, w.d)[chains])[None]
    Sg = to64(S.reshape(-1, w.d, w.d)[chains])[None]
    gate_prefill(og, o_ref, Sg, S_ref, TOL[w.dtype])
