"""GPU parity: the CUDA kernels (through the C ABI) against the fp64 oracle.

Gates (relative L2, o and S_T separately, over the whole tensor and over every
chain on its own): 1e-4 for fp32 inputs, 2e-2 for bf16 inputs with the fp32
state.  A failing gate names the worst chain.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_token_mixer_gb300 import fw
from linear_token_mixer_gb300 import inputs as I
from tests.parity_util import TOL, gate, gate_prefill, oracle_prefill, rel_l2, select_chains, to64

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from linear_token_mixer_gb300 import build as B
    B.build()
    fw.lib()
    torch.cuda.init()


def _small(mode, dtype, d, T, B=2, H=3, s0=True, phi=None, seed=1):
    base = I.WORKLOADS["falcon1_bf16" if mode == "falcon1" else "linattn_bf16"]
    w = base.with_shape(B=B, H=H, T=T, d=d, dtype=dtype, s0_std=0.1 if s0 else 0.0,
                        phi=phi or base.phi)
    return w, I.prefill_inputs(w, seed=seed)


def _gpu(x):
    return {k: (t.to(DEV) if t is not None else None) for k, t in x.items()}


def _check_prefill(w, x, algo, k_init=None, tol=None):
    g = _gpu(x)
    o, S = fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], g["S0"], mode=w.mode,
                      phi=w.phi, eps=w.eps, algo=algo,
                      k_init=None if k_init is None else k_init.to(DEV))
    fw.check()
    o_ref, S_ref = oracle_prefill(w.mode, w.phi, w.eps, x, k_init=k_init)
    return gate_prefill(to64(o), o_ref, to64(S), S_ref, tol or TOL[w.dtype])


# ---------------------------------------------------------------- recurrent

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("mode", ["falcon1", "linattn"])
@pytest.mark.parametrize("T", [1, 2, 3, 65, 200])
def test_recurrent_small(d, dtype, mode, T):
    w, x = _small(mode, dtype, d, T, s0=(T % 2 == 1))
    _check_prefill(w, x, "recurrent")


@pytest.mark.parametrize("phi", ["identity", "elu1"])
@pytest.mark.parametrize("mode", ["falcon1", "linattn"])
def test_recurrent_feature_maps(phi, mode):
    w, x = _small(mode, torch.float32, 64, 37, phi=phi)
    _check_prefill(w, x, "recurrent")


def test_falcon1_fp32_workload_full_size():
    """B=1 H=2 T=256 d=64 fp32: rel-L2 <= 1e-4 on o and S_T."""
    w = I.WORKLOADS["falcon1_fp32"]
    x = I.prefill_inputs(w)
    _check_prefill(w, x, "auto")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_k_init_continuation(dtype):
    w, x = _small("falcon1", dtype, 128, 50)
    kin = torch.randn(2, 3, 128).to(dtype)
    _check_prefill(w, x, "auto", k_init=kin)


def test_s0_aliases_s_t():
    w, x = _small("falcon1", torch.bfloat16, 128, 70)
    g = _gpu(x)
    S = g["S0"].clone()
    o, S2 = fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], S, S_T=S, eps=w.eps)
    fw.check()
    o_ref, S_ref = oracle_prefill("falcon1", "identity", w.eps, x)
    assert S2.data_ptr() == S.data_ptr()
    assert rel_l2(to64(S), S_ref) <= 2e-2 and rel_l2(to64(o), o_ref) <= 2e-2


# ---------------------------------------------------------------- decode

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("mode", ["falcon1", "linattn"])
def test_decode_small(d, dtype, mode):
    steps, Bn, H = 6, 3, 2
    x = I.decode_inputs(steps, Bn, H, d, dtype=dtype, seed=5)
    phi = "identity" if mode == "falcon1" else "elu1"
    S0 = torch.randn(Bn, H, d, d, generator=torch.Generator().manual_seed(3)) * 0.1
    Sg = S0.to(DEV)
    Sr = S0.double().numpy()
    tol = TOL[dtype]
    for s in range(steps):
        args = [x[n][s] for n in ("q", "k_prev", "v", "beta", "lam")]
        og = fw.step(*[a.to(DEV) for a in args[:3]],
                     args[3].to(DEV) if mode == "falcon1" else None,
                     args[4].to(DEV) if mode == "falcon1" else None, Sg, mode=mode, phi=phi)
        o_r, Sr = oracle.step(*args[:3], args[3] if mode == "falcon1" else None,
                              args[4] if mode == "falcon1" else None, Sr, mode=mode, phi=phi)
        assert rel_l2(to64(og), o_r) <= tol
    fw.check()
    assert rel_l2(to64(Sg), Sr) <= tol


def test_decode_workload_full_size_sampled():
    """256 x 32 states, d = 128, 1024 consecutive steps on the GPU exactly as
    the benchmark runs them; 12 sampled states are replayed by the oracle over
    all 1024 steps (o of every step and the final state)."""
    cfg = I.DECODE
    steps, Bn, H, d = cfg["steps"], cfg["batch"], cfg["H"], cfg["d"]
    x = I.decode_inputs(steps, Bn, H, d, device=DEV)
    S = torch.zeros(Bn, H, d, d, device=DEV)
    idx = torch.tensor([0, 1, 31, 32, 977, 4095, 4096, 5000, 6553, 8000, 8190, 8191])
    outs = []
    for s in range(steps):
        o = fw.step(x["q"][s], x["k_prev"][s], x["v"][s], x["beta"][s], x["lam"][s], S,
                    eps=cfg["eps"])
        outs.append(o.reshape(-1, d)[idx.to(DEV)].float())
    fw.check()
    o_gpu = torch.stack(outs).cpu().double().numpy()          # [steps, n, d]
    sub = {k: t.reshape(steps, -1, *t.shape[3:])[:, idx.to(DEV)].cpu() for k, t in x.items()}
    Sr = np.zeros((len(idx), d, d))
    o_ref = np.zeros_like(o_gpu)
    for s in range(steps):
        o_ref[s], Sr = oracle.step(sub["q"][s], sub["k_prev"][s], sub["v"][s], sub["beta"][s],
                                   sub["lam"][s], Sr, eps=cfg["eps"])
    S_gpu = S.reshape(-1, d, d)[idx.to(DEV)].cpu().double().numpy()
    # o is [steps, state, d]: move the state axis first to gate each state alone
    gate(o_gpu.transpose(1, 0, 2), o_ref.transpose(1, 0, 2), 2e-2, "o", lead=1)
    gate(S_gpu, Sr, 2e-2, "S", lead=1)


def test_prefill_equals_decode_steps():
    """prefill(T) equals T fw_step calls with beta = 0 on the first step and
    k_prev = k_{t-1} after (GPU against GPU, fp32)."""
    w, x = _small("falcon1", torch.float32, 128, 24)
    g = _gpu(x)
    o, S = fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], g["S0"], algo="recurrent")
    St = g["S0"].clone()
    for t in range(24):
        kp = g["k"][:, :, t - 1] if t > 0 else torch.zeros_like(g["k"][:, :, 0])
        b = g["beta"][:, :, t].contiguous() if t > 0 else torch.zeros_like(g["beta"][:, :, 0])
        ot = fw.step(g["q"][:, :, t].contiguous(), kp.contiguous(), g["v"][:, :, t].contiguous(),
                     b, g["lam"][:, :, t].contiguous(), St)
        assert rel_l2(to64(ot), to64(o[:, :, t])) <= 1e-5
    fw.check()
    assert rel_l2(to64(St), to64(S)) <= 1e-5


# ---------------------------------------------------------------- full-size bf16 workloads

@pytest.mark.parametrize("name,chains", [
    ("linattn_bf16", [0, 1, 17, 64, 100, 127]),
    ("falcon1_bf16", [0, 5, 33, 64, 90, 127]),
    ("falcon1_long", [0, 13, 31]),
])
def test_bf16_workloads_full_size_sampled(name, chains):
    """Full-size bf16 workloads through the default (benchmarked) kernel; the
    oracle replays sampled chains in full."""
    w = I.WORKLOADS[name]
    x = I.prefill_inputs(w, device=DEV)
    o, S = fw.prefill(x["q"], x["k"], x["v"], x["beta"], x["lam"], x["S0"], mode=w.mode,
                      phi=w.phi, eps=w.eps)
    fw.check()
    sub = select_chains(x, chains)
    o_ref, S_ref = oracle_prefill(w.mode, w.phi, w.eps, sub)
    d = w.d
    o_s = o.reshape(-1, w.T, d)[torch.as_tensor(chains, device=DEV)].cpu().unsqueeze(0)
    S_s = S.reshape(-1, d, d)[torch.as_tensor(chains, device=DEV)].cpu().unsqueeze(0)
    gate_prefill(to64(o_s), o_ref, to64(S_s), S_ref, 2e-2)


# ---------------------------------------------------------------- chunked tensor-core kernel

@pytest.mark.parametrize("mode,phi", [("falcon1", "identity"), ("linattn", "elu1"),
                                      ("linattn", "identity")])
@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 130, 257])
def test_chunked_small(mode, phi, T):
    w, x = _small(mode, torch.bfloat16, 128, T, s0=(T % 2 == 0), phi=phi, seed=T)
    _check_prefill(w, x, "chunked")


def test_chunked_declines_falcon1_elu1():
    """Falcon-1 with phi = elu+1 is not taken by the chunked kernel (bf16
    rounding of phi(k) ~ 1 + k loses the key's varying part); the default
    path serves it with the per-token fp32 kernel within the bf16 gate."""
    w, x = _small("falcon1", torch.bfloat16, 128, 63, phi="elu1")
    g = _gpu(x)
    with pytest.raises(fw.FwError) as ei:
        fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], g["S0"], phi="elu1",
                   algo="chunked")
    assert ei.value.status == -8
    _check_prefill(w, x, "auto")


@pytest.mark.parametrize("T", [5, 64, 200])
def test_chunked_k_init(T):
    w, x = _small("falcon1", torch.bfloat16, 128, T)
    kin = torch.randn(2, 3, 128).to(torch.bfloat16)
    _check_prefill(w, x, "chunked", k_init=kin)


def test_chunked_nonpositive_decay_and_zero_steps():
    """Tokens with gamma <= 0 (tiny keys, large lambda), beta = 0 tokens and
    zero keys: the chunk form uses no division by decay products."""
    w, x = _small("falcon1", torch.bfloat16, 128, 190)
    k = x["k"].float()
    k[:, :, 10] *= 1e-3
    k[:, :, 70] *= 1e-3
    k[:, :, 100] = 0.0
    x["k"] = k.to(torch.bfloat16)
    x["lam"][:, :, 11] = 0.5
    x["lam"][:, :, 71] = 0.5
    x["beta"][:, :, 11] = 1.9
    x["beta"][:, :, 71] = 1.9
    x["beta"][:, :, 40:44] = 0.0
    kf = x["k"].double()
    n = (kf[:, :, 10] ** 2).sum(-1)
    eta = x["beta"][:, :, 11].double() / (n + 0.5 + 1e-6)
    assert (1 - eta * 0.5).max() < 0.0
    _check_prefill(w, x, "chunked")


@pytest.mark.parametrize("mode", ["falcon1", "linattn"])
def test_chunked_matches_recurrent_kernel(mode):
    """The two CUDA kernels agree with each other (and the oracle) on a
    mid-size case spanning many chunks."""
    w, x = _small(mode, torch.bfloat16, 128, 1000, B=2, H=4)
    g = _gpu(x)
    outs = {}
    for algo in ("chunked", "recurrent"):
        outs[algo] = fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], g["S0"],
                                mode=w.mode, phi=w.phi, eps=w.eps, algo=algo)
    fw.check()
    o_ref, S_ref = oracle_prefill(w.mode, w.phi, w.eps, x)
    for algo, (o, S) in outs.items():
        assert rel_l2(to64(o), o_ref) <= 2e-2, algo
        assert rel_l2(to64(S), S_ref) <= 2e-2, algo
    assert rel_l2(to64(outs["chunked"][1]), to64(outs["recurrent"][1])) <= 2e-2


def test_chunked_timeout_path_reports_and_recovers():
    """A bounded wait on a barrier nothing arrives on runs out: the kernel
    reports FW_ERR_TIMEOUT through fw_check, frees its resources and the
    context stays usable for the next call."""
    L = fw.lib()
    w, x = _small("falcon1", torch.bfloat16, 128, 300)
    g = _gpu(x)
    L.fw_set_wait_limit_us(2000)
    L.fw_debug_force_timeout(1)
    try:
        fw.prefill(g["q"], g["k"], g["v"], g["beta"], g["lam"], g["S0"], algo="chunked")
        with pytest.raises(fw.FwError) as ei:
            fw.check()
        assert ei.value.status == -7
    finally:
        L.fw_debug_force_timeout(0)
        L.fw_set_wait_limit_us(0)
    fw.check()  # error word was cleared
    _check_prefill(w, x, "chunked")
