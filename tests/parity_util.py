"""Helpers for the GPU-vs-oracle parity tests."""
import numpy as np
import torch

import oracle

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}   # relative L2 gates


def rel_l2(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(got - ref)
    if den == 0:
        return float(num)
    return float(num / den)


def per_chain(got, ref, lead=2):
    """Relative L2 of every chain: the first `lead` axes ([B, H]) index the
    chains, the rest is one chain's tensor.  Returns an array of B*H values."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    n = int(np.prod(ref.shape[:lead]))
    g = got.reshape(n, -1)
    r = ref.reshape(n, -1)
    num = np.linalg.norm(g - r, axis=1)
    den = np.linalg.norm(r, axis=1)
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), num)


def gate(got, ref, tol, what="", lead=2):
    """Gate the whole tensor and every chain on its own at `tol`; the message
    names the worst chain (flat b*H + h index) and its relative L2."""
    whole = rel_l2(got, ref)
    pc = per_chain(got, ref, lead)
    worst = int(np.argmax(pc)) if pc.size else -1
    wv = float(pc[worst]) if pc.size else 0.0
    assert whole <= tol and wv <= tol, (
        "%s: rel-L2 whole %.3e, worst chain %d at %.3e (gate %.0e)" % (what, whole, worst, wv, tol))
    return whole, wv


def gate_prefill(o, o_ref, S, S_ref, tol):
    """o [B,H,T,d] and S_T [B,H,d,d] against the oracle, whole and per chain."""
    eo = gate(o, o_ref, tol, "o")
    es = gate(S, S_ref, tol, "S_T")
    return eo, es


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_prefill(w_mode, phi, eps, x, k_init=None, rbw=False, same_pair=False):
    """Run the oracle on CPU copies of the input dict x (tensors on any device)."""
    c = {k: (t.cpu() if t is not None else None) for k, t in x.items()}
    if w_mode in ("falcon1", "falcon1a"):
        return oracle.falcon1(c["q"], c["k"], c["v"], c["beta"], c["lam"], S0=c["S0"],
                              k_init=None if k_init is None else k_init.cpu(), phi=phi, eps=eps,
                              inner=(w_mode == "falcon1a"), rbw=rbw, same_pair=same_pair)
    return oracle.linattn(c["q"], c["k"], c["v"], S0=c["S0"], phi=phi, rbw=rbw)


def select_chains(x, idx):
    """Flatten [B,H,...] to chains and keep the chains in idx (on CPU)."""
    out = {}
    for k, t in x.items():
        if t is None:
            out[k] = None
            continue
        flat = t.reshape((-1,) + tuple(t.shape[2:]))
        out[k] = flat[torch.as_tensor(idx, device=flat.device)].cpu().unsqueeze(0)
    return out
