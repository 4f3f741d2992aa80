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
