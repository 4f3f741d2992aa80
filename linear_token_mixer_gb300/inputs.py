"""Seeded synthetic inputs for the fast-weight recurrence workloads.

This module only draws random numbers; it holds none of the method's
arithmetic.  It serves both the CUDA path (tests, bench) and the fp64 oracle
(tests, CPU baseline), so both always see bit-identical inputs.

Workloads (all synthetic; the pages fix no dataset for this path):

* ``falcon1_fp32``   Falcon-1, fp32, B=1 H=2 T=256 d=64; q,k,v ~ N(0,1), keys
  L2-normalised, phi = identity, beta ~ U(0.1,1), lambda ~ U(0,0.05),
  eps = 1e-6, S0 = 0.
* ``linattn_bf16``   plain causal linear attention, bf16 in / fp32 state,
  B=8 H=16 T=4096 d=128; q,k,v ~ N(0,1)/sqrt(128); phi = elu+1; S0 = 0.
* ``falcon1_bf16``   Falcon-1 chunked prefill, bf16 / fp32 state, B=8 H=16
  T=4096 d=128; q,v ~ N(0,1); keys L2-normalised; beta ~ U(0.1,1.5);
  lambda ~ U(0,0.1); eps = 1e-6; S0 ~ N(0, 0.01) (variance 0.01, std 0.1).
* ``falcon1_long``   long-context Falcon-1, bf16 / fp32 state, B=1 H=32
  T=32768 d=128; q,v ~ N(0,1); keys = uniform direction times a
  LogNormal(0,1) norm (not normalised); beta ~ U(1.5,1.99);
  lambda ~ U(0,0.01); eps = 1e-6; S0 = 0.
* ``falcon3_bf16``, ``falcon3a_bf16``  Falcon-3 / 3A with a window of W = 4
  pairs on the Falcon-1 bf16 shapes and distributions (the pages fix no
  window size; 4 is a small window of the kind the method is meant for).
* ``decode``         single-token Falcon-1 decode: 256 sequences x H=32,
  d=128, fp32 state starting at 0, 1024 consecutive steps, each with fresh
  bf16 q, k_prev, v ~ N(0,1), k_prev L2-normalised, beta ~ U(0.1,1),
  lambda ~ U(0,0.05), eps = 1e-6.

Key normalisation happens in fp32 before the cast to the input dtype, so the
rounded keys are close to, not exactly, unit length.  Values are drawn with a
``torch.Generator`` on the requested device in a fixed order (q, k, v, beta,
lambda, S0).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    mode: str            # "falcon1" | "falcon1a" | "falcon2" | "falcon2a" | "falcon3"
                         # | "falcon3a" | "linattn"
    phi: str             # "identity" | "elu1"
    dtype: torch.dtype   # dtype of q, k, v, o
    B: int
    H: int
    T: int
    d: int
    qkv_scale: float     # std of q, v (and of k before normalisation)
    key_norm: str        # "unit" | "lognormal" | "none"
    beta: tuple          # U(lo, hi)
    lam: tuple           # U(lo, hi)
    s0_std: float        # 0 -> S0 is None
    eps: float = 1e-6
    seed: int = 0
    window: int = 1      # Falcon-3 / 3A: pairs in the window

    def with_shape(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "falcon1_fp32": Workload("falcon1_fp32", "falcon1", "identity", torch.float32,
                             1, 2, 256, 64, 1.0, "unit", (0.1, 1.0), (0.0, 0.05), 0.0,
                             seed=20261203),
    "linattn_bf16": Workload("linattn_bf16", "linattn", "elu1", torch.bfloat16,
                             8, 16, 4096, 128, 1.0 / math.sqrt(128.0), "none",
                             (0.0, 0.0), (0.0, 0.0), 0.0, seed=20261204),
    "falcon1_bf16": Workload("falcon1_bf16", "falcon1", "identity", torch.bfloat16,
                             8, 16, 4096, 128, 1.0, "unit", (0.1, 1.5), (0.0, 0.1), 0.1,
                             seed=20261205),
    "falcon1_long": Workload("falcon1_long", "falcon1", "identity", torch.bfloat16,
                             1, 32, 32768, 128, 1.0, "lognormal", (1.5, 1.99), (0.0, 0.01),
                             0.0, seed=20261206),
    # the inner-product family and the per-channel step on the Falcon-1 bf16
    # shapes and distributions (beta per value channel for Falcon-2)
    "falcon1a_bf16": Workload("falcon1a_bf16", "falcon1a", "identity", torch.bfloat16,
                              8, 16, 4096, 128, 1.0, "unit", (0.1, 1.5), (0.0, 0.1), 0.1,
                              seed=20261208),
    "falcon2_bf16": Workload("falcon2_bf16", "falcon2", "identity", torch.bfloat16,
                             8, 16, 4096, 128, 1.0, "unit", (0.1, 1.5), (0.0, 0.1), 0.1,
                             seed=20261209),
    # the window family: one step on the average loss of the last 4 pairs
    "falcon3_bf16": Workload("falcon3_bf16", "falcon3", "identity", torch.bfloat16,
                             8, 16, 4096, 128, 1.0, "unit", (0.1, 1.5), (0.0, 0.1), 0.1,
                             seed=20261210, window=4),
    "falcon3a_bf16": Workload("falcon3a_bf16", "falcon3a", "identity", torch.bfloat16,
                              8, 16, 4096, 128, 1.0, "unit", (0.1, 1.5), (0.0, 0.1), 0.1,
                              seed=20261211, window=4),
}

DECODE = dict(batch=256, H=32, d=128, steps=1024, beta=(0.1, 1.0), lam=(0.0, 0.05),
              eps=1e-6, seed=20261207)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _uniform(shape, lo, hi, g, device):
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


def _keys(shape, kind, scale, g, device):
    k = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if kind == "unit":
        k = k / k.norm(dim=-1, keepdim=True)
    elif kind == "lognormal":
        direction = k / k.norm(dim=-1, keepdim=True)
        norm = torch.exp(torch.randn(shape[:-1] + (1,), generator=g, device=device,
                                     dtype=torch.float32))
        k = direction * norm
    else:
        k = k * scale
    return k


def prefill_inputs(w: Workload, device="cpu", seed=None):
    """Return a dict q, k, v, beta, lam (None for linattn), S0 (or None)."""
    g = _gen(device, w.seed if seed is None else seed)
    shp = (w.B, w.H, w.T, w.d)
    q = (torch.randn(shp, generator=g, device=device, dtype=torch.float32) * w.qkv_scale)
    k = _keys(shp, w.key_norm, w.qkv_scale, g, device)
    v = (torch.randn(shp, generator=g, device=device, dtype=torch.float32) * w.qkv_scale)
    out = dict(q=q.to(w.dtype), k=k.to(w.dtype), v=v.to(w.dtype), beta=None, lam=None,
               S0=None)
    if w.mode in ("falcon1", "falcon1a", "falcon3", "falcon3a"):
        out["beta"] = _uniform((w.B, w.H, w.T), *w.beta, g, device)
        out["lam"] = _uniform((w.B, w.H, w.T), *w.lam, g, device)
    elif w.mode in ("falcon2", "falcon2a"):   # a step size per value channel
        out["beta"] = _uniform((w.B, w.H, w.T, w.d), *w.beta, g, device)
        out["lam"] = _uniform((w.B, w.H, w.T), *w.lam, g, device)
    if w.s0_std > 0:
        out["S0"] = torch.randn((w.B, w.H, w.d, w.d), generator=g, device=device,
                                dtype=torch.float32) * w.s0_std
    return out


def decode_inputs(steps, batch, H, d, device="cpu", seed=None, dtype=torch.bfloat16):
    """Per-step decode inputs, all steps drawn up front: q, k_prev, v
    [steps, batch, H, d] in ``dtype``; beta, lam [steps, batch, H] fp32."""
    g = _gen(device, DECODE["seed"] if seed is None else seed)
    shp = (steps, batch, H, d)
    q = torch.randn(shp, generator=g, device=device, dtype=torch.float32)
    k = _keys(shp, "unit", 1.0, g, device)
    v = torch.randn(shp, generator=g, device=device, dtype=torch.float32)
    beta = _uniform((steps, batch, H), *DECODE["beta"], g, device)
    lam = _uniform((steps, batch, H), *DECODE["lam"], g, device)
    return dict(q=q.to(dtype), k_prev=k.to(dtype), v=v.to(dtype), beta=beta, lam=lam)
