"""fp64 CPU oracle for the causal fast-weight memory recurrence.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never imports, links or calls it, and the two share no code.

The arithmetic lives in ``fw_oracle.c`` (plain sequential double-precision
loops, one token at a time, see its header for the passages it follows).  This
module only builds that file with gcc, loads it with ctypes and moves numpy
arrays in and out.  Inputs are widened to float64 exactly (bf16 and fp32 values
are exactly representable in float64), so the oracle sees the same numbers as
the GPU.

Pins: every function here is pinned by the CPU tests in
``tests/test_oracle_pins.py`` (exact recall, textbook NLMS, ridge fixed point,
first-token boundary, masked quadratic form of linear attention, orthonormal
recall, per-step descent, norm bound, hand-worked golden cases), the variants
by ``tests/test_oracle_variants.py`` and the Falcon-3 window by
``tests/test_oracle_window.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fw_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

PHI = {"identity": 0, "elu1": 1}
MODE = {"falcon1": 0, "linattn": 1, "falcon1a": 2, "falcon2": 3, "falcon2a": 4,
        "falcon3": 5, "falcon3a": 6}
FLAG_RBW, FLAG_SAME_PAIR = 1, 2


def build(force: bool = False) -> str:
    """Compile fw_oracle.c into liboracle.so next to it (gcc, -O2, no fast-math)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            L = ctypes.c_long
            I = ctypes.c_int
            D = ctypes.c_double
            lib.orc_falcon1.argtypes = [L, L, I, I, P, P, P, P, P, P, P, I, D, I, I, P, P, I]
            lib.orc_linattn.argtypes = [L, L, I, I, P, P, P, P, I, I, P, P, I]
            lib.orc_step.argtypes = [L, I, I, I, I, P, P, P, P, P, I, D, P, P, I]
            lib.orc_falcon3.argtypes = [L, L, I, I, I, P, P, P, P, P, P, P, P, P, P, I, D, I, I,
                                        P, P, P, P, P, P, I]
            lib.orc_step3.argtypes = [L, I, I, I, I, I, P, P, P, P, P, I, D, P, P, P, P, P, P,
                                      P, P, I]
            for f in (lib.orc_falcon1, lib.orc_linattn, lib.orc_step, lib.orc_falcon3,
                      lib.orc_step3):
                f.restype = None
            _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor: widen exactly on the CPU
        import torch
        a = a.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _flags(rbw, same_pair):
    return (FLAG_RBW if rbw else 0) | (FLAG_SAME_PAIR if same_pair else 0)


def falcon1(q, k, v, beta, lam, S0=None, k_init=None, phi="identity", eps=1e-6,
            nthreads=None, inner=False, rbw=False, same_pair=False):
    """Falcon-1 prefill (inner=True: the inner-product family, Falcon-1A).
    q,k [..., T, dk]; v [..., T, dv]; beta, lam [..., T]; S0 [..., dk, dv] or
    None (zero state); k_init [..., dk] or None (x_1 = 0).  rbw: read before
    the write; same_pair: x_t = phi(k_t).
    Returns (o [..., T, dv], S_T [..., dk, dv]) as float64 numpy arrays."""
    q, k, v, beta, lam = map(_f64, (q, k, v, beta, lam))
    S0, k_init = _f64(S0), _f64(k_init)
    lead = q.shape[:-2]
    T, dk = q.shape[-2:]
    dv = v.shape[-1]
    nc = int(np.prod(lead)) if lead else 1
    assert k.shape == q.shape and v.shape == lead + (T, dv)
    assert beta.shape == lead + (T,) and lam.shape == lead + (T,)
    o = np.zeros(lead + (T, dv))
    S = np.zeros(lead + (dk, dv))
    _load().orc_falcon1(nc, T, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(lam),
                        _ptr(S0), _ptr(k_init), PHI[phi], float(eps),
                        MODE["falcon1a" if inner else "falcon1"], _flags(rbw, same_pair),
                        _ptr(o), _ptr(S), nthreads or default_threads())
    return o, S


def falcon2(q, k, v, beta, lam, S0=None, k_init=None, phi="identity", eps=1e-6,
            nthreads=None, inner=False, rbw=False, same_pair=False):
    """Falcon-2 prefill: a step per value channel (inner=True: Falcon-2A).
    As falcon1, with beta [..., T, dv].  Returns (o, S_T) as float64 arrays."""
    q, k, v, beta, lam = map(_f64, (q, k, v, beta, lam))
    S0, k_init = _f64(S0), _f64(k_init)
    lead = q.shape[:-2]
    T, dk = q.shape[-2:]
    dv = v.shape[-1]
    nc = int(np.prod(lead)) if lead else 1
    assert k.shape == q.shape and v.shape == lead + (T, dv)
    assert beta.shape == lead + (T, dv) and lam.shape == lead + (T,)
    o = np.zeros(lead + (T, dv))
    S = np.zeros(lead + (dk, dv))
    _load().orc_falcon1(nc, T, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(lam),
                        _ptr(S0), _ptr(k_init), PHI[phi], float(eps),
                        MODE["falcon2a" if inner else "falcon2"], _flags(rbw, same_pair),
                        _ptr(o), _ptr(S), nthreads or default_threads())
    return o, S


def linattn(q, k, v, S0=None, phi="elu1", nthreads=None, rbw=False):
    """Plain causal linear attention (rbw: read before the write).
    Returns (o, S_T) as float64 arrays."""
    q, k, v = map(_f64, (q, k, v))
    S0 = _f64(S0)
    lead = q.shape[:-2]
    T, dk = q.shape[-2:]
    dv = v.shape[-1]
    nc = int(np.prod(lead)) if lead else 1
    o = np.zeros(lead + (T, dv))
    S = np.zeros(lead + (dk, dv))
    _load().orc_linattn(nc, T, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(S0), PHI[phi],
                        _flags(rbw, False), _ptr(o), _ptr(S), nthreads or default_threads())
    return o, S


def step(q, k_prev, v, beta, lam, S, mode="falcon1", phi="identity", eps=1e-6,
         nthreads=None, rbw=False):
    """One decode step (mode falcon1, falcon1a, falcon2, falcon2a or linattn;
    rbw: o = S_old^T q).  q,k_prev [..., dk]; v [..., dv]; beta, lam [...]
    (beta [..., dv] for falcon2 / falcon2a; both may be None in linattn mode);
    S [..., dk, dv].  Returns (o, S_new) as new arrays."""
    q, k_prev, v = map(_f64, (q, k_prev, v))
    beta, lam = _f64(beta), _f64(lam)
    S = _f64(S).copy()
    lead = q.shape[:-1]
    dk = q.shape[-1]
    dv = v.shape[-1]
    ns = int(np.prod(lead)) if lead else 1
    o = np.zeros(lead + (dv,))
    _load().orc_step(ns, dk, dv, MODE[mode], _flags(rbw, False), _ptr(q), _ptr(k_prev),
                     _ptr(v), _ptr(beta),
                     _ptr(lam), PHI[phi], float(eps), _ptr(S), _ptr(o),
                     nthreads or default_threads())
    return o, S


def _window_in(win, lead, W, dk, dv):
    """Carried window (x [..., W-1, dk], y [..., W-1, dv], n [...]) or None."""
    if win is None or W == 1:
        return None, None, None
    cx, cy = _f64(win[0]), _f64(win[1])
    cn = np.ascontiguousarray(np.asarray(win[2], dtype=np.int32))
    assert cx.shape == lead + (W - 1, dk) and cy.shape == lead + (W - 1, dv)
    assert cn.shape == lead and cn.min() >= 0 and cn.max() <= W - 1
    return cx, cy, cn


def falcon3(q, k, v, beta, lam, W, S0=None, k_init=None, win=None, phi="identity", eps=1e-6,
            nthreads=None, inner=False, rbw=False, same_pair=False, want_mu=False):
    """Falcon-3 prefill with a window of the last W pairs (inner=True:
    Falcon-3A).  Shapes as falcon1 (beta, lam [..., T]); win is the window
    carried from an earlier call, (x [..., W-1, dk] with phi applied,
    y [..., W-1, dv], n [...] pairs held in the newest slots), or None.
    Returns (o, S_T, win_out) or, with want_mu, (o, S_T, win_out, mu [..., T])."""
    q, k, v, beta, lam = map(_f64, (q, k, v, beta, lam))
    S0, k_init = _f64(S0), _f64(k_init)
    lead = q.shape[:-2]
    T, dk = q.shape[-2:]
    dv = v.shape[-1]
    nc = int(np.prod(lead)) if lead else 1
    assert 1 <= W <= 64
    assert k.shape == q.shape and v.shape == lead + (T, dv)
    assert beta.shape == lead + (T,) and lam.shape == lead + (T,)
    cx, cy, cn = _window_in(win, lead, W, dk, dv)
    o = np.zeros(lead + (T, dv))
    S = np.zeros(lead + (dk, dv))
    ox = np.zeros(lead + (W - 1, dk))
    oy = np.zeros(lead + (W - 1, dv))
    on = np.zeros(lead, dtype=np.int32)
    mu = np.zeros(lead + (T,))
    _load().orc_falcon3(nc, T, dk, dv, W, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(lam),
                        _ptr(S0), _ptr(k_init), _ptr(cx), _ptr(cy), _ptr(cn), PHI[phi],
                        float(eps), MODE["falcon3a" if inner else "falcon3"],
                        _flags(rbw, same_pair), _ptr(o), _ptr(S), _ptr(ox), _ptr(oy),
                        _ptr(on), _ptr(mu), nthreads or default_threads())
    out = (o, S, (ox, oy, on))
    return out + (mu,) if want_mu else out


def step3(q, k_prev, v, beta, lam, S, W, win=None, phi="identity", eps=1e-6, nthreads=None,
          inner=False, rbw=False):
    """One Falcon-3 (inner=True: 3A) decode step with a window of W pairs:
    the carried window win (as falcon3's, or None = empty) plus the new pair
    (phi(k_prev), v).  q,k_prev [..., dk]; v [..., dv]; beta, lam [...];
    S [..., dk, dv].  Returns (o, S_new, win_out) as new arrays."""
    q, k_prev, v, beta, lam = map(_f64, (q, k_prev, v, beta, lam))
    S = _f64(S).copy()
    lead = q.shape[:-1]
    dk = q.shape[-1]
    dv = v.shape[-1]
    ns = int(np.prod(lead)) if lead else 1
    assert 1 <= W <= 64
    cx, cy, cn = _window_in(win, lead, W, dk, dv)
    o = np.zeros(lead + (dv,))
    ox = np.zeros(lead + (W - 1, dk))
    oy = np.zeros(lead + (W - 1, dv))
    on = np.zeros(lead, dtype=np.int32)
    _load().orc_step3(ns, dk, dv, W, MODE["falcon3a" if inner else "falcon3"],
                      _flags(rbw, False), _ptr(q), _ptr(k_prev), _ptr(v), _ptr(beta),
                      _ptr(lam), PHI[phi], float(eps), _ptr(S), _ptr(cx), _ptr(cy), _ptr(cn),
                      _ptr(o), _ptr(ox), _ptr(oy), _ptr(on), nthreads or default_threads())
    return o, S, (ox, oy, on)
