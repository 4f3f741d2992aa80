"""Thin ctypes binding of libfw.so (include/fw.h) over torch CUDA tensors.

Argument marshalling only: every step of the recurrence runs in the library's
CUDA kernels.  There is no CPU path; if libfw.so is missing or fails to load,
every call raises.  torch supplies device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfw.so")

FW_F32, FW_BF16 = 0, 1
MODES = {"falcon1": 0, "linattn": 1, "falcon1a": 2, "falcon2": 3, "falcon2a": 4,
         "falcon3": 5, "falcon3a": 6}
WINDOW_MAX = 8
FLAG_RBW, FLAG_SAME_PAIR = 1, 2
PHIS = {"identity": 0, "elu1": 1}
ALGOS = {"auto": 0, "recurrent": 1, "chunked": 2}
DTYPES = {torch.float32: FW_F32, torch.bfloat16: FW_BF16}

FW_OK = 0
STATUS = {0: "FW_OK", -1: "FW_ERR_NULL", -2: "FW_ERR_SHAPE", -3: "FW_ERR_DTYPE",
          -4: "FW_ERR_ALIGN", -5: "FW_ERR_MODE", -6: "FW_ERR_CUDA", -7: "FW_ERR_TIMEOUT",
          -8: "FW_ERR_UNSUPPORTED", -9: "FW_ERR_ARG", -10: "FW_ERR_DEVICE", -11: "FW_ERR_SCRATCH"}


class FwError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = lib().fw_status_string(status).decode()
        if status == -6:
            msg += " (cudaError %d)" % lib().fw_last_cuda_error()
        super().__init__("%s: %s" % (where, msg))


class fw_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("T", ctypes.c_int64),
                ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32)]


class fw_window(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("y", ctypes.c_void_p), ("n", ctypes.c_void_p)]


EXPORTS = ("fw_prefill", "fw_prefill_ex", "fw_prefill_noalloc", "fw_step", "fw_step_ex", "fw_window_prefill",
           "fw_window_step", "fw_check",
           "fw_status_string", "fw_version", "fw_last_cuda_error", "fw_set_wait_limit_us",
           "fw_debug_force_timeout", "fw_debug_segment_split")

_lib = None


def lib():
    """Load libfw.so (building it first is the caller's job: see build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libfw.so is not built (run linear_token_mixer_gb300/build.py); "
                               "there is no fallback path")
        L = ctypes.CDLL(LIB_PATH)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        SP = ctypes.POINTER(fw_shape)
        L.fw_prefill.argtypes = [P, P, P, P, P, P, P, P, SP, I, I, I, F, P]
        U = ctypes.c_uint
        L.fw_prefill_ex.argtypes = [P, P, P, P, P, P, P, P, P, SP, I, I, I, F, U, I, P]
        L.fw_prefill_noalloc.argtypes = L.fw_prefill_ex.argtypes
        L.fw_step.argtypes = [P, P, P, P, P, P, P, SP, I, I, I, F, P]
        L.fw_step_ex.argtypes = [P, P, P, P, P, P, P, SP, I, I, I, F, U, P]
        WP = ctypes.POINTER(fw_window)
        L.fw_window_prefill.argtypes = [P, P, P, P, P, P, P, WP, P, P, WP, SP, I, I, I, I, F, U,
                                        P]
        L.fw_window_step.argtypes = [P, P, P, P, P, P, WP, P, WP, SP, I, I, I, I, F, U, P]
        L.fw_check.argtypes = [P]
        L.fw_status_string.argtypes = [I]
        L.fw_status_string.restype = ctypes.c_char_p
        L.fw_version.argtypes = []
        L.fw_last_cuda_error.argtypes = []
        L.fw_set_wait_limit_us.argtypes = [ctypes.c_longlong]
        L.fw_set_wait_limit_us.restype = None
        L.fw_debug_force_timeout.argtypes = [I]
        L.fw_debug_force_timeout.restype = None
        L.fw_debug_segment_split.argtypes = [I]
        L.fw_debug_segment_split.restype = None
        for f in (L.fw_prefill, L.fw_prefill_ex, L.fw_prefill_noalloc, L.fw_step, L.fw_step_ex,
                  L.fw_window_prefill,
                  L.fw_window_step, L.fw_check, L.fw_version, L.fw_last_cuda_error):
            f.restype = I
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("fw: tensors must live on a CUDA device (no CPU path)")
    if not t.is_contiguous():
        raise ValueError("fw: tensors must be contiguous")
    return t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _flags(rbw, same_pair):
    return (FLAG_RBW if rbw else 0) | (FLAG_SAME_PAIR if same_pair else 0)


def prefill(q, k, v, beta=None, lam=None, S0=None, *, mode="falcon1", phi="identity",
            eps=1e-6, k_init=None, algo="auto", o=None, S_T=None, stream=None, rbw=False,
            same_pair=False, noalloc=False):
    """Run the recurrence over q, k, v [B, H, T, d] (fp32 or bf16).

    mode: "falcon1", "falcon1a", "falcon2", "falcon2a" or "linattn"; rbw reads
    before the write, same_pair pairs each key with its own value.  Returns
    (o [B,H,T,d] in q's dtype, S_T [B,H,d,d] fp32).  beta, lam [B,H,T] fp32 are
    required in the falcon modes (beta [B,H,T,d] for falcon2 / falcon2a).  S0
    [B,H,d,d] fp32 or None.  noalloc: call fw_prefill_noalloc (the library's
    workspace from its static buffer; pass o and S_T to allocate nothing here
    either)."""
    B, H, T, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    if S_T is None:
        S_T = torch.empty((B, H, d, d), device=q.device, dtype=torch.float32)
    shp = fw_shape(B, H, T, d, v.shape[-1])
    fn = lib().fw_prefill_noalloc if noalloc else lib().fw_prefill_ex
    st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(lam), _ptr(S0), _ptr(k_init), _ptr(o),
            _ptr(S_T), ctypes.byref(shp), DTYPES.get(q.dtype, -1), MODES[mode], PHIS[phi],
            float(eps), _flags(rbw, same_pair), ALGOS[algo], _stream(stream))
    if st != FW_OK:
        raise FwError(st, "fw_prefill_noalloc" if noalloc else "fw_prefill")
    return o, S_T


def step(q, k_prev, v, beta, lam, S, *, mode="falcon1", phi="identity", eps=1e-6, o=None,
         stream=None, rbw=False):
    """One decode step for q, k_prev, v [B, H, d]; S [B, H, d, d] fp32 is
    updated in place (rbw: o = S_old^T q).  Returns o [B, H, d] in q's dtype."""
    B, H, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    shp = fw_shape(B, H, 1, d, v.shape[-1])
    st = lib().fw_step_ex(_ptr(q), _ptr(k_prev), _ptr(v), _ptr(beta), _ptr(lam), _ptr(S),
                          _ptr(o), ctypes.byref(shp), DTYPES.get(q.dtype, -1), MODES[mode],
                          PHIS[phi], float(eps), _flags(rbw, False), _stream(stream))
    if st != FW_OK:
        raise FwError(st, "fw_step")
    return o


def new_window(B, H, d, window, device="cuda"):
    """An empty carried window (x, y, n) for `window` pairs: x, y
    [B, H, window-1, d] fp32, n [B, H] int32, all zero."""
    return (torch.zeros((B, H, window - 1, d), device=device, dtype=torch.float32),
            torch.zeros((B, H, window - 1, d), device=device, dtype=torch.float32),
            torch.zeros((B, H), device=device, dtype=torch.int32))


def _window(w):
    if w is None:
        return None
    x, y, n = w
    if n.dtype != torch.int32 or x.dtype != torch.float32 or y.dtype != torch.float32:
        raise ValueError("fw: a window is (x fp32, y fp32, n int32)")
    return ctypes.byref(fw_window(_ptr(x), _ptr(y), _ptr(n)))


def window_prefill(q, k, v, beta, lam, window, S0=None, *, mode="falcon3", phi="identity",
                   eps=1e-6, k_init=None, win_in=None, win_out=None, o=None, S_T=None,
                   stream=None, rbw=False, same_pair=False):
    """Falcon-3 ("falcon3") or 3A ("falcon3a") over q, k, v [B, H, T, d] with a
    window of `window` pairs.  win_in: the window carried from an earlier call
    (as returned here), or None; win_out: tensors to receive the window after
    the last token (allocated when None).  Returns (o, S_T, win_out)."""
    B, H, T, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    if S_T is None:
        S_T = torch.empty((B, H, d, d), device=q.device, dtype=torch.float32)
    if win_out is None:
        win_out = new_window(B, H, d, window, q.device)
    shp = fw_shape(B, H, T, d, v.shape[-1])
    st = lib().fw_window_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(lam), _ptr(S0),
                                 _ptr(k_init), _window(win_in), _ptr(o), _ptr(S_T),
                                 _window(win_out), ctypes.byref(shp), int(window),
                                 DTYPES.get(q.dtype, -1), MODES[mode], PHIS[phi], float(eps),
                                 _flags(rbw, same_pair), _stream(stream))
    if st != FW_OK:
        raise FwError(st, "fw_window_prefill")
    return o, S_T, win_out


def window_step(q, k_prev, v, beta, lam, S, window, win_in=None, win_out=None, *,
                mode="falcon3", phi="identity", eps=1e-6, o=None, stream=None, rbw=False):
    """One Falcon-3 / 3A decode step for q, k_prev, v [B, H, d]; S [B, H, d, d]
    fp32 is updated in place; the window moves from win_in (None: empty) to
    win_out (allocated when None; must not be win_in).  Returns (o, win_out)."""
    B, H, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    if win_out is None:
        win_out = new_window(B, H, d, window, q.device)
    shp = fw_shape(B, H, 1, d, v.shape[-1])
    st = lib().fw_window_step(_ptr(q), _ptr(k_prev), _ptr(v), _ptr(beta), _ptr(lam), _ptr(S),
                              _window(win_in), _ptr(o), _window(win_out), ctypes.byref(shp),
                              int(window), DTYPES.get(q.dtype, -1), MODES[mode], PHIS[phi],
                              float(eps), _flags(rbw, False), _stream(stream))
    if st != FW_OK:
        raise FwError(st, "fw_window_step")
    return o, win_out


def check(stream=None):
    """Synchronise the stream and raise if a bounded device wait ran out."""
    st = lib().fw_check(_stream(stream))
    if st != FW_OK:
        raise FwError(st, "fw_check")
