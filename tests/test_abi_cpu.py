"""Host-side checks of the C ABI that need no GPU: the library loads and
exports every function include/fw.h declares, and argument validation rejects
bad calls before touching any device.

The validation tests pass small fake addresses; they are skipped when a GPU
is visible so that no fake pointer could ever reach a launch.
"""
import ctypes
import os
import re

import pytest
import torch

from linear_token_mixer_gb300 import build as B
from linear_token_mixer_gb300 import fw

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    B.build()
    return fw.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fw.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fw_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_binding_exports():
    assert set(declared_functions()) == set(fw.EXPORTS)


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_version_and_status_strings(L):
    assert L.fw_version() == 120
    for code, name in fw.STATUS.items():
        assert L.fw_status_string(code).decode().startswith(name)
    assert L.fw_status_string(12345) == b"unknown status"


no_gpu = pytest.mark.skipif(torch.cuda.is_available(),
                            reason="fake-pointer validation checks run only without a GPU")

A = 0x10000        # fake, 16-byte aligned addresses: validation never dereferences
P = [A + 0x100000 * i for i in range(12)]


def call_prefill(L, q=P[0], k=P[1], v=P[2], beta=P[3], lam=P[4], S0=None, k_init=None, o=P[5],
                 S_T=P[6], shape=(1, 1, 8, 64, 64), dtype=1, mode=0, phi=0, eps=1e-6,
                 flags=0, algo=0):
    shp = fw.fw_shape(*shape) if shape is not None else None
    return L.fw_prefill_ex(q, k, v, beta, lam, S0, k_init, o, S_T,
                           ctypes.byref(shp) if shp is not None else None,
                           dtype, mode, phi, eps, flags, algo, None)


@no_gpu
@pytest.mark.parametrize("kw,code", [
    (dict(shape=None), -1), (dict(q=None), -1), (dict(o=None), -1), (dict(S_T=None), -1),
    (dict(beta=None), -1), (dict(lam=None), -1),
    (dict(shape=(0, 1, 8, 64, 64)), -2), (dict(shape=(1, 0, 8, 64, 64)), -2),
    (dict(shape=(1, 1, 0, 64, 64)), -2), (dict(shape=(1, 1, 8, 96, 96)), -2),
    (dict(shape=(1, 1, 8, 64, 128)), -2), (dict(shape=(1, 1, 8, 32, 32)), -2),
    (dict(dtype=7), -3), (dict(mode=9), -5), (dict(phi=9), -5), (dict(algo=5), -5),
    (dict(flags=4), -5), (dict(flags=0x80000000), -5),
    (dict(mode=2, beta=None), -1), (dict(mode=2, lam=None), -1), (dict(mode=2, eps=-1.0), -9),
    (dict(mode=2, beta=P[3] + 4), -4), (dict(mode=3, beta=None), -1), (dict(mode=4, lam=None), -1),
    (dict(mode=5), -5), (dict(mode=3, beta=P[3] + 8), -4),
    (dict(q=P[0] + 8), -4), (dict(o=P[5] + 2), -4), (dict(S0=P[7] + 4), -4),
    (dict(k_init=P[8] + 2), -4), (dict(beta=P[3] + 4), -4),
    (dict(eps=-1.0), -9), (dict(eps=float("nan")), -9), (dict(o=P[0]), -9),
    (dict(S_T=P[1]), -9), (dict(S0=P[6] + 16), -9),
    (dict(k_init=P[5] + 16), -9), (dict(k_init=P[6] + 64), -9),   # an output overlaps k_init
])
def test_prefill_validation(L, kw, code):
    assert call_prefill(L, **kw) == code


@no_gpu
@pytest.mark.parametrize("kw", [
    dict(shape=None), dict(q=None), dict(shape=(1, 1, 0, 64, 64)), dict(dtype=7), dict(mode=9),
    dict(algo=5), dict(flags=4), dict(q=P[0] + 8), dict(eps=-1.0), dict(o=P[0]),
    dict(k_init=P[5] + 16), dict(mode=2, beta=None), dict(), dict(mode=1, beta=None, lam=None),
])
def test_prefill_noalloc_validates_as_prefill_ex(L, kw):
    # same arguments, same checks, same codes (a valid call stops at the device query here)
    args = dict(q=P[0], k=P[1], v=P[2], beta=P[3], lam=P[4], S0=None, k_init=None, o=P[5],
                S_T=P[6], shape=(1, 1, 8, 64, 64), dtype=1, mode=0, phi=0, eps=1e-6, flags=0, algo=0)
    args.update(kw)
    shp = fw.fw_shape(*args["shape"]) if args["shape"] is not None else None
    st = L.fw_prefill_noalloc(args["q"], args["k"], args["v"], args["beta"], args["lam"], args["S0"],
                              args["k_init"], args["o"], args["S_T"],
                              ctypes.byref(shp) if shp is not None else None, args["dtype"],
                              args["mode"], args["phi"], args["eps"], args["flags"], args["algo"], None)
    assert st == call_prefill(L, **kw)


@no_gpu
def test_linattn_needs_no_gates(L):
    # beta/lambda may be NULL in linear-attention mode: validation passes and the
    # call fails only at the device query (there is no GPU here).
    assert call_prefill(L, beta=None, lam=None, mode=1, dtype=7) == -3
    assert call_prefill(L, beta=None, lam=None, mode=1) in (-6, -10)


@no_gpu
def test_chunked_unsupported_shapes(L):
    # fp32 or d = 64 calls are not taken by the chunked kernel.
    assert call_prefill(L, dtype=0, shape=(1, 1, 8, 128, 128), algo=2) == -8
    assert call_prefill(L, dtype=1, shape=(1, 1, 8, 64, 64), algo=2) == -8
    # Falcon-1 with phi = elu+1 stays on the per-token kernel.
    assert call_prefill(L, dtype=1, shape=(1, 1, 8, 128, 128), phi=1, algo=2) == -8
    # so does Falcon-1A with elu+1; the read / pairing flags are taken (the call
    # then fails only at the device query, there is no GPU here)
    assert call_prefill(L, dtype=1, shape=(1, 1, 8, 128, 128), mode=2, phi=1, algo=2) == -8
    for flags in (1, 2, 3):
        assert call_prefill(L, dtype=1, shape=(1, 1, 8, 128, 128), flags=flags,
                            algo=2) in (-6, -10)
    assert call_prefill(L, dtype=1, shape=(1, 1, 8, 128, 128), mode=2, algo=2) in (-6, -10)
    # a step per value channel is taken for bf16, d = 128, phi = identity (the
    # call then fails only at the device query); fp32, d = 64 and elu+1 are not
    for mode in (3, 4):
        assert call_prefill(L, dtype=1, shape=(1, 1, 8, 128, 128), mode=mode, algo=2) in (-6, -10)
        assert call_prefill(L, dtype=0, shape=(1, 1, 8, 128, 128), mode=mode, algo=2) == -8
        assert call_prefill(L, dtype=1, shape=(1, 1, 8, 64, 64), mode=mode, algo=2) == -8
        assert call_prefill(L, dtype=1, shape=(1, 1, 8, 128, 128), mode=mode, phi=1, algo=2) == -8


@no_gpu
@pytest.mark.parametrize("kw,code", [
    (dict(shape=(1, 1, 2, 64, 64)), -2), (dict(q=None), -1), (dict(S=None), -1),
    (dict(beta=None), -1), (dict(S=P[6] + 4), -4), (dict(o=P[0]), -9), (dict(dtype=5), -3),
    (dict(mode=2, lam=None), -1), (dict(flags=8), -5), (dict(mode=7), -5),
])
def test_step_validation(L, kw, code):
    args = dict(q=P[0], k=P[1], v=P[2], beta=P[3], lam=P[4], S=P[6], o=P[5],
                shape=(2, 2, 1, 64, 64), dtype=1, mode=0, phi=0, eps=1e-6, flags=0)
    args.update(kw)
    shp = fw.fw_shape(*args["shape"])
    st = L.fw_step_ex(args["q"], args["k"], args["v"], args["beta"], args["lam"], args["S"],
                      args["o"], ctypes.byref(shp), args["dtype"], args["mode"], args["phi"],
                      args["eps"], args["flags"], None)
    assert st == code
    if args["flags"] == 0:   # fw_step is fw_step_ex with no flags
        st2 = L.fw_step(args["q"], args["k"], args["v"], args["beta"], args["lam"], args["S"],
                        args["o"], ctypes.byref(shp), args["dtype"], args["mode"], args["phi"],
                        args["eps"], None)
        assert st2 == code


@no_gpu
def test_valid_call_without_gpu_reports_cuda_error(L):
    st = call_prefill(L)
    assert st in (-6, -10)
    if st == -6:
        assert L.fw_last_cuda_error() != 0


def test_binding_refuses_cpu_tensors(L):
    x = torch.zeros(1, 1, 4, 64)
    with pytest.raises(ValueError):
        fw.prefill(x, x, x, torch.zeros(1, 1, 4), torch.zeros(1, 1, 4))


def _win(x, y, n):
    return ctypes.byref(fw.fw_window(x, y, n))


def call_window_prefill(L, q=P[0], k=P[1], v=P[2], beta=P[3], lam=P[4], S0=None, k_init=None,
                        win_in=None, o=P[5], S_T=P[6], win_out=None, shape=(1, 1, 8, 64, 64),
                        window=4, dtype=1, mode=5, phi=0, eps=1e-6, flags=0):
    shp = fw.fw_shape(*shape)
    return L.fw_window_prefill(q, k, v, beta, lam, S0, k_init, win_in, o, S_T, win_out,
                               ctypes.byref(shp), window, dtype, mode, phi, eps, flags, None)


W_IN = (P[7], P[8], P[9])
W_OUT = (P[10], P[11], P[11] + 0x80000)


@no_gpu
@pytest.mark.parametrize("kw,code", [
    (dict(mode=0), -5), (dict(mode=1), -5), (dict(mode=3), -5), (dict(mode=7), -5),
    (dict(window=0), -2), (dict(window=9), -2), (dict(flags=4), -5),
    (dict(beta=None), -1), (dict(lam=None), -1), (dict(q=None), -1), (dict(S_T=None), -1),
    (dict(eps=-1.0), -9), (dict(q=P[0] + 8), -4), (dict(k_init=P[8] + 2), -4),
    (dict(o=P[1]), -9), (dict(S_T=P[0]), -9),
    (dict(win_in=_win(P[7], None, P[9])), -1), (dict(win_out=_win(P[10], P[11], None)), -1),
    (dict(win_in=_win(P[7] + 4, P[8], P[9])), -4), (dict(win_out=_win(*W_OUT[:2], P[9] + 2)), -4),
    (dict(win_in=_win(*W_IN), win_out=_win(P[7], P[11], P[10])), -9),    # out overlaps in
    (dict(win_out=_win(P[0], P[11], P[10])), -9),                         # out overlaps q
    (dict(win_out=_win(P[10], P[10], P[11])), -9),                        # x and y overlap
    (dict(win_in=_win(P[5], P[8], P[9])), -9),                            # in overlaps o
])
def test_window_prefill_validation(L, kw, code):
    assert call_window_prefill(L, **kw) == code


@no_gpu
def test_window_prefill_valid_calls_reach_the_device_query(L):
    for kw in (dict(), dict(mode=6), dict(window=1), dict(window=8), dict(flags=3),
               dict(win_in=_win(*W_IN), win_out=_win(*W_OUT)),
               # with a window of one pair nothing is carried: the structs are not read
               dict(window=1, win_in=_win(None, None, None), win_out=_win(P[0], P[0], P[0]))):
        assert call_window_prefill(L, **kw) in (-6, -10), kw


@no_gpu
@pytest.mark.parametrize("kw,code", [
    (dict(shape=(1, 1, 2, 64, 64)), -2), (dict(window=0), -2), (dict(window=9), -2),
    (dict(mode=0), -5), (dict(flags=2), -5), (dict(q=None), -1), (dict(S=None), -1),
    (dict(beta=None), -1), (dict(S=P[6] + 4), -4), (dict(o=P[0]), -9),
    (dict(win_in=_win(*W_IN), win_out=_win(*W_IN)), -9),
    (dict(win_out=_win(P[6], P[11], P[10])), -9),                         # out overlaps S
])
def test_window_step_validation(L, kw, code):
    args = dict(q=P[0], k=P[1], v=P[2], beta=P[3], lam=P[4], S=P[6], win_in=None, o=P[5],
                win_out=None, shape=(2, 2, 1, 64, 64), window=4, dtype=1, mode=5, phi=0,
                eps=1e-6, flags=0)
    args.update(kw)
    shp = fw.fw_shape(*args.pop("shape"))
    st = L.fw_window_step(args["q"], args["k"], args["v"], args["beta"], args["lam"], args["S"],
                          args["win_in"], args["o"], args["win_out"], ctypes.byref(shp),
                          args["window"], args["dtype"], args["mode"], args["phi"], args["eps"],
                          args["flags"], None)
    assert st == code


@no_gpu
def test_window_step_valid_call_reaches_the_device_query(L):
    shp = fw.fw_shape(2, 2, 1, 64, 64)
    st = L.fw_window_step(P[0], P[1], P[2], P[3], P[4], P[6], _win(*W_IN), P[5], _win(*W_OUT),
                          ctypes.byref(shp), 4, 1, 6, 0, 1e-6, 1, None)
    assert st in (-6, -10)
