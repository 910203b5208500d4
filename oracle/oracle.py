"""Python access to the fp64 CPU oracle of the head-wise recurrent scan.

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module. The CUDA library shares no
code with it and never calls it.

The arithmetic lives in ``rnn_oracle.c`` (plain C, fp64); this file compiles it
with gcc on first use and marshals numpy arrays. Layouts and the readings of
the cells are documented in ``rnn_oracle.h`` / ``rnn_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rnn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

FUNCTIONS = {"lstm": 0, "gru": 1, "elman": 2, "slstm": 3, "slstm_logsig": 4}
GATES = {"lstm": 4, "gru": 3, "elman": 1, "slstm": 4, "slstm_logsig": 4}
STATES = {"lstm": 2, "gru": 1, "elman": 1, "slstm": 4, "slstm_logsig": 4}


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library; returns its path."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)) or (
            os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                              os.path.getmtime(os.path.join(_HERE, "rnn_oracle.h"))))
        if force or stale:
            os.makedirs(_BUILD, exist_ok=True)
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", tmp,
                                   _SRC, "-lm", "-lpthread"])
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        lib.oracle_fwd.argtypes = [i, i, i, i, i, dp, dp, dp, dp, dp, dp, i, i]
        lib.oracle_bwd.argtypes = [i, i, i, i, i, dp, dp, dp, dp, dp, dp, dp, dp, dp, dp, i, i]
        lib.oracle_fwd.restype = i
        lib.oracle_bwd.restype = i
        _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor: exact widening to fp64
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


ROUND_BF16 = 1


def fwd(function: str, Wx, R, b, states0=None, nthreads: int = 1, round_bf16: bool = False):
    """Forward scan. Wx [B,T,G,N,D], R [G,N,D,D], b [G,N,D], states0 [S,B,1,N,D]
    (None = zeros). Returns (states [S,B,T,N,D], last [S,B,1,N,D]) in fp64.
    round_bf16: the bfloat16 storage mode (contraction operands rounded to bf16)."""
    Wx, R, b, s0 = _f64(Wx), _f64(R), _f64(b), _f64(states0)
    B, T, G, N, D = Wx.shape
    S = STATES[function]
    assert G == GATES[function] and R.shape == (G, N, D, D) and b.shape == (G, N, D)
    if s0 is not None:
        assert s0.shape == (S, B, 1, N, D)
    states = np.zeros((S, B, T, N, D))
    last = np.zeros((S, B, 1, N, D))
    rc = _load().oracle_fwd(FUNCTIONS[function], B, T, N, D, _ptr(Wx), _ptr(R), _ptr(b),
                            _ptr(s0), _ptr(states), _ptr(last), ROUND_BF16 if round_bf16 else 0,
                            nthreads)
    if rc != 0:
        raise ValueError("oracle_fwd rejected its arguments")
    return states, last


def bwd(function: str, Wx, R, b, states0=None, dstates=None, dlast=None, nthreads: int = 1,
        round_bf16: bool = False):
    """Backward through time. Returns (dWx, dR, db, dstates0) in fp64."""
    Wx, R, b, s0 = _f64(Wx), _f64(R), _f64(b), _f64(states0)
    dst, dl = _f64(dstates), _f64(dlast)
    B, T, G, N, D = Wx.shape
    S = STATES[function]
    assert G == GATES[function]
    if dst is not None:
        assert dst.shape == (S, B, T, N, D)
    if dl is not None:
        assert dl.shape == (S, B, 1, N, D)
    dWx = np.zeros_like(Wx)
    dR = np.zeros((G, N, D, D))
    db = np.zeros((G, N, D))
    ds0 = np.zeros((S, B, 1, N, D))
    rc = _load().oracle_bwd(FUNCTIONS[function], B, T, N, D, _ptr(Wx), _ptr(R), _ptr(b),
                            _ptr(s0), _ptr(dst), _ptr(dl), _ptr(dWx), _ptr(dR), _ptr(db),
                            _ptr(ds0), ROUND_BF16 if round_bf16 else 0, nthreads)
    if rc != 0:
        raise ValueError("oracle_bwd rejected its arguments")
    return dWx, dR, db, ds0
