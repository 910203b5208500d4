"""fp64 oracle of stacked layers: the input projection followed by the scan,
layer after layer (each layer's input is the previous layer's h, [B, T, N*D]),
and its backward through all layers.

TEST INFRASTRUCTURE: only the tests may import this module; it chains the
scan oracle (oracle.py) and the projection oracle (projection.py).
"""
from __future__ import annotations

import numpy as np

from . import oracle, projection


def _np(a):
    return None if a is None else projection._f64(a)


def fwd(function, x, layers, nthreads=8):
    """x [B, T, I]; layers: dicts W_x, bias_x (opt), R, b, states (opt).
    Returns (h [B, T, N*D], [(states, last)...], [Wx...]) in float64."""
    x = _np(x)
    B, T = x.shape[:2]
    h = x
    outs, wxs = [], []
    for L in layers:
        R = _np(L["R"])
        G, N, D = R.shape[:3]
        Wx = projection.fwd(h.reshape(B * T, -1), L["W_x"], L.get("bias_x")).reshape(B, T, G, N, D)
        st, last = oracle.fwd(function, Wx, R, _np(L["b"]), _np(L.get("states")), nthreads=nthreads)
        outs.append((st, last))
        wxs.append(Wx)
        h = st[0].reshape(B, T, N * D)
    return h, outs, wxs


def bwd(function, x, layers, dh, nthreads=8):
    """Gradients of sum(h_last * dh) with respect to x and every layer's
    parameters and initial states: (dx, [dict(W_x, bias_x, R, b, states)...])."""
    x = _np(x)
    B, T = x.shape[:2]
    h_last, outs, wxs = fwd(function, x, layers, nthreads)
    grads = [None] * len(layers)
    up = _np(dh)  # gradient reaching the current layer's h, [B, T, N*D]
    for l in range(len(layers) - 1, -1, -1):
        L = layers[l]
        R = _np(L["R"])
        G, N, D = R.shape[:3]
        st, _ = outs[l]
        S = st.shape[0]
        dstates = np.zeros_like(st)
        dstates[0] = up.reshape(B, T, N, D)
        dWx, dR, db, ds0 = oracle.bwd(function, wxs[l], R, _np(L["b"]), _np(L.get("states")), dstates, None,
                                      nthreads=nthreads)
        inp = x if l == 0 else outs[l - 1][0][0].reshape(B, T, -1)
        dinp, dW, dbias = projection.bwd(inp.reshape(B * T, -1), L["W_x"], dWx.reshape(B * T, -1))
        grads[l] = dict(W_x=dW, bias_x=dbias, R=dR, b=db, states=ds0)
        up = dinp.reshape(B, T, -1)
    return up, grads
