"""fp64 oracle of the input projection ahead of the scan.

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module; the CUDA library shares no
code with it.

developnotes "deep learning operators", section 5.3 LSTM (MyLSTM.forward)
forms each gate's input branch as x_t W_ih^T + b_ih before adding the recurrent
branch; the FlashRNN announcement's flashrnn() takes that product, Wx, as its
input. With W_x in the weight_ih layout [C][I] (C = G N D rows in the order of
Wx's (g, n, d) axes) and the rows m = (b, t) of the sequence:
    Wx[m, c] = sum_i x[m, i] W_x[c, i] + bias[c]
and its gradients given dWx:
    dx = dWx W_x,   dW_x = dWx^T x,   dbias = sum_m dWx[m, :].
The definition written out with a library matmul, in float64.
"""
from __future__ import annotations

import numpy as np


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor: bf16 / fp32 / fp64 convert exactly
        import torch
        a = a.detach().cpu().to(torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


def fwd(x, W, bias=None):
    """x [BT, I], W [C, I], bias [C] or None -> Wx [BT, C] (float64)."""
    x, W, bias = _f64(x), _f64(W), _f64(bias)
    out = x @ W.T
    if bias is not None:
        out = out + bias[None, :]
    return out


def bwd(x, W, dWx):
    """Gradients of sum(fwd(x, W, bias) * dWx): (dx [BT, I], dW [C, I], dbias [C])."""
    x, W, dWx = _f64(x), _f64(W), _f64(dWx)
    return dWx @ W, dWx.T @ x, dWx.sum(axis=0)
