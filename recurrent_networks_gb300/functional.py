"""The functional entry point, shaped like the FlashRNN announcement's usage
example (hottg.com/neural/9889): ``states, last = flashrnn(Wx, R, b, states=...,
function=..., backend=...)`` with no parameters bound to the function.

PyTorch provides memory, streams and autograd bookkeeping only; the forward and
the backward through time run in librnn_gb300.so's kernels via the C ABI.
"""
from __future__ import annotations

import torch

from . import _lib

BACKENDS = {"auto": "auto", "cuda_fused": "fused", "fused": "fused", "cuda": "alternating",
            "alternating": "alternating", "simt": "simt", "grid": "grid"}


def _dims(Wx, R, function, backend):
    B, T, G, N, D = Wx.shape
    if G != _lib.rnn_num_gates(function):
        raise ValueError(f"{function} needs G={_lib.rnn_num_gates(function)} gates, Wx has {G}")
    if tuple(R.shape) != (G, N, D, D):
        raise ValueError(f"R must be [G,N,D,D]={(G, N, D, D)}, got {tuple(R.shape)}")
    if Wx.dtype not in _lib.DTYPES:
        raise TypeError(f"unsupported dtype {Wx.dtype}")
    return _lib.make_dims(B, T, N, D, function, Wx.dtype, BACKENDS[backend])


def _ws(dims, kind, device):
    n = _lib.rnn_workspace_size(dims, kind)
    return torch.empty(n, dtype=torch.uint8, device=device)


class _ScanFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, Wx, R, b, states0, function, backend):
        dims = _dims(Wx, R, function, backend)
        S = _lib.rnn_num_states(function)
        B, T, G, N, D = Wx.shape
        Wx, R, b = Wx.contiguous(), R.contiguous(), b.contiguous()
        s0 = states0.contiguous() if states0 is not None else None
        states = torch.empty((S, B, T, N, D), dtype=Wx.dtype, device=Wx.device)
        last = torch.empty((S, B, 1, N, D), dtype=Wx.dtype, device=Wx.device)
        need_grad = any(ctx.needs_input_grad[:4])
        tape = torch.empty(_lib.rnn_tape_size(dims), dtype=torch.uint8, device=Wx.device) if need_grad else None
        ws = _ws(dims, _lib.WS_FWD, Wx.device)
        _lib.rnn_fwd(dims, Wx, R, b, s0, states, last, tape, ws)
        ctx.dims = dims
        ctx.has_s0 = s0 is not None
        ctx.save_for_backward(Wx, R, b, s0, states, tape)
        return states, last

    @staticmethod
    def backward(ctx, dstates, dlast):
        Wx, R, b, s0, states, tape = ctx.saved_tensors
        dims = ctx.dims
        dstates = dstates.contiguous() if dstates is not None else None
        dlast = dlast.contiguous() if dlast is not None else None
        dWx = torch.empty_like(Wx) if ctx.needs_input_grad[0] else None
        dR = torch.empty_like(R) if ctx.needs_input_grad[1] else None
        db = torch.empty_like(b) if ctx.needs_input_grad[2] else None
        ds0 = torch.empty_like(s0) if (ctx.has_s0 and ctx.needs_input_grad[3]) else None
        ws = _ws(dims, _lib.WS_BWD, Wx.device)
        _lib.rnn_bwd(dims, Wx, R, b, s0, states, tape, dstates, dlast, dWx, dR, db, ds0, ws)
        return dWx, dR, db, ds0, None, None


def flashrnn(Wx, R, b, states=None, function: str = "lstm", backend: str = "auto"):
    """Head-wise recurrent scan. Wx [B,T,G,N,D], R [G,N,D,D], b [G,N,D],
    states [S,B,1,N,D] or None (zeros). Returns (states [S,B,T,N,D], last
    [S,B,1,N,D]). function: lstm | gru | elman | slstm. backend: auto |
    cuda_fused (fused) | cuda (alternating) | simt."""
    if not Wx.is_cuda:
        raise RuntimeError("flashrnn runs on CUDA tensors only (there is no CPU path)")
    return _ScanFn.apply(Wx, R, b, states, function, backend)


class _ProjFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, W, bias):
        BT, I = x.shape
        C = W.shape[0]
        x, W = x.contiguous(), W.contiguous()
        bias = bias.contiguous() if bias is not None else None
        Wx = torch.empty((BT, C), dtype=x.dtype, device=x.device)
        ws = torch.empty(_lib.rnn_input_proj_workspace_size(BT, I, C), dtype=torch.uint8, device=x.device)
        _lib.rnn_input_proj_fwd(BT, I, C, x, W, bias, Wx, ws)
        ctx.has_bias = bias is not None
        ctx.save_for_backward(x, W)
        return Wx

    @staticmethod
    def backward(ctx, dWx):
        x, W = ctx.saved_tensors
        BT, I = x.shape
        C = W.shape[0]
        dWx = dWx.contiguous()
        dx = torch.empty_like(x) if ctx.needs_input_grad[0] else None
        dW = torch.empty_like(W) if ctx.needs_input_grad[1] else None
        db = torch.empty((C,), dtype=x.dtype, device=x.device) if (ctx.has_bias and ctx.needs_input_grad[2]) else None
        ws = torch.empty(_lib.rnn_input_proj_workspace_size(BT, I, C), dtype=torch.uint8, device=x.device)
        _lib.rnn_input_proj_bwd(BT, I, C, x, W, dWx, dx, dW, db, ws)
        return dx, dW, db


def input_projection(x, W, bias=None):
    """Wx = x W^T (+ bias) on the tensor cores: x [..., I], W [C, I] (the
    weight_ih layout), bias [C] or None; returns [..., C]. bf16, CUDA only."""
    if not x.is_cuda:
        raise RuntimeError("input_projection runs on CUDA tensors only (there is no CPU path)")
    lead = x.shape[:-1]
    y = _ProjFn.apply(x.reshape(-1, x.shape[-1]), W, bias)
    return y.reshape(*lead, W.shape[0])


def flashrnn_stack(x, layers, function: str = "lstm", backend: str = "auto"):
    """Stacked layers: layer l projects its input (x for l = 0, the previous
    layer's h, [B, T, N*D], otherwise) with W_x [G*N*D, I_l] (+ bias_x) and
    runs the head-wise scan with R, b and initial states (or zeros).
    layers: sequence of dicts with keys W_x, bias_x (optional), R, b, states
    (optional). Returns (h of the last layer [B, T, N*D], [(states, last) of
    every layer]). Differentiable end to end (autograd chains the kernels'
    backward passes)."""
    B, T = x.shape[0], x.shape[1]
    h = x
    outs = []
    for layer in layers:
        R = layer["R"]
        G, N, D = R.shape[0], R.shape[1], R.shape[2]
        Wx = input_projection(h, layer["W_x"], layer.get("bias_x")).reshape(B, T, G, N, D)
        states, last = flashrnn(Wx, R, layer["b"], layer.get("states"), function, backend)
        outs.append((states, last))
        h = states[0].reshape(B, T, N * D)
    return h, outs
