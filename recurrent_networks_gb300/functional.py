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
