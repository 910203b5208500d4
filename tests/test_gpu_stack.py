"""Stacked layers on the GPU (tensor-core input projection + scan per layer,
autograd chaining the kernels' backward passes) against the chained fp64
oracle (oracle/stack.py, itself pinned to torch.nn.LSTM(num_layers=2)).

Tolerances (bf16 storage through two layers): the last layer's h within the
stated 3e-2 max-abs; every gradient within 3e-2 L2-normwise relative error
and cosine >= 0.999 of the plain oracle. Each layer adds one bf16 rounding of
Wx and of h on top of the single-layer error budget of 2e-2."""
import numpy as np
import pytest
import torch

from oracle import stack
from recurrent_networks_gb300.functional import flashrnn_stack

pytestmark = pytest.mark.gpu


def _l2(got, ref):
    got = got.detach().float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64).reshape(got.shape)
    l2 = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    cos = float((got * ref).sum() / (np.linalg.norm(got) * np.linalg.norm(ref) + 1e-300))
    return l2, cos


@pytest.mark.parametrize("fn,N", [("lstm", 2), ("gru", 1), ("slstm", 1)])
def test_two_layer_stack_matches_chained_oracle(fn, N):
    B, T, I, D = 5, 24, 72, 64
    G = {"lstm": 4, "gru": 3, "slstm": 4}[fn]
    S = {"lstm": 2, "gru": 1, "slstm": 4}[fn]
    g = torch.Generator().manual_seed(31)
    bf = lambda t: t.to(torch.bfloat16).cuda().requires_grad_(True)
    x = bf(torch.randn(B, T, I, generator=g))
    layers = []
    for l in range(2):
        Il = I if l == 0 else N * D
        s0 = torch.randn(S, B, 1, N, D, generator=g)
        if fn == "slstm":
            s0[2], s0[3] = 1.0, 0.0
        layers.append(dict(W_x=bf(torch.randn(G * N * D, Il, generator=g) / Il ** 0.5),
                           bias_x=bf(torch.randn(G * N * D, generator=g) * 0.1),
                           R=bf(torch.randn(G, N, D, D, generator=g) / D ** 0.5),
                           b=bf(torch.randn(G, N, D, generator=g)),
                           states=bf(s0)))
    h, outs = flashrnn_stack(x, layers, fn)
    dh = torch.randn(B, T, N * D, generator=g).to(torch.bfloat16).cuda()
    h.backward(dh)

    ref_h, _, _ = stack.fwd(fn, x, layers)
    err_h = np.abs(h.detach().float().cpu().numpy() - ref_h).max()
    assert err_h <= 3e-2, err_h
    ref_dx, ref_grads = stack.bwd(fn, x, layers, dh)
    l2, cos = _l2(x.grad, ref_dx)
    assert l2 <= 3e-2 and cos >= 0.999, ("dx", l2, cos)
    for l in range(2):
        for k in ("W_x", "bias_x", "R", "b", "states"):
            l2, cos = _l2(layers[l][k].grad, ref_grads[l][k])
            assert l2 <= 3e-2 and cos >= 0.999, (l, k, l2, cos)
