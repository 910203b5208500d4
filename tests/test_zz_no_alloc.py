"""rnn_bwd_noalloc: the backward for callers that cannot allocate device
memory (it uses the library's fixed device scratch instead of a workspace).
Its results must equal those of rnn_bwd, call after call."""
import ctypes

import pytest
import torch

from recurrent_networks_gb300 import _lib
from recurrent_networks_gb300.synth import make_inputs

from parity_util import check_grad, run_bwd, run_fwd, to_np


def test_oversized_problem_is_rejected_before_any_work():
    # GRU needs B*T*G*N*D bf16 gradients of scratch: 2*4096*3*4*256*2 bytes > 16 MiB
    d = _lib.make_dims(2, 4096, 4, 256, "gru", torch.bfloat16)
    lib = _lib.load()
    rc = lib.rnn_bwd_noalloc(ctypes.byref(d), 256, 256, 256, None, 256, 256, None, None, 256, None,
                             None, None, None)
    assert rc == _lib.RNN_ENOSPC


@pytest.mark.gpu
@pytest.mark.parametrize("fn,want_dwx", [("gru", True), ("lstm", False), ("slstm", True)])
def test_noalloc_matches_rnn_bwd_two_calls(fn, want_dwx):
    B, T, N, D = 5, 23, 2, 64
    for call, seed in enumerate((11, 12)):  # two calls in a row, different inputs
        inp = make_inputs(fn, B, T, N, D, torch.bfloat16, seed=seed, device="cuda")
        st, last, tape = run_fwd(fn, inp, "auto")
        ref = run_bwd(fn, inp, st, tape, "auto")
        dims = _lib.make_dims(B, T, N, D, fn, torch.bfloat16, "auto")
        dWx = torch.full_like(inp["Wx"], float("nan")) if want_dwx else None
        dR = torch.full_like(inp["R"], float("nan"))
        db = torch.full_like(inp["b"], float("nan"))
        ds0 = torch.full_like(inp["states0"], float("nan"))
        _lib.rnn_bwd_noalloc(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], st, tape,
                             inp["dstates"], None, dWx, dR, db, ds0)
        torch.cuda.synchronize()
        got = (dWx, dR, db, ds0)
        for name, g, r in zip(("dWx", "dR", "db", "dstates0"), got, ref):
            if g is None:
                continue
            check_grad(f"{fn} {name} (call {call})", torch.bfloat16, g, to_np(r))
