"""rnn_bwd_noalloc: the backward for callers that cannot allocate device
memory (it uses the library's fixed device scratch instead of a workspace).
Its results must match rnn_bwd's and the oracle's, call after call, on the
cluster kernels, the plain kernel and the AUTO fallback from the grid plan.
This file is collected last so that a run stopping at its first failure has
run every other test before it."""
import ctypes

import pytest
import torch

from recurrent_networks_gb300 import _lib
from recurrent_networks_gb300.synth import make_inputs

from parity_util import check_grads, run_bwd, run_fwd


def test_oversized_problem_is_rejected_before_any_work():
    # GRU needs B*T*G*N*D bf16 gradients of scratch: 2*4096*3*4*256*2 bytes > 16 MiB
    d = _lib.make_dims(2, 4096, 4, 256, "gru", torch.bfloat16)
    lib = _lib.load()
    rc = lib.rnn_bwd_noalloc(ctypes.byref(d), 256, 256, 256, None, 256, 256, None, None, 256, None,
                             None, None, None)
    assert rc == _lib.RNN_ENOSPC


def test_argument_bounds_match_rnn_bwd():
    lib = _lib.load()
    # every function id and path id rnn_bwd accepts passes validation; paths
    # whose buffers need a workspace are refused as unsupported, not invalid
    for fn in range(5):
        d = _lib.make_dims(2, 4096, 4, 256, fn, torch.bfloat16, "auto")
        rc = lib.rnn_bwd_noalloc(ctypes.byref(d), 256, 256, 256, None, 256, 256, None, None, None, None,
                                 None, None, None)
        assert rc == _lib.RNN_ENOSPC, fn  # dWx NULL: dr of this size does not fit, for every function
    for path in ("grid", "alternating"):
        d = _lib.make_dims(2, 8, 1, 64, "lstm", torch.bfloat16, path)
        rc = lib.rnn_bwd_noalloc(ctypes.byref(d), 256, 256, 256, None, 256, 256, None, None, 256, None,
                                 None, None, None)
        assert rc == _lib.RNN_EUNSUPPORTED, path
    for bad in (_lib.make_dims(0, 8, 1, 64), _lib.make_dims(2, 8, 1, 64, 5), _lib.make_dims(2, 8, 1, 64, "lstm",
                                                                                           torch.bfloat16, 5)):
        rc = lib.rnn_bwd_noalloc(ctypes.byref(bad), 256, 256, 256, None, 256, 256, None, None, 256, None,
                                 None, None, None)
        assert rc == _lib.RNN_EINVAL


def _noalloc(fn, inp, st, tape, want_dwx, dlast, path="auto"):
    B, T, G, N, D = inp["Wx"].shape
    dims = _lib.make_dims(B, T, N, D, fn, inp["Wx"].dtype, path)
    dWx = torch.full_like(inp["Wx"], float("nan")) if want_dwx else None
    dR = torch.full_like(inp["R"], float("nan"))
    db = torch.full_like(inp["b"], float("nan"))
    ds0 = torch.full_like(inp["states0"], float("nan"))
    _lib.rnn_bwd_noalloc(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], st, tape,
                         inp["dstates"], dlast, dWx, dR, db, ds0)
    _lib.rnn_bwd_noalloc_status()
    return dWx, dR, db, ds0


def _close_to_rnn_bwd(name, got, ref, dtype):
    """Same kernels as rnn_bwd: dWx and dstates0 bit-identical; dR and db may
    take their fp32 sums in another order (split-K partials or not)."""
    for k, (g, r) in enumerate(zip(got, ref)):
        if g is None:
            continue
        if k in (0, 3):
            assert torch.equal(g, r), f"{name}: {('dWx', 'dR', 'db', 'dstates0')[k]} differs from rnn_bwd"
        else:
            scale = r.float().abs().max().item()
            err = (g.float() - r.float()).abs().max().item()
            tol = (1e-5 if dtype == torch.float32 else 1e-2) * max(scale, 1e-30)
            assert err <= tol, f"{name}: {('dWx', 'dR', 'db', 'dstates0')[k]} err {err:.3g} > {tol:.3g}"


NOALLOC_CASES = [
    # (fn, B, T, N, D, dtype, want dWx, with dlast)
    ("gru", 5, 23, 2, 64, torch.bfloat16, True, False),
    ("lstm", 5, 23, 2, 64, torch.bfloat16, False, True),
    ("slstm", 5, 23, 2, 64, torch.bfloat16, True, False),
    ("slstm_logsig", 5, 23, 2, 64, torch.bfloat16, True, True),
    ("elman", 4, 17, 1, 128, torch.bfloat16, True, True),
    ("lstm", 2, 16, 1, 32, torch.float32, True, True),
    ("gru", 2, 16, 1, 32, torch.float32, True, False),
    ("lstm", 3, 9, 1, 1024, torch.bfloat16, True, False),   # AUTO plans the grid kernels: plain kernel here
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", NOALLOC_CASES, ids=lambda c: "%s-B%dT%dN%dD%d-%s-dwx%d-dlast%d" % (
    c[0], c[1], c[2], c[3], c[4], "f32" if c[5] == torch.float32 else "bf16", c[6], c[7]))
def test_noalloc_matches_rnn_bwd_and_oracle_two_calls(case):
    fn, B, T, N, D, dtype, want_dwx, with_dlast = case
    for call, seed in enumerate((11, 12)):  # two calls in a row, different inputs
        inp = make_inputs(fn, B, T, N, D, dtype, seed=seed, device="cuda")
        st, last, tape = run_fwd(fn, inp, "auto")
        dl = (torch.randn(last.shape, generator=torch.Generator().manual_seed(seed)).to(dtype).cuda()
              if with_dlast else None)
        got = _noalloc(fn, inp, st, tape, want_dwx, dl)
        check_grads(fn, inp, got, dlast=dl)
        if D <= 256:  # the same kernels as rnn_bwd (the grid plan's fallback is checked by the oracle alone)
            ref = run_bwd(fn, inp, st, tape, "auto", dlast=dl)
            _close_to_rnn_bwd(f"{fn} call {call}", got, ref, dtype)


@pytest.mark.gpu
def test_noalloc_zero_length_matches_rnn_bwd():
    fn, B, N, D = "lstm", 3, 2, 64
    inp = make_inputs(fn, B, 0, N, D, torch.bfloat16, seed=5, device="cuda")
    st, last, tape = run_fwd(fn, inp, "auto")
    dl = torch.randn(last.shape, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).cuda()
    got = _noalloc(fn, inp, st, tape, True, dl)
    ref = run_bwd(fn, inp, st, tape, "auto", dlast=dl)
    for g, r in zip(got[1:], ref[1:]):
        assert torch.equal(g, r)
    assert torch.equal(got[3], dl)
