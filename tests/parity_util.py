"""Shared helpers of the parity tests: run the CUDA path through the C ABI,
run the oracle, compare with the stated tolerances.

Tolerances (stated once, used by every parity test):
  fp32 storage: max |err| <= 1e-4 on every state; gradients normwise-max
                relative error max|g - g*| / max|g*| <= 1e-3; reference = the
                plain fp64 oracle.
  bf16 storage (fp32 arithmetic): states against the plain fp64 oracle:
                max |err| <= 3e-2 on h, other states |err| <= 3e-2 * max(1,|ref|)
                (bf16 keeps 8 significant bits). Gradients against the oracle
                in its bfloat16-operand mode (the contraction operands h and
                dr rounded to bf16, as the kernels' tensor-core operands are):
                L2-normwise relative ||g - g*|| / ||g*|| <= 2e-2 and cosine
                >= 0.9995 for every cell, and normwise-max relative <= 2e-2 for
                the cells whose gradient is continuous (LSTM, GRU, Elman).
                sLSTM is exempt from the max-norm bound: the derivative of its
                stabiliser max(a_f + m, a_i) jumps at ties, and bf16 rounding of
                h (plus fp32 summation order) moves near-ties to the other branch,
                which changes single elements of dWx by O(|dm|) and, through the
                carried dm, earlier steps too. The L2 / cosine bounds therefore
                widen to 1.5x the oracle's own distance between its bf16-operand
                and plain-fp64 gradients whenever that is larger: 3-5% L2 for
                sLSTM at D = 192..512, ~0.1% for LSTM (check_grads).
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle
from recurrent_networks_gb300 import _lib

TOL = {
    torch.float32: dict(h=1e-4, states=1e-4, states_rel=False, grad=1e-3, cos=None),
    torch.bfloat16: dict(h=3e-2, states=3e-2, states_rel=True, grad=2e-2, cos=0.9995),
}


def run_fwd(fn, inp, path="auto", want_tape=True, stream=None):
    Wx, R, b, s0 = (inp[k] for k in ("Wx", "R", "b", "states0"))
    B, T, G, N, D = Wx.shape
    S = _lib.rnn_num_states(fn)
    dims = _lib.make_dims(B, T, N, D, fn, Wx.dtype, path)
    states = torch.full((S, B, T, N, D), float("nan"), dtype=Wx.dtype, device=Wx.device)
    last = torch.full((S, B, 1, N, D), float("nan"), dtype=Wx.dtype, device=Wx.device)
    tape = torch.empty(_lib.rnn_tape_size(dims), dtype=torch.uint8, device=Wx.device) if want_tape else None
    ws = torch.empty(_lib.rnn_workspace_size(dims, _lib.WS_FWD), dtype=torch.uint8, device=Wx.device)
    _lib.rnn_fwd(dims, Wx, R, b, s0, states, last, tape, ws, stream)
    _lib.rnn_check_status(ws, stream)
    return states, last, tape


def run_bwd(fn, inp, states, tape, path="auto", dlast=None):
    Wx, R, b, s0, dst = (inp[k] for k in ("Wx", "R", "b", "states0", "dstates"))
    B, T, G, N, D = Wx.shape
    dims = _lib.make_dims(B, T, N, D, fn, Wx.dtype, path)
    kind = _lib.WS_BWD if tape is not None else _lib.WS_BWD_RECOMPUTE
    ws = torch.empty(_lib.rnn_workspace_size(dims, kind), dtype=torch.uint8, device=Wx.device)
    dWx = torch.full_like(Wx, float("nan"))
    dR = torch.full_like(R, float("nan"))
    db = torch.full_like(b, float("nan"))
    ds0 = torch.full_like(s0, float("nan")) if s0 is not None else None
    _lib.rnn_bwd(dims, Wx, R, b, s0, states, tape, dst, dlast, dWx, dR, db, ds0, ws)
    _lib.rnn_check_status(ws)
    return dWx, dR, db, ds0


def to_np(t):
    return t.detach().float().cpu().double().numpy()


def check_states(fn, dtype, got, ref, what="states", calib=None):
    """h against the stated bound; the other states (c, n, m) against theirs.
    calib: the oracle's states in its bfloat16-operand mode for the same
    inputs. Over long sequences the rounding of h to bf16 alone moves the
    integrating states (sLSTM c, n, m over 2048 steps: ~10% of max(1, |x|));
    the bound on those states then widens to 1.5x the oracle's own distance
    between its bf16-operand and plain-fp64 states, as for the gradients."""
    tol = TOL[dtype]
    got = to_np(got)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err_h = np.abs(got[0] - ref[0]).max() if got[0].size else 0.0
    assert err_h <= tol["h"], f"{fn} {what} h: max abs err {err_h:.3g} > {tol['h']}"
    for s in range(1, got.shape[0]):
        den = np.maximum(1.0, np.abs(ref[s])) if tol["states_rel"] else 1.0
        e = np.abs(got[s] - ref[s]) / den
        m = e.max() if e.size else 0.0
        bound = tol["states"]
        if calib is not None and e.size:
            bound = max(bound, 1.5 * float((np.abs(calib[s] - ref[s]) / den).max()))
        assert m <= bound, f"{fn} {what} state {s}: err {m:.3g} > {bound:.3g}"
    return err_h


def grad_errors(got, ref):
    """(normwise-max relative, L2-normwise relative, cosine) of got vs ref."""
    got = to_np(got) if not isinstance(got, np.ndarray) else got
    scale = np.abs(ref).max()
    rel = np.abs(got - ref).max() / scale if scale > 0 else float(np.abs(got).max())
    nr = np.linalg.norm(ref)
    l2 = np.linalg.norm(got - ref) / nr if nr > 0 else float(np.linalg.norm(got))
    cos = float((got * ref).sum() / (np.linalg.norm(got) * nr + 1e-300)) if got.size > 1 else 1.0
    return float(rel), float(l2), cos


def check_grad(name, dtype, got, ref):
    tol = TOL[dtype]
    got = to_np(got)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    scale = np.abs(ref).max()
    if scale == 0:
        assert np.abs(got).max() == 0, f"{name}: expected zeros"
        return 0.0
    rel, l2, cos = grad_errors(got, ref)
    continuous = not name.startswith("slstm")
    if dtype == torch.float32 or continuous:
        assert rel <= tol["grad"], f"{name}: normwise-max relative err {rel:.3g} > {tol['grad']}"
    if tol["cos"] is not None and got.size > 1:
        assert l2 <= tol["grad"], f"{name}: L2-normwise relative err {l2:.3g} > {tol['grad']}"
        assert cos >= tol["cos"], f"{name}: cosine {cos:.6f} < {tol['cos']}"
    return rel


def check_grads(fn, inp, got, dlast=None):
    """All four gradients (dWx, dR, db, dstates0) of the CUDA path against the
    oracle. fp32: the TOL bounds against the plain oracle. bf16: against the
    oracle's bfloat16-operand mode; the L2 / cosine bounds widen to 1.5x the
    distance between the oracle's own bf16-operand and plain-fp64 gradients
    when that is larger (the gradient's sensitivity to bf16 rounding of h: a
    few percent for sLSTM, whose stabiliser max flips branch at near-ties,
    ~0.1% for LSTM)."""
    names = ("dWx", "dR", "db", "dstates0")
    dtype = inp["Wx"].dtype
    ref = oracle_bwd(fn, inp, dlast=dlast)
    plain = oracle_bwd(fn, inp, dlast=dlast, round_bf16=False) if dtype == torch.bfloat16 else None
    for k, (name, g) in enumerate(zip(names, got)):
        if g is None:
            continue
        if plain is None:
            check_grad(f"{fn} {name}", dtype, g, ref[k])
            continue
        tol = TOL[dtype]
        arr = to_np(g)
        assert np.all(np.isfinite(arr)), f"{fn} {name}: non-finite values"
        if np.abs(ref[k]).max() == 0:
            assert np.abs(arr).max() == 0, f"{fn} {name}: expected zeros"
            continue
        _, l2_s, cos_s = grad_errors(plain[k], ref[k])
        rel, l2, cos = grad_errors(arr, ref[k])
        l2_tol = max(tol["grad"], 1.5 * l2_s)
        cos_tol = min(tol["cos"], 1.0 - 1.5 * (1.0 - cos_s))
        if not fn.startswith("slstm"):
            assert rel <= tol["grad"], f"{fn} {name}: normwise-max relative err {rel:.3g} > {tol['grad']}"
        assert l2 <= l2_tol, f"{fn} {name}: L2-normwise relative err {l2:.3g} > {l2_tol:.3g}"
        assert cos >= cos_tol, f"{fn} {name}: cosine {cos:.6f} < {cos_tol:.6f}"


def is_bf16(inp):
    return inp["Wx"].dtype == torch.bfloat16


def oracle_fwd(fn, inp, nthreads=8, round_bf16=False):
    return oracle.fwd(fn, inp["Wx"], inp["R"], inp["b"], inp["states0"], nthreads=nthreads,
                      round_bf16=round_bf16)


def oracle_bwd(fn, inp, dlast=None, nthreads=8, round_bf16=None):
    """Gradients; for bf16 inputs the oracle runs in its bfloat16-operand mode."""
    if round_bf16 is None:
        round_bf16 = is_bf16(inp)
    return oracle.bwd(fn, inp["Wx"], inp["R"], inp["b"], inp["states0"], inp["dstates"], dlast,
                      nthreads=nthreads, round_bf16=round_bf16)
