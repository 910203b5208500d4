"""Parity at the measured workloads' full sizes, in the launch configuration the
benchmark times (the planner's automatic choice: cluster kernels for D <= 256,
the cooperative grid kernels for D = 1024).

Batch rows are independent sequences. So the oracle runs on a sample of
them (the first and the last batch row, every head, all T steps), and the
matching slices of the GPU's full-batch outputs must agree with it within
tests/parity_util.py's tolerances. dR and db sum over every batch row; they
are checked by a property that holds at any size: they equal the fp32
contraction of the GPU's own h_{t-1} with its own recurrent-branch
gradients (dr = dWx for LSTM and sLSTM)."""
import numpy as np
import pytest
import torch

from recurrent_networks_gb300 import _lib
from recurrent_networks_gb300.synth import WORKLOADS, workload_inputs

from parity_util import check_grads, check_states, oracle_fwd, run_bwd, run_fwd

pytestmark = pytest.mark.gpu

CASES = [(2, "lstm"), (3, "gru"), (3, "elman"), (4, "slstm"), (5, "lstm")]


def _rows(inp, rows):
    out = {}
    for k, v in inp.items():
        if v is None or k in ("R", "b"):
            out[k] = v
        elif k == "Wx":
            out[k] = v[rows]
        else:  # [S, B, ...]
            out[k] = v[:, rows]
    return out


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"w{c[0]}-{c[1]}")
def test_workload_full_size(case):
    k, fn = case
    w = WORKLOADS[k]
    B, T, N, D = w["B"], w["T"], w["N"], w["D"]
    inp = workload_inputs(k, function=fn, device="cuda")
    dims = _lib.make_dims(B, T, N, D, fn, w["dtype"], "auto")
    rc, plan = _lib.rnn_plan_describe(dims)
    assert rc == 0 and ("path=fused" in plan or "path=grid" in plan), plan
    st, last, tape = run_fwd(fn, inp, "auto")
    rows = [0, B - 1]
    sub = _rows(inp, rows)
    ref_st, ref_last = oracle_fwd(fn, sub, nthreads=8)
    cal_st, cal_last = oracle_fwd(fn, sub, nthreads=8, round_bf16=True) if w["dtype"] == torch.bfloat16 else (None, None)
    check_states(fn, w["dtype"], st[:, rows], ref_st, calib=cal_st)
    check_states(fn, w["dtype"], last[:, rows], ref_last, "last", calib=cal_last)
    if not w["backward"]:
        return
    dWx, dR, db, ds0 = run_bwd(fn, inp, st, tape, "auto")
    check_grads(fn, sub, (dWx[rows], None, None, ds0[:, rows]))
    # dR[g, n] = sum_{b,t} h_{t-1}[b, n, :]^T dr[b, t, g, n, :], db = sum dr
    h = st[0].float()                                          # [B, T, N, D]
    hprev = torch.cat([inp["states0"][0].float(), h[:, :-1]], dim=1)  # [B, T, N, D]
    dr = dWx.float()                                           # [B, T, G, N, D]
    G = dr.shape[2]
    for g in range(G):
        for n in range(N):
            ref = hprev[:, :, n, :].reshape(B * T, D).t() @ dr[:, :, g, n, :].reshape(B * T, D)
            got = dR[g, n].float()
            rel = ((got - ref).norm() / ref.norm()).item()
            assert rel <= 1e-2, (g, n, rel)
    ref_db = dr.sum(dim=(0, 1))
    rel = ((db.float() - ref_db).norm() / ref_db.norm()).item()
    assert rel <= 1e-2, rel
    assert np.isfinite(dR.float().cpu().numpy()).all()
