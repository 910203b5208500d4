"""Parity at the measured workloads' full sizes, in the launch configuration the
benchmark times (the planner's automatic choice: cluster kernels for D <= 256,
the cooperative grid kernels for D = 1024).

The fp64 oracle runs on every batch row, every head and every step, on all
host cores, and every output of the CUDA path is compared with it element by
element: states and last states against the plain oracle, the four gradients
(dWx, dR, db, dstates0) against its bfloat16-operand mode, with the bounds of
tests/parity_util.py. dR and db sum over all B*T (row, step) pairs, so this is
the check of the full-size weight-gradient GEMM and column sums against the
definition, not against the GPU's own intermediate values."""
import os

import numpy as np
import pytest
import torch

from oracle import oracle
from recurrent_networks_gb300 import _lib
from recurrent_networks_gb300.synth import WORKLOADS, workload_inputs

from parity_util import check_grads, check_states, run_bwd, run_fwd

pytestmark = pytest.mark.gpu

CASES = [(2, "lstm"), (3, "gru"), (3, "elman"), (4, "slstm"), (5, "lstm")]


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"w{c[0]}-{c[1]}")
def test_workload_full_size(case):
    k, fn = case
    w = WORKLOADS[k]
    B, T, N, D = w["B"], w["T"], w["N"], w["D"]
    bf16 = w["dtype"] == torch.bfloat16
    host = workload_inputs(k, function=fn)
    inp = {key: (v.cuda() if v is not None else None) for key, v in host.items()}
    dims = _lib.make_dims(B, T, N, D, fn, w["dtype"], "auto")
    rc, plan = _lib.rnn_plan_describe(dims)
    assert rc == 0 and ("path=fused" in plan or "path=grid" in plan), plan
    st, last, tape = run_fwd(fn, inp, "auto")
    nt = _cores()
    ref_st, ref_last = oracle.fwd(fn, host["Wx"], host["R"], host["b"], host["states0"], nthreads=nt)
    # the bf16-operand states calibrate the long-sequence bounds of sLSTM's c, n, m
    # (and h past the 1024 steps the stated bound covers)
    cal_st, cal_last = (oracle.fwd(fn, host["Wx"], host["R"], host["b"], host["states0"], nthreads=nt,
                                   round_bf16=True) if (bf16 and (fn.startswith("slstm") or T > 1024))
                        else (None, None))
    check_states(fn, w["dtype"], st, ref_st, calib=cal_st)
    check_states(fn, w["dtype"], last, ref_last, "last", calib=cal_last, t0=T - 1)
    del ref_st, cal_st
    if not w["backward"]:
        return
    got = run_bwd(fn, inp, st, tape, "auto")
    ref = oracle.bwd(fn, host["Wx"], host["R"], host["b"], host["states0"], host["dstates"], nthreads=nt,
                     round_bf16=bf16)
    # the widening of the bf16 bounds needs the plain gradients too: only sLSTM
    # has a distance between the two modes above the base bounds
    plain = (oracle.bwd(fn, host["Wx"], host["R"], host["b"], host["states0"], host["dstates"], nthreads=nt)
             if (bf16 and fn.startswith("slstm")) else False)
    check_grads(fn, host, got, ref=ref, plain=plain, label=w["name"])
    assert np.isfinite(got[1].float().cpu().numpy()).all()
