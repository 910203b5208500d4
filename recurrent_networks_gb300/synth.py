"""Seeded synthetic inputs for the head-wise recurrent scan (shared by the
tests, the benchmark and the oracle side; no arithmetic of the method here).

Recipe (the workloads the scan is measured on): Wx ~ N(0,1) [B,T,G,N,D],
R ~ N(0,1/D) [G,N,D,D], b ~ N(0,1) [G,N,D], initial states ~ N(0,1)
[S,B,1,N,D] (sLSTM: normaliser n = 1 and stabiliser m = 0 exactly), upstream
gradients ~ N(0,1) on all states [S,B,T,N,D]. Drawn in fp32 on the CPU from
torch.Generator().manual_seed(seed) in the order Wx, R, b, states0, dstates,
then cast to the storage dtype.
"""
from __future__ import annotations

import math

import torch

GATES = {"lstm": 4, "gru": 3, "elman": 1, "slstm": 4, "slstm_logsig": 4}
STATES = {"lstm": 2, "gru": 1, "elman": 1, "slstm": 4, "slstm_logsig": 4}

# The five measured workloads. Seeds are 1000 + index.
WORKLOADS = {
    1: dict(name="lstm_f32_B2_T16_N1_D32", fns=("lstm",), dtype=torch.float32,
            B=2, T=16, N=1, D=32, backward=True),
    2: dict(name="lstm_bf16_B8_T1024_N3_D256", fns=("lstm",), dtype=torch.bfloat16,
            B=8, T=1024, N=3, D=256, backward=True),
    3: dict(name="gru_elman_bf16_B16_T1024_N4_D128", fns=("gru", "elman"), dtype=torch.bfloat16,
            B=16, T=1024, N=4, D=128, backward=False),
    4: dict(name="slstm_bf16_B16_T2048_N4_D192", fns=("slstm",), dtype=torch.bfloat16,
            B=16, T=2048, N=4, D=192, backward=True),
    5: dict(name="lstm_bf16_B32_T4096_N1_D1024", fns=("lstm",), dtype=torch.bfloat16,
            B=32, T=4096, N=1, D=1024, backward=True),
}


def make_inputs(function: str, B: int, T: int, N: int, D: int, dtype=torch.bfloat16,
                seed: int = 0, with_grads: bool = True, device: str | torch.device = "cpu"):
    """Returns dict(Wx, R, b, states0, dstates) (dstates None unless with_grads)."""
    G, S = GATES[function], STATES[function]
    g = torch.Generator().manual_seed(seed)
    Wx = torch.randn((B, T, G, N, D), generator=g)
    R = torch.randn((G, N, D, D), generator=g) / math.sqrt(D)
    b = torch.randn((G, N, D), generator=g)
    s0 = torch.randn((S, B, 1, N, D), generator=g)
    if function.startswith("slstm"):
        s0[2] = 1.0
        s0[3] = 0.0
    dst = torch.randn((S, B, T, N, D), generator=g) if with_grads else None
    out = dict(Wx=Wx, R=R, b=b, states0=s0, dstates=dst)
    return {k: (v.to(dtype).to(device) if v is not None else None) for k, v in out.items()}


def workload_inputs(index: int, function: str | None = None, with_grads: bool | None = None,
                    device="cpu"):
    w = WORKLOADS[index]
    fn = function or w["fns"][0]
    wg = w["backward"] if with_grads is None else with_grads
    return make_inputs(fn, w["B"], w["T"], w["N"], w["D"], w["dtype"], seed=1000 + index,
                       with_grads=wg, device=device)
