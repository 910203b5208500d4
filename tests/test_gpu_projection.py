"""GPU parity of the input projection (tcgen05 GEMMs) against its fp64 oracle,
and of the projection chained into the scan.

Tolerance: inputs are bf16, products accumulate in fp32 and each output is
rounded once to bf16 (relative error <= 2^-9 per element); against the fp64
oracle of the same bf16 inputs: L2-normwise relative error <= 5e-3 and
normwise-max relative error <= 1e-2."""
import numpy as np
import pytest
import torch

from oracle import projection
from recurrent_networks_gb300 import _lib
from recurrent_networks_gb300.synth import make_inputs

from parity_util import check_states, oracle_fwd, run_fwd

pytestmark = pytest.mark.gpu


def _close(got, ref, what):
    got = got.detach().float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all(), what
    scale = np.abs(ref).max()
    rel = np.abs(got - ref).max() / scale
    l2 = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert l2 <= 5e-3 and rel <= 1e-2, f"{what}: L2 {l2:.3g}, max {rel:.3g}"


# (BT, I, C): ragged 128-tiles in every dimension, K shorter than one 64-chunk
# (BT = 37 for dW), several K chunks, a dW long enough for split-K partials;
# the last takes 128 x 256 tiles in all three GEMMs (dW split three ways)
# with ragged edges in every dimension
CASES = [(256, 64, 128, True), (300, 72, 200, False), (37, 128, 96, True), (2048, 256, 768, True),
         (8192, 256, 3072, False), (8200, 1000, 3000, True)]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "BT%dI%dC%d%s" % (c[0], c[1], c[2], "-bias" if c[3] else ""))
def test_projection_parity(case):
    BT, I, C, with_bias = case
    g = torch.Generator().manual_seed(BT + I + C)
    x = torch.randn(BT, I, generator=g).to(torch.bfloat16).cuda()
    W = (torch.randn(C, I, generator=g) / I ** 0.5).to(torch.bfloat16).cuda()
    bias = torch.randn(C, generator=g).to(torch.bfloat16).cuda() if with_bias else None
    dWx = torch.randn(BT, C, generator=g).to(torch.bfloat16).cuda()
    ws = torch.empty(_lib.rnn_input_proj_workspace_size(BT, I, C), dtype=torch.uint8, device="cuda")
    Wx = torch.full((BT, C), float("nan"), dtype=torch.bfloat16, device="cuda")
    _lib.rnn_input_proj_fwd(BT, I, C, x, W, bias, Wx, ws)
    _lib.rnn_check_status(ws)
    _close(Wx, projection.fwd(x, W, bias), "Wx")
    dx = torch.full((BT, I), float("nan"), dtype=torch.bfloat16, device="cuda")
    dW = torch.full((C, I), float("nan"), dtype=torch.bfloat16, device="cuda")
    db = torch.full((C,), float("nan"), dtype=torch.bfloat16, device="cuda")
    _lib.rnn_input_proj_bwd(BT, I, C, x, W, dWx, dx, dW, db, ws)
    _lib.rnn_check_status(ws)
    rdx, rdW, rdb = projection.bwd(x, W, dWx)
    _close(dx, rdx, "dx")
    _close(dW, rdW, "dW")
    _close(db, rdb, "dbias")


def test_projection_rejects_bad_sizes():
    x = torch.zeros(8, 60, dtype=torch.bfloat16, device="cuda")
    assert _lib.rnn_input_proj_workspace_size(8, 60, 128) == 0
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.RnnError):
        _lib.rnn_input_proj_fwd(8, 60, 128, x, x, None, x, ws)


def test_projection_chained_into_the_scan():
    """x -> Wx (tensor-core projection, bf16) -> cluster scan, against the
    oracle projection chained into the oracle scan."""
    B, T, N, D, I = 6, 40, 2, 64, 96
    G = 4
    g = torch.Generator().manual_seed(77)
    x = torch.randn(B, T, I, generator=g).to(torch.bfloat16).cuda()
    W = (torch.randn(G * N * D, I, generator=g) / I ** 0.5).to(torch.bfloat16).cuda()
    bias = torch.randn(G * N * D, generator=g).to(torch.bfloat16).cuda()
    inp = make_inputs("lstm", B, T, N, D, torch.bfloat16, seed=78, device="cuda")
    BT, C = B * T, G * N * D
    ws = torch.empty(_lib.rnn_input_proj_workspace_size(BT, I, C), dtype=torch.uint8, device="cuda")
    Wx = torch.empty((B, T, G, N, D), dtype=torch.bfloat16, device="cuda")
    _lib.rnn_input_proj_fwd(BT, I, C, x, W, bias, Wx, ws)
    inp["Wx"] = Wx
    st, last, _ = run_fwd("lstm", inp, "auto")
    ref_wx = projection.fwd(x.reshape(BT, I), W, bias).reshape(B, T, G, N, D)
    ref = dict(inp)
    ref["Wx"] = ref_wx
    ref_st, _ = oracle_fwd("lstm", ref)
    check_states("lstm", torch.bfloat16, st, ref_st)
