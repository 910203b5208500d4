"""GPU parity: the CUDA path through the C ABI against the fp64 oracle,
element by element, at sizes the oracle finishes in seconds (several tiles and
ragged tails). Tolerances are those of tests/parity_util.py."""
import numpy as np
import pytest
import torch

from recurrent_networks_gb300 import _lib
from recurrent_networks_gb300.synth import make_inputs

from parity_util import (check_grad, check_grads, check_states, oracle_bwd, oracle_fwd, run_bwd, run_fwd)

pytestmark = pytest.mark.gpu

FNS = ["lstm", "gru", "elman", "slstm", "slstm_logsig"]
DTYPES = [torch.float32, torch.bfloat16]
SMALL = [(3, 37, 2, 48), (1, 5, 1, 16), (9, 20, 3, 64)]


def assert_states_close(a, b, tol=2e-2):
    """Two bf16 paths with the same arithmetic: h within tol, the other states
    within tol relative to max(1, |x|) (one bf16 ulp of a c of 8 is 0.03)."""
    a, b = a.float(), b.float()
    dh = (a[0] - b[0]).abs().max().item()
    assert dh <= tol, dh
    if a.shape[0] > 1:
        rel = ((a[1:] - b[1:]).abs() / b[1:].abs().clamp_min(1.0)).max().item()
        assert rel <= tol, rel


def _inputs(fn, shape, dtype, seed):
    B, T, N, D = shape
    return make_inputs(fn, B, T, N, D, dtype, seed=seed, device="cuda")


def _full_check(fn, inp, dtype, path, backward=True, recompute=False):
    st, last, tape = run_fwd(fn, inp, path)
    ref_st, ref_last = oracle_fwd(fn, inp)
    check_states(fn, dtype, st, ref_st)
    check_states(fn, dtype, last, ref_last, "last")
    if not backward:
        return
    dWx, dR, db, ds0 = run_bwd(fn, inp, st, None if recompute else tape, path)
    check_grads(fn, inp, (dWx, dR, db, ds0))


@pytest.mark.parametrize("fn", FNS)
@pytest.mark.parametrize("dtype", DTYPES, ids=["f32", "bf16"])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "B%dT%dN%dD%d" % s)
def test_simt_parity(fn, dtype, shape):
    inp = _inputs(fn, shape, dtype, seed=100 * FNS.index(fn) + SMALL.index(shape))
    _full_check(fn, inp, dtype, "simt")


@pytest.mark.parametrize("fn", FNS)
def test_backward_recomputes_tape(fn):
    inp = _inputs(fn, (2, 9, 1, 32), torch.float32, seed=77)
    _full_check(fn, inp, torch.float32, "auto", recompute=True)


@pytest.mark.parametrize("fn", FNS)
def test_zero_length_and_null_initial_state(fn):
    inp = _inputs(fn, (2, 0, 1, 32), torch.float32, seed=3)
    st, last, tape = run_fwd(fn, inp, "auto")
    assert st.numel() == 0
    torch.testing.assert_close(last, inp["states0"], rtol=0, atol=0)
    dl = torch.randn_like(inp["states0"])
    dWx, dR, db, ds0 = run_bwd(fn, inp, st, tape, "auto", dlast=dl)
    torch.testing.assert_close(ds0, dl, rtol=0, atol=0)
    assert not dR.any() and not db.any()
    # states0 = NULL means zeros
    inp = _inputs(fn, (2, 6, 1, 32), torch.float32, seed=4)
    st1, _, _ = run_fwd(fn, dict(inp, states0=None), "auto", want_tape=False)
    st2, _, _ = run_fwd(fn, dict(inp, states0=torch.zeros_like(inp["states0"])), "auto", want_tape=False)
    torch.testing.assert_close(st1, st2, rtol=0, atol=0)


def test_workload_1_full():
    """LSTM fp32, B=2 T=16 N=1 D=32: every element of every output."""
    from recurrent_networks_gb300.synth import workload_inputs
    inp = workload_inputs(1, device="cuda")
    _full_check("lstm", inp, torch.float32, "auto")


def test_autograd_function_matches_abi():
    from recurrent_networks_gb300 import flashrnn
    inp = _inputs("lstm", (3, 11, 2, 32), torch.float32, seed=5)
    leaves = {k: inp[k].clone().requires_grad_(True) for k in ("Wx", "R", "b", "states0")}
    st, last = flashrnn(leaves["Wx"], leaves["R"], leaves["b"], leaves["states0"], function="lstm")
    dl = torch.randn_like(last)
    ((st * inp["dstates"]).sum() + (last * dl).sum()).backward()
    ref_st, _ = oracle_fwd("lstm", inp)
    rdWx, rdR, rdb, rds0 = oracle_bwd("lstm", inp, dlast=dl.cpu().double().numpy())
    check_states("lstm", torch.float32, st, ref_st)
    check_grad("dWx", torch.float32, leaves["Wx"].grad, rdWx)
    check_grad("dR", torch.float32, leaves["R"].grad, rdR)
    check_grad("db", torch.float32, leaves["b"].grad, rdb)
    check_grad("ds0", torch.float32, leaves["states0"].grad, rds0)


# ---------------------------------------------------------------- cluster kernels
# (fn, B, T, N, D, env restriction of the planner: cluster size C, n-tiles NT, k-tiles KT)
FUSED_CASES = [
    ("lstm", 3, 37, 2, 64, dict(C=1)),
    ("lstm", 3, 37, 2, 64, dict(C=2, NT=2)),
    ("lstm", 3, 37, 2, 64, dict(C=4, KT=4)),
    ("lstm", 9, 21, 1, 128, dict(C=8)),
    ("lstm", 5, 19, 1, 256, dict(C=16)),
    ("lstm", 8, 40, 3, 256, dict(C=8, KT=4)),
    ("gru", 9, 20, 3, 48, dict(C=3)),
    ("gru", 16, 25, 2, 128, dict(C=4, NT=2)),
    ("elman", 16, 33, 1, 128, dict(C=2)),
    ("elman", 7, 18, 2, 64, dict(C=2, KT=4)),
    ("slstm", 5, 29, 2, 96, dict(C=3, KT=3)),
    ("slstm", 16, 23, 1, 192, dict(C=12, NT=2)),
    ("slstm", 4, 17, 1, 192, dict(C=12)),
    ("slstm_logsig", 6, 31, 2, 128, dict(C=8)),
]


def _restrict(monkeypatch, restr):
    for k in ("C", "NT", "KT", "MT"):
        monkeypatch.delenv(f"RNN_PLAN_{k}", raising=False)
    for k, v in restr.items():
        monkeypatch.setenv(f"RNN_PLAN_{k}", str(v))


@pytest.mark.parametrize("case", FUSED_CASES,
                         ids=lambda c: "%s-B%dT%dN%dD%d-" % c[:5] + "-".join(f"{k}{v}" for k, v in c[5].items()))
def test_fused_forward_parity(case, monkeypatch):
    fn, B, T, N, D, restr = case
    _restrict(monkeypatch, restr)
    inp = _inputs(fn, (B, T, N, D), torch.bfloat16, seed=500 + B + T + D)
    dims = _lib.make_dims(B, T, N, D, fn, torch.bfloat16, "fused")
    rc, desc = _lib.rnn_plan_describe(dims)
    assert rc == 0 and "path=fused" in desc and f"C={restr['C']} " in desc, desc
    st, last, tape = run_fwd(fn, inp, "fused")
    ref_st, ref_last = oracle_fwd(fn, inp)
    check_states(fn, torch.bfloat16, st, ref_st)
    check_states(fn, torch.bfloat16, last, ref_last, "last")
    # the backward (plain path) consumes the cluster kernel's tape
    dWx, dR, db, ds0 = run_bwd(fn, inp, st, tape, "simt")
    check_grads(fn, inp, (dWx, dR, db, ds0))


def test_fused_matches_simt_forward_closely(monkeypatch):
    """Same arithmetic (bf16 operands, fp32 accumulation) on both paths: the
    states agree far more closely than either does with the fp64 oracle."""
    _restrict(monkeypatch, dict(C=4))
    inp = _inputs("lstm", (6, 30, 2, 128), torch.bfloat16, seed=42)
    st_f, _, _ = run_fwd("lstm", inp, "fused", want_tape=False)
    st_s, _, _ = run_fwd("lstm", inp, "simt", want_tape=False)
    assert_states_close(st_f, st_s)


BWD_CASES = [
    ("lstm", 3, 37, 2, 64, dict(C=2)),
    ("lstm", 3, 37, 2, 64, dict(C=4, NT=2)),
    ("lstm", 9, 21, 1, 128, dict(C=8, MT=2)),
    ("lstm", 5, 19, 1, 256, dict(C=16)),
    ("lstm", 8, 40, 3, 256, dict(C=8)),
    ("gru", 9, 20, 3, 48, dict(C=3)),
    ("gru", 16, 25, 2, 128, dict(C=4, NT=2)),
    ("elman", 7, 18, 2, 64, dict(C=2)),
    ("elman", 16, 33, 1, 128, dict(C=2)),
    ("slstm", 5, 29, 2, 96, dict(C=3)),
    ("slstm", 16, 23, 1, 192, dict(C=12, NT=2)),
    ("slstm", 4, 17, 1, 192, dict(C=12)),
    ("slstm_logsig", 6, 31, 2, 128, dict(C=8)),
]


@pytest.mark.parametrize("case", BWD_CASES,
                         ids=lambda c: "%s-B%dT%dN%dD%d-" % c[:5] + "-".join(f"{k}{v}" for k, v in c[5].items()))
def test_fused_backward_parity(case, monkeypatch):
    fn, B, T, N, D, restr = case
    _restrict(monkeypatch, restr)
    inp = _inputs(fn, (B, T, N, D), torch.bfloat16, seed=700 + B + T + D)
    dims = _lib.make_dims(B, T, N, D, fn, torch.bfloat16, "fused")
    rc, desc = _lib.rnn_plan_describe(dims, True)
    assert rc == 0 and "path=fused" in desc and f"C={restr['C']} " in desc, desc
    st, last, tape = run_fwd(fn, inp, "fused")
    dl = torch.randn(last.shape, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16).cuda()
    dWx, dR, db, ds0 = run_bwd(fn, inp, st, tape, "fused", dlast=dl)
    check_grads(fn, inp, (dWx, dR, db, ds0), dlast=dl)
    # the plain path on the same tape gives nearly the same gradients
    sdWx, _, _, sds0 = run_bwd(fn, inp, st, tape, "simt", dlast=dl)
    d1 = (dWx.float() - sdWx.float()).abs().max().item() / max(sdWx.float().abs().max().item(), 1e-30)
    assert d1 <= 2e-2, d1


# tape = NULL: the backward rebuilds the tape inside its workspace by running the
# same forward kernels (the gate recompute), on the bf16 cluster and grid paths
RECOMPUTE_CASES = [
    ("fused", "lstm", 5, 19, 1, 256, dict(C=16)),
    ("fused", "gru", 9, 20, 3, 48, dict(C=3)),
    ("fused", "slstm", 5, 29, 2, 96, dict(C=3)),
    ("grid", "lstm", 3, 9, 1, 1024, dict(C=64)),
    ("grid", "gru", 9, 19, 2, 128, dict(C=8)),
    ("grid", "slstm_logsig", 5, 13, 1, 512, dict(C=32)),
]


@pytest.mark.parametrize("case", RECOMPUTE_CASES,
                         ids=lambda c: "%s-%s-B%dT%dN%dD%d-" % c[:6] + "-".join(f"{k}{v}" for k, v in c[6].items()))
def test_backward_recomputes_tape_bf16(case, monkeypatch):
    path, fn, B, T, N, D, restr = case
    _restrict(monkeypatch, restr)
    inp = _inputs(fn, (B, T, N, D), torch.bfloat16, seed=1100 + B + T + D)
    dims = _lib.make_dims(B, T, N, D, fn, torch.bfloat16, path)
    for bwd in (False, True):
        rc, desc = _lib.rnn_plan_describe(dims, bwd)
        assert rc == 0 and f"path={path}" in desc, desc
    st, last, tape = run_fwd(fn, inp, path)
    dl = torch.randn(last.shape, generator=torch.Generator().manual_seed(8)).to(torch.bfloat16).cuda()
    got = run_bwd(fn, inp, st, None, path, dlast=dl)
    check_grads(fn, inp, got, dlast=dl)
    # the rebuilt tape is the forward's tape: the gradients equal those taken with it
    with_tape = run_bwd(fn, inp, st, tape, path, dlast=dl)
    for name, a, b in zip(("dWx", "dR", "db", "dstates0"), got, with_tape):
        assert torch.equal(a, b), f"{name} differs between the rebuilt and the stored tape"


# ---------------------------------------------------------------- grid kernels
GRID_CASES = [
    ("lstm", 5, 23, 1, 256, dict(C=16)),
    ("lstm", 3, 9, 1, 1024, dict(C=64)),
    ("gru", 9, 19, 2, 128, dict(C=8)),
    ("elman", 16, 21, 2, 256, dict(C=16, NT=2)),
    ("slstm", 4, 17, 1, 512, dict(C=32)),
    ("slstm_logsig", 5, 13, 1, 512, dict(C=32)),
    ("lstm", 13, 9, 1, 512, dict(C=32, NT=2)),   # 16-row batch tile with 13 rows: ragged bulk-copy gathers
]


@pytest.mark.parametrize("case", GRID_CASES,
                         ids=lambda c: "%s-B%dT%dN%dD%d-" % c[:5] + "-".join(f"{k}{v}" for k, v in c[5].items()))
def test_grid_parity(case, monkeypatch):
    fn, B, T, N, D, restr = case
    _restrict(monkeypatch, restr)
    inp = _inputs(fn, (B, T, N, D), torch.bfloat16, seed=900 + B + T + D)
    dims = _lib.make_dims(B, T, N, D, fn, torch.bfloat16, "grid")
    for bwd in (False, True):
        rc, desc = _lib.rnn_plan_describe(dims, bwd)
        assert rc == 0 and "path=grid" in desc, desc
    st, last, tape = run_fwd(fn, inp, "grid")
    ref_st, ref_last = oracle_fwd(fn, inp)
    check_states(fn, torch.bfloat16, st, ref_st)
    check_states(fn, torch.bfloat16, last, ref_last, "last")
    dl = torch.randn(last.shape, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).cuda()
    dWx, dR, db, ds0 = run_bwd(fn, inp, st, tape, "grid", dlast=dl)
    check_grads(fn, inp, (dWx, dR, db, ds0), dlast=dl)


def test_grid_die_placement_changes_nothing(monkeypatch):
    """The grid kernels' die placement (each batch group's CTAs on one die of
    the GPU, its step counter homed in L2 there) only moves CTAs between SMs:
    states and gradients are bitwise those of the block-index placement, and
    both match the oracle."""
    layout = _lib.rnn_die_layout()
    if layout is None:
        pytest.skip("the device shows no two-die structure")
    assert min(layout) > 0 and sum(layout) == torch.cuda.get_device_properties(0).multi_processor_count
    _restrict(monkeypatch, dict(C=32, NT=2))
    fn, B, T, N, D = "lstm", 20, 33, 2, 512  # 2 heads x 2 batch blocks: 4 groups of 32 CTAs
    inp = _inputs(fn, (B, T, N, D), torch.bfloat16, seed=4242)
    outs = {}
    for mode in ("1", "0"):
        monkeypatch.setenv("RNN_DIE_PLACEMENT", mode)
        st, last, tape = run_fwd(fn, inp, "grid")
        outs[mode] = (st, last) + tuple(run_bwd(fn, inp, st, tape, "grid"))
    for name, a, b in zip(("states", "last", "dWx", "dR", "db", "dstates0"), outs["1"], outs["0"]):
        assert torch.equal(a, b), f"{name} differs between the die and the block-index placement"
    ref_st, _ = oracle_fwd(fn, inp)
    check_states(fn, torch.bfloat16, outs["1"][0], ref_st)
    check_grads(fn, inp, outs["1"][2:])


@pytest.mark.parametrize("fn", ["lstm", "gru"])
def test_grid_dr_beside_the_scan(fn, monkeypatch):
    """dR computed by the grid backward's spare CTAs beside the scan (chunks of
    64-step tiles, a ragged last tile, the initial-state rows, two heads and two
    batch blocks; GRU's recurrent-branch gradient in its own buffer) matches the
    oracle, and the dR GEMM after the scan within a bf16 rounding; the other
    gradients do not depend on where dR is computed."""
    _restrict(monkeypatch, dict(C=16, NT=2))
    B, T, N, D = 20, 16 * 64 + 37, 2, 256
    inp = _inputs(fn, (B, T, N, D), torch.bfloat16, seed=4545)
    st, last, tape = run_fwd(fn, inp, "grid")
    got = {}
    for mode in ("1", "0"):
        monkeypatch.setenv("RNN_DR_BESIDE", mode)
        got[mode] = run_bwd(fn, inp, st, tape, "grid")
    check_grads(fn, inp, got["1"])
    for name, a, b in zip(("dWx", "db", "dstates0"), (got["1"][0], got["1"][2], got["1"][3]),
                          (got["0"][0], got["0"][2], got["0"][3])):
        assert torch.equal(a, b), f"{name} depends on where dR is computed"
    a, b = got["1"][1].float(), got["0"][1].float()
    assert (a - b).abs().max().item() <= 1e-2 * b.abs().max().item()


def test_grid_path_in_a_cuda_graph(monkeypatch):
    """A forward and backward on the grid kernels captured into a CUDA graph
    and replayed give the eager results bit for bit: with the workspace's
    counter blocks measured before the capture (die placement inside the
    graph), and with a fresh workspace, whose capture skips the measurement
    (groups by block index)."""
    _restrict(monkeypatch, dict(C=32, NT=2))
    fn, B, T, N, D = "lstm", 20, 17, 2, 512
    inp = _inputs(fn, (B, T, N, D), torch.bfloat16, seed=4343)
    dims = _lib.make_dims(B, T, N, D, fn, torch.bfloat16, "grid")
    S = _lib.rnn_num_states(fn)

    def buffers():
        return dict(states=torch.empty((S, B, T, N, D), dtype=torch.bfloat16, device="cuda"),
                    last=torch.empty((S, B, 1, N, D), dtype=torch.bfloat16, device="cuda"),
                    tape=torch.empty(_lib.rnn_tape_size(dims), dtype=torch.uint8, device="cuda"),
                    ws=torch.empty(_lib.rnn_workspace_size(dims, _lib.WS_BWD), dtype=torch.uint8, device="cuda"),
                    dWx=torch.empty_like(inp["Wx"]), dR=torch.empty_like(inp["R"]),
                    db=torch.empty_like(inp["b"]), ds0=torch.empty_like(inp["states0"]))

    def step(o):
        _lib.rnn_fwd(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], o["states"], o["last"], o["tape"], o["ws"])
        _lib.rnn_bwd(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], o["states"], o["tape"], inp["dstates"],
                     None, o["dWx"], o["dR"], o["db"], o["ds0"], o["ws"])

    names = ("states", "last", "dWx", "dR", "db", "ds0")
    eager = buffers()
    step(eager)
    torch.cuda.synchronize()
    _lib.rnn_check_status(eager["ws"])
    for fresh in (False, True):
        o = buffers() if fresh else eager
        ref = {k: eager[k].clone() for k in names}
        for k in names:
            o[k].fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(o)
        g.replay()
        torch.cuda.synchronize()
        _lib.rnn_check_status(o["ws"])
        for k in names:
            assert torch.equal(o[k], ref[k]), f"{k} differs after replay (fresh workspace: {fresh})"


def test_grid_reuses_its_workspace(monkeypatch):
    """Two grid forward + backward runs of different lengths on one workspace:
    the second must not see the first's step counters or exchange rows."""
    _restrict(monkeypatch, dict(C=16))
    B, N, D = 5, 1, 256
    dims_long = _lib.make_dims(B, 12, N, D, "lstm", torch.bfloat16, "grid")
    ws = torch.empty(_lib.rnn_workspace_size(dims_long, _lib.WS_BWD), dtype=torch.uint8, device="cuda")
    for T, seed in ((12, 61), (5, 62)):
        inp = _inputs("lstm", (B, T, N, D), torch.bfloat16, seed=seed)
        dims = _lib.make_dims(B, T, N, D, "lstm", torch.bfloat16, "grid")
        st = torch.full((2, B, T, N, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        last = torch.full((2, B, 1, N, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        tape = torch.empty(_lib.rnn_tape_size(dims), dtype=torch.uint8, device="cuda")
        _lib.rnn_fwd(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], st, last, tape, ws)
        _lib.rnn_check_status(ws)
        ref_st, _ = oracle_fwd("lstm", inp)
        check_states("lstm", torch.bfloat16, st, ref_st)
        dWx, dR, db, ds0 = (torch.full_like(inp[k], float("nan")) for k in ("Wx", "R", "b", "states0"))
        _lib.rnn_bwd(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], st, tape, inp["dstates"], None,
                     dWx, dR, db, ds0, ws)
        _lib.rnn_check_status(ws)
        check_grads("lstm", inp, (dWx, dR, db, ds0))


def test_grid_and_cluster_forward_agree(monkeypatch):
    _restrict(monkeypatch, dict(C=16))
    inp = _inputs("lstm", (8, 40, 2, 256), torch.bfloat16, seed=77)
    st_g, _, _ = run_fwd("lstm", inp, "grid", want_tape=False)
    st_f, _, _ = run_fwd("lstm", inp, "fused", want_tape=False)
    assert_states_close(st_g, st_f)


# ---------------------------------------------------------- alternating path
ALT_CASES = [
    ("lstm", 5, 13, 2, 64),
    ("gru", 9, 11, 1, 48),
    ("elman", 16, 9, 2, 128),
    ("slstm", 20, 7, 1, 64),     # two m-tiles per batch tile
    ("lstm", 3, 6, 1, 1024),
    ("gru", 33, 4, 1, 256),      # two batch tiles, ragged
    ("slstm_logsig", 7, 9, 2, 64),
]


@pytest.mark.parametrize("case", ALT_CASES, ids=lambda c: "%s-B%dT%dN%dD%d" % c)
def test_alternating_parity(case):
    fn, B, T, N, D = case
    inp = _inputs(fn, (B, T, N, D), torch.bfloat16, seed=1300 + B + T + D)
    dims = _lib.make_dims(B, T, N, D, fn, torch.bfloat16, "alternating")
    for bwd in (False, True):
        rc, desc = _lib.rnn_plan_describe(dims, bwd)
        assert rc == 0 and "path=alternating" in desc, desc
    st, last, tape = run_fwd(fn, inp, "alternating")
    ref_st, ref_last = oracle_fwd(fn, inp)
    check_states(fn, torch.bfloat16, st, ref_st)
    check_states(fn, torch.bfloat16, last, ref_last, "last")
    dl = torch.randn(last.shape, generator=torch.Generator().manual_seed(6)).to(torch.bfloat16).cuda()
    dWx, dR, db, ds0 = run_bwd(fn, inp, st, tape, "alternating", dlast=dl)
    check_grads(fn, inp, (dWx, dR, db, ds0), dlast=dl)
    # the tape is shared by every path: the plain backward on it agrees
    sdWx, _, _, _ = run_bwd(fn, inp, st, tape, "simt", dlast=dl)
    d1 = (dWx.float() - sdWx.float()).abs().max().item() / max(sdWx.float().abs().max().item(), 1e-30)
    assert d1 <= 2e-2, d1


def test_alternating_replays_its_graph():
    """Calls with the same buffers replay the captured graph: identical results
    for identical inputs, and new values written into the input buffers are
    picked up (the graph holds pointers, not data)."""
    fn, B, T, N, D = "lstm", 4, 10, 1, 128
    inp = _inputs(fn, (B, T, N, D), torch.bfloat16, seed=1401)
    S = _lib.rnn_num_states(fn)
    dims = _lib.make_dims(B, T, N, D, fn, torch.bfloat16, "alternating")
    states = torch.empty((S, B, T, N, D), dtype=torch.bfloat16, device="cuda")
    last = torch.empty((S, B, 1, N, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(_lib.rnn_workspace_size(dims, _lib.WS_FWD), dtype=torch.uint8, device="cuda")
    before = _lib.rnn_kernel_launches()
    outs = []
    for k in range(3):
        if k == 2:
            inp["Wx"].mul_(0.5)
        _lib.rnn_fwd(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], states, last, None, ws)
        _lib.rnn_check_status(ws)
        outs.append(states.clone())
    assert _lib.rnn_kernel_launches() - before == 3 * (T + 1)
    assert torch.equal(outs[0], outs[1])
    ref_st, _ = oracle_fwd(fn, inp)
    check_states(fn, torch.bfloat16, outs[2], ref_st)


def test_auto_takes_alternating_when_r_does_not_fit():
    fn, B, T, N, D = "lstm", 17, 5, 1, 2048
    dims = _lib.make_dims(B, T, N, D, fn, torch.bfloat16, "auto")
    for bwd in (False, True):
        rc, desc = _lib.rnn_plan_describe(dims, bwd)
        assert rc == 0 and "path=alternating" in desc, desc
    inp = _inputs(fn, (B, T, N, D), torch.bfloat16, seed=1402)
    st, last, tape = run_fwd(fn, inp, "auto")
    ref_st, _ = oracle_fwd(fn, inp)
    check_states(fn, torch.bfloat16, st, ref_st)
    dWx, dR, db, ds0 = run_bwd(fn, inp, st, tape, "auto")
    check_grads(fn, inp, (dWx, dR, db, ds0))


# ------------------------------------------------- weight gradients (tcgen05)
@pytest.mark.parametrize("case", [("lstm", 3, 200, 2, 192), ("gru", 70, 9, 1, 64), ("slstm", 2, 130, 1, 320),
                                  ("elman", 5, 100, 3, 136), ("lstm", 4, 70, 2, 200)],
                         ids=lambda c: "%s-B%dT%dN%dD%d" % c)
def test_weight_gradient_tiles(case):
    """dR and db through the tensor-memory GEMM: ragged tiles (D = 192, 320 with
    128 x 192 and 128 x 256 tiles), runs of steps that end inside a 64-step tile
    (T = 200, 130, 9, 100, 70), a batch wider than one 64-row initial-state tile
    (B = 70), split-K partial sums; D = 136 and 200 (not multiples of 64) take
    one TMA box per 64-unit slab instead of one gathered box per operand."""
    fn, B, T, N, D = case
    inp = _inputs(fn, (B, T, N, D), torch.bfloat16, seed=1500 + B + T + D)
    st, last, tape = run_fwd(fn, inp, "simt")
    dWx, dR, db, ds0 = run_bwd(fn, inp, st, tape, "simt")
    check_grads(fn, inp, (dWx, dR, db, ds0))
