"""The kernel planner (an integer constraint solver over tile and cluster sizes,
the role the FlashRNN announcement's overview gives its ConstrINT tuner),
checked on the CPU through the C ABI:

- brute force: every candidate point (cluster size C, n-tiles NT, k-tiles KT,
  all-gates flag; backward m-tiles MT; grid C, NT, KT) of a grid of (cell, B,
  D) is judged feasible or not by a restatement of the constraints below, and
  the library must admit exactly those points, with the same shared-memory
  footprint;
- requests no point satisfies return RNN_EUNSUPPORTED with a reason;
- a stated device (fewer SMs, smaller clusters, less shared memory) removes
  exactly the points its limits exclude;
- the latency model orders the measured cluster sizes as the measurements do,
  and its choice is the fastest point of a timed sweep of every feasible plan.
"""
import itertools
import os

import pytest
import torch

from recurrent_networks_gb300 import _lib

G_OF = {"lstm": 4, "gru": 3, "elman": 1, "slstm": 4, "slstm_logsig": 4}
S_OF = {"lstm": 2, "gru": 1, "elman": 1, "slstm": 4, "slstm_logsig": 4}
NS = 4              # Wx / tape ring depth
RED_STRIDE = 20     # floats per batch row of a partial-sum tile
PPT = 2             # (row, unit) pairs a thread carries
MAX_KS = 8
MAX_KTA = 8
CLUSTER_SIZES = [1, 2, 3, 4, 6, 8, 12, 16]
FWD_POINTS = [(1, kt, False) for kt in (4, 6, 8, 12, 16)] + [(nt, kt, True) for nt in (1, 2) for kt in (2, 3, 4)]
BWD_POINTS = [(nt, mt) for nt in (1, 2) for mt in (1, 2)]
GRID_C = [8, 16, 32, 64, 128]
GRID_FWD_KT = [8, 16, 32]
GRID_BWD_KT = [8, 16, 24, 32]


class Limits:
    def __init__(self, sms=152, smem=227 * 1024, max_cluster=16):
        self.sms, self.smem, self.max_cluster = sms, smem, max_cluster


def _take(off, nbytes):
    return (off + nbytes + 127) & ~127


def _fwd_smem(G, D, U, BC, KS):
    C, UP = D // U, U + 8
    off = _take(0, 8 * (3 + NS))                       # barriers
    off = _take(off, NS * BC * G * U * 2)              # Wx ring
    off = _take(off, 2 * C * BC * UP * 2)              # h_{t-1}, double-buffered
    off = _take(off, (U // 16) * KS * G * BC * RED_STRIDE * 4)  # K-split partial sums
    off = _take(off, 2 * BC * UP * 2)                  # staged h_t
    return off


def _ring(S, K, U, BC):
    tape = BC * K * U * 4
    dst_off = (tape + 127) & ~127
    return (dst_off + S * BC * U * 2 + 127) & ~127


def _bwd_smem(G, S, K, U, BC, C):
    off = _take(0, 8 * (2 + NS))
    off = _take(off, NS * _ring(S, K, U, BC))
    off = _take(off, 2 * C * U * BC * 4)               # received partial sums of dh
    off = _take(off, 2 * BC * (G * U + 8) * 2)         # own dr, bf16
    off = _take(off, S * BC * U * 4)                   # initial states
    off = _take(off, G * BC * U * 4)                   # running db sums of the pairs
    return off


def _grid_bwd_smem(G, S, K, D, U, BC, KS):
    off = _take(0, 8 * (NS + 1))
    off = _take(off, NS * _ring(S, K, U, BC))
    off = _take(off, BC * (G * D + 8) * 2)             # the group's dr
    off = _take(off, (U // 16) * KS * BC * RED_STRIDE * 4)
    off = _take(off, S * BC * U * 4)
    off = _take(off, S * BC * U * 4)
    off = _take(off, G * BC * U * 4)                   # running db sums of the pairs
    return off


def _fwd_warps(U, GQ, KS, nb):
    return max((U // 16) * GQ * KS, -(-(nb * U) // (PPT * 32)))


def fwd_point(fn, B, N, D, C, NT, KT, allg, lim):
    """Forward cluster kernel: (smem bytes) when every constraint holds, else None."""
    G, S = G_OF[fn], S_OF[fn]
    if C > lim.max_cluster or D % C:
        return None
    U = D // C
    if U % 16 or D % 16 or (D // 16) % KT:
        return None
    KS = D // 16 // KT
    if KS > MAX_KS:
        return None
    GW = G if allg else 1
    GQ, CH = G // GW, (2 if GW == 1 else 1)
    BC = 8 * NT
    warps = _fwd_warps(U, GQ, KS, min(B, BC))
    if not 1 <= warps <= 8 or 4 * GW * KT + 4 * GW * CH * NT + 80 > 255:
        return None
    smem = _fwd_smem(G, D, U, BC, KS)
    if smem > lim.smem or lim.sms // C < 1:
        return None
    return smem


def bwd_point(fn, B, N, D, C, NT, MT, lim):
    G, S = G_OF[fn], S_OF[fn]
    K = (4 if fn == "gru" else G) + S
    if C > lim.max_cluster or D % C:
        return None
    U = D // C
    if U % 16 or D % 16:
        return None
    KTA = G * U // 16
    if not 1 <= KTA <= MAX_KTA or (D // 16) % MT:
        return None
    warps = D // 16 // MT
    BC = 8 * NT
    if not 1 <= warps <= 8 or min(B, BC) * U > PPT * warps * 32 or 32 * MT + 4 * MT * NT + 64 > 255:
        return None
    smem = _bwd_smem(G, S, K, U, BC, C)
    if smem > lim.smem or lim.sms // C < 1:
        return None
    return smem


def grid_point(fn, B, N, D, C, NT, KT, bwd, lim):
    G, S = G_OF[fn], S_OF[fn]
    K = (4 if fn == "gru" else G) + S
    if D % C:
        return None
    U = D // C
    if U % 16 or D % 16:
        return None
    klen = G * D if bwd else D
    if (klen // 16) % KT:
        return None
    KS = klen // 16 // KT
    BC = 8 * NT
    warps = (U // 16) * KS if bwd else _fwd_warps(U, G, KS, min(B, BC))
    groups = N * -(-B // BC)
    regs = 4 * KT + 4 * NT + 64 if bwd else 4 * KT + 8 * NT + 80
    if not 1 <= warps <= 8 or groups * C > lim.sms or regs > 255:
        return None
    smem = _grid_bwd_smem(G, S, K, D, U, BC, KS) if bwd else _fwd_smem(G, D, U, BC, KS)
    return None if smem > lim.smem else smem


def _parse(desc):
    return dict(kv.split("=", 1) for kv in desc.split() if "=" in kv)


@pytest.fixture
def planner(monkeypatch):
    """Plans through the library with the RNN_PLAN_* restriction variables
    and a stated device (GB300 limits unless a test states others)."""
    for k in ("C", "NT", "KT", "MT", "ALLG"):
        monkeypatch.delenv(f"RNN_PLAN_{k}", raising=False)
    _lib.rnn_plan_set_limits(152, 227 * 1024, 16)

    def plan(fn, B, N, D, path, bwd, dtype=torch.bfloat16, **restrict):
        for k in ("C", "NT", "KT", "MT", "ALLG"):
            if k in restrict:
                os.environ[f"RNN_PLAN_{k}"] = str(int(restrict[k]))
            else:
                os.environ.pop(f"RNN_PLAN_{k}", None)
        rc, desc = _lib.rnn_plan_describe(_lib.make_dims(B, 64, N, D, fn, dtype, path), bwd)
        return rc, desc

    yield plan
    for k in ("C", "NT", "KT", "MT", "ALLG"):
        os.environ.pop(f"RNN_PLAN_{k}", None)
    _lib.rnn_plan_set_limits(0)


GRID_OF_PROBLEMS = list(itertools.product(["lstm", "gru", "elman", "slstm"], [1, 8, 16, 32],
                                          [32, 48, 64, 96, 128, 192, 256, 512, 1024]))


@pytest.mark.parametrize("fn", ["lstm", "gru", "elman", "slstm"])
def test_forward_cluster_points_match_brute_force(planner, fn):
    lim = Limits()
    checked = 0
    for _, B, D in (p for p in GRID_OF_PROBLEMS if p[0] == fn):
        for C in CLUSTER_SIZES:
            for NT, KT, allg in FWD_POINTS:
                want = fwd_point(fn, B, 1, D, C, NT, KT, allg, lim)
                rc, desc = planner(fn, B, 1, D, "fused", False, C=C, NT=NT, KT=KT, ALLG=allg)
                if want is None:
                    assert rc == _lib.RNN_EUNSUPPORTED, (fn, B, D, C, NT, KT, allg, desc)
                    assert desc.startswith("unsupported:")
                else:
                    assert rc == 0, (fn, B, D, C, NT, KT, allg, desc)
                    p = _parse(desc)
                    assert (int(p["C"]), int(p["NT"]), int(p["KT"]), int(p["allg"])) == (C, NT, KT, int(allg))
                    assert int(p["smem"]) == want and int(p["U"]) == D // C
                checked += 1
    assert checked > 1000


@pytest.mark.parametrize("fn", ["lstm", "gru", "elman", "slstm"])
def test_backward_cluster_points_match_brute_force(planner, fn):
    lim = Limits()
    for _, B, D in (p for p in GRID_OF_PROBLEMS if p[0] == fn):
        for C in CLUSTER_SIZES:
            for NT, MT in BWD_POINTS:
                want = bwd_point(fn, B, 1, D, C, NT, MT, lim)
                rc, desc = planner(fn, B, 1, D, "fused", True, C=C, NT=NT, MT=MT)
                if want is None:
                    assert rc == _lib.RNN_EUNSUPPORTED, (fn, B, D, C, NT, MT, desc)
                else:
                    assert rc == 0, (fn, B, D, C, NT, MT, desc)
                    p = _parse(desc)
                    assert (int(p["C"]), int(p["NT"]), int(p["MT"])) == (C, NT, MT)
                    assert int(p["smem"]) == want


@pytest.mark.parametrize("bwd", [False, True], ids=["fwd", "bwd"])
def test_grid_points_match_brute_force(planner, bwd):
    lim = Limits()
    for fn, B, D in GRID_OF_PROBLEMS:
        for C in GRID_C:
            for NT in (1, 2):
                for KT in (GRID_BWD_KT if bwd else GRID_FWD_KT):
                    want = grid_point(fn, B, 1, D, C, NT, KT, bwd, lim)
                    rc, desc = planner(fn, B, 1, D, "grid", bwd, C=C, NT=NT, KT=KT)
                    if want is None:
                        assert rc == _lib.RNN_EUNSUPPORTED, (fn, B, D, C, NT, KT, desc)
                    else:
                        assert rc == 0, (fn, B, D, C, NT, KT, desc)
                        assert int(_parse(desc)["smem"]) == want


def test_unrestricted_choice_is_the_cheapest_feasible_point(planner):
    """With no restriction the planner returns the feasible point of smallest
    modelled step latency (each point's model read back through a restricted
    plan)."""
    for fn, B, N, D in [("lstm", 8, 3, 256), ("slstm", 16, 4, 192), ("gru", 16, 4, 128), ("elman", 16, 4, 128)]:
        rc, desc = planner(fn, B, N, D, "fused", False)
        assert rc == 0
        best = float(_parse(desc)["model_ns"])
        models = []
        for C in CLUSTER_SIZES:
            for NT, KT, allg in FWD_POINTS:
                r, d = planner(fn, B, N, D, "fused", False, C=C, NT=NT, KT=KT, ALLG=allg)
                if r == 0:
                    models.append(float(_parse(d)["model_ns"]))
        assert int(_parse(desc)["candidates"]) == len(models)
        assert best == pytest.approx(min(models))


def test_model_orders_the_measured_cluster_sizes(planner):
    """LSTM bf16 B=8 N=3 D=256 was measured with clusters of 16 and of 8 (the
    same kernels): forward 2185 vs 2649 cycles per step, backward 2568 vs
    2930. The model must order them the same way, and the unrestricted plan
    must be the cluster of 16 (forward 1781, backward 2024 cycles since);
    sLSTM B=16 N=4 D=192 runs on clusters of 12."""
    for bwd in (False, True):
        m = {}
        for C in (8, 16):
            rc, desc = planner("lstm", 8, 3, 256, "fused", bwd, C=C)
            assert rc == 0
            m[C] = float(_parse(desc)["model_ns"])
        assert m[16] < m[8]
        rc, desc = planner("lstm", 8, 3, 256, "auto", bwd)
        assert "path=fused" in desc and _parse(desc)["C"] == "16"
        rc, desc = planner("slstm", 16, 4, 192, "auto", bwd)
        assert "path=fused" in desc and _parse(desc)["C"] == "12"


def test_infeasible_requests_are_unsupported_with_a_reason(planner):
    # R of D = 2048 fits no cluster: no cluster point exists
    rc, desc = planner("lstm", 8, 1, 2048, "fused", False)
    assert rc == _lib.RNN_EUNSUPPORTED and "no cluster plan" in desc
    # the cluster and grid kernels are bf16-only
    for path in ("fused", "grid", "alternating"):
        rc, desc = planner("lstm", 2, 1, 32, path, False, dtype=torch.float32)
        assert rc == _lib.RNN_EUNSUPPORTED and desc.startswith("unsupported:"), (path, desc)
    # a head size that is not a multiple of 16 units
    rc, desc = planner("lstm", 8, 1, 200, "fused", True)
    assert rc == _lib.RNN_EUNSUPPORTED
    # AUTO always finds a plan: the plain kernel takes what nothing else fits
    rc, desc = planner("lstm", 2, 1, 32, "auto", False, dtype=torch.float32)
    assert rc == 0 and "path=simt" in desc
    rc, desc = planner("lstm", 8, 1, 200, "auto", True)
    assert rc == 0 and "path=simt" in desc


def test_stated_device_limits_remove_points(planner):
    # clusters of at most 8: no point above, and the D = 256 LSTM takes C <= 8
    _lib.rnn_plan_set_limits(152, 227 * 1024, 8)
    rc, desc = planner("lstm", 8, 3, 256, "auto", False)
    assert rc == 0 and "path=fused" in desc and int(_parse(desc)["C"]) <= 8
    rc, desc = planner("lstm", 8, 3, 256, "fused", False, C=16)
    assert rc == _lib.RNN_EUNSUPPORTED
    # 32 SMs cannot hold the 64-CTA group the D = 1024 grid kernel needs;
    # AUTO then streams R per step (the alternating path)
    _lib.rnn_plan_set_limits(32, 227 * 1024, 16)
    rc, desc = planner("lstm", 32, 1, 1024, "grid", False)
    assert rc == _lib.RNN_EUNSUPPORTED
    rc, desc = planner("lstm", 32, 1, 1024, "auto", False)
    assert rc == 0 and "path=alternating" in desc
    # less shared memory per CTA: the brute force follows the stated limit
    lim = Limits(sms=152, smem=64 * 1024, max_cluster=16)
    _lib.rnn_plan_set_limits(lim.sms, lim.smem, lim.max_cluster)
    for C in CLUSTER_SIZES:
        for NT, KT, allg in FWD_POINTS:
            want = fwd_point("lstm", 16, 1, 256, C, NT, KT, allg, lim)
            rc, _ = planner("lstm", 16, 1, 256, "fused", False, C=C, NT=NT, KT=KT, ALLG=allg)
            assert (rc == 0) == (want is not None), (C, NT, KT, allg)


def test_bad_limits_are_rejected():
    lib = _lib.load()
    assert lib.rnn_plan_set_limits(152, 100, 16) == _lib.RNN_EINVAL
    assert lib.rnn_plan_set_limits(152, 227 * 1024, 17) == _lib.RNN_EINVAL
    assert lib.rnn_plan_set_limits(0, 0, 0) == _lib.RNN_OK


# The fastest plan of a timed sweep of every feasible cluster plan on one GB300
# (profiles/planner_sweep_cluster_scan.md): the planner's unrestricted choice
# must be that point.
MEASURED_BEST = [
    # (cell, B, N, D, backward, C, NT, KT or MT)
    ("lstm", 8, 3, 256, False, 16, 1, 8),
    ("lstm", 8, 3, 256, True, 16, 1, 2),
    ("slstm", 16, 4, 192, False, 12, 1, 6),
    ("slstm", 16, 4, 192, True, 12, 1, 2),
]


@pytest.mark.parametrize("case", MEASURED_BEST, ids=lambda c: "%s-D%d-%s" % (c[0], c[3], "bwd" if c[4] else "fwd"))
def test_choice_is_the_measured_fastest_plan(planner, case):
    fn, B, N, D, bwd, C, NT, X = case
    rc, desc = planner(fn, B, N, D, "fused", bwd)
    assert rc == 0
    p = _parse(desc)
    assert (int(p["C"]), int(p["NT"]), int(p["MT"] if bwd else p["KT"])) == (C, NT, X), desc
