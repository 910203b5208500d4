"""Failure detection without a GPU fault: every device-side wait of the
persistent kernels is bounded; when one runs out the kernel records a status
word that the host reads (RNN_ETIMEOUT) and the context stays usable.

The test makes a wait run out on purpose: CTA 0 waits on an mbarrier that
nothing signals (rnn_debug_inject_wait); the step exchange is left untouched,
so the results must still be correct."""
import pytest
import torch

from recurrent_networks_gb300 import _lib
from recurrent_networks_gb300.synth import make_inputs

from parity_util import run_fwd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("path,shape", [("fused", (5, 12, 2, 64)), ("grid", (5, 12, 1, 256))])
def test_injected_wait_times_out_and_is_reported(path, shape):
    B, T, N, D = shape
    inp = make_inputs("lstm", B, T, N, D, torch.bfloat16, seed=31, device="cuda")
    ref, _, _ = run_fwd("lstm", inp, path, want_tape=False)
    try:
        _lib.rnn_debug_inject_wait(4, 20_000_000)  # 20 ms
        with pytest.raises(_lib.RnnError) as err:
            run_fwd("lstm", inp, path, want_tape=False)
        assert err.value.status == _lib.RNN_ETIMEOUT
    finally:
        _lib.rnn_debug_inject_wait(-1)
    # the kernel ran to its end with the real exchange intact: same states
    dims = _lib.make_dims(B, T, N, D, "lstm", torch.bfloat16, path)
    S = 2
    states = torch.empty((S, B, T, N, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(_lib.rnn_workspace_size(dims, _lib.WS_FWD), dtype=torch.uint8, device="cuda")
    _lib.rnn_debug_inject_wait(2, 5_000_000)
    try:
        _lib.rnn_fwd(dims, inp["Wx"], inp["R"], inp["b"], inp["states0"], states, None, None, ws)
        torch.cuda.synchronize()
        assert torch.equal(states, ref)
        with pytest.raises(_lib.RnnError):
            _lib.rnn_check_status(ws)
    finally:
        _lib.rnn_debug_inject_wait(-1)
    # and the context is still usable: a clean run reports no error
    st, _, _ = run_fwd("lstm", inp, path, want_tape=False)
    assert torch.equal(st, ref)


def test_injection_arguments_validated():
    assert _lib.load().rnn_debug_inject_wait(3, 0) == _lib.RNN_EINVAL
    assert _lib.load().rnn_debug_inject_wait(-1, 0) == _lib.RNN_OK


def test_exchange_floor_runs_and_reports():
    """The exchange-only kernel completes with status 0 and a cycles-per-step
    figure that grows with the number of peers (more bulk copies per step)."""
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    cyc = {}
    for C in (2, 16):
        _lib.rnn_exchange_floor(C, 384, 500, out)
        torch.cuda.synchronize()
        v = out.cpu().tolist()
        assert v[1] == 0, v
        assert 100 < v[0] < 1_000_000, v
        cyc[C] = v[0]
    assert cyc[16] > cyc[2], cyc
    with pytest.raises(_lib.RnnError):
        _lib.rnn_exchange_floor(17, 384, 500, out)


def test_grid_exchange_floor_runs_and_reports():
    """The grid kernels' L2 exchange alone completes with status 0; two groups
    of 64 CTAs pulling 16 rows of 1024 units take longer per step than one
    group of 16 CTAs pulling 8 rows of 256."""
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    scratch = torch.empty(2 * 2 * 16 * 1024 * 2 + 32768, dtype=torch.uint8, device="cuda")
    cyc = {}
    for C, groups, rows, D in ((16, 1, 8, 256), (64, 2, 16, 1024)):
        _lib.rnn_exchange_floor_grid(C, groups, rows, D, 500, scratch, out)
        torch.cuda.synchronize()
        v = out.cpu().tolist()
        assert v[1] == 0, v
        assert 100 < v[0] < 1_000_000, v
        cyc[D] = v[0]
    assert cyc[1024] > cyc[256], cyc
