"""The C-ABI library builds, loads and exports every declared entry point;
host-side validation and size queries work without a GPU."""
import ctypes
import os
import re

import pytest
import torch

from recurrent_networks_gb300 import _lib, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "rnn.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rnn_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(build.build())
    names = declared_symbols()
    assert "rnn_fwd" in names and "rnn_bwd" in names
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/rnn.h but not exported"
    assert set(_lib.EXPORTS) <= set(names)


def test_gate_and_state_counts():
    assert [_lib.rnn_num_gates(f) for f in range(4)] == [4, 3, 1, 4]
    assert [_lib.rnn_num_states(f) for f in range(4)] == [2, 1, 1, 4]
    assert _lib.rnn_num_gates(7) == -1


def test_sizes():
    d = _lib.make_dims(8, 1024, 3, 256, "lstm", torch.bfloat16)
    assert _lib.rnn_tape_size(d) == 1024 * 8 * 3 * 6 * 256 * 4
    ws_f = _lib.rnn_workspace_size(d, _lib.WS_FWD)
    ws_b = _lib.rnn_workspace_size(d, _lib.WS_BWD)
    ws_r = _lib.rnn_workspace_size(d, _lib.WS_BWD_RECOMPUTE)
    assert ws_f >= 256 and ws_f % 256 == 0
    assert ws_b >= ws_f + 8 * 1024 * 4 * 3 * 256 * 2
    assert ws_r >= ws_b + _lib.rnn_tape_size(d)
    assert _lib.rnn_workspace_size(_lib.make_dims(0, 4, 1, 8), 0) == 0
    assert _lib.rnn_tape_size(_lib.make_dims(2, 4, 1, 8, "slstm")) == 4 * 2 * 1 * 8 * 8 * 4


@pytest.mark.parametrize("bad", [dict(B=0), dict(N=0), dict(D=0), dict(T=-1)])
def test_invalid_dims_rejected_on_host(bad):
    kw = dict(B=2, T=3, N=1, D=8)
    kw.update(bad)
    d = _lib.make_dims(kw["B"], kw["T"], kw["N"], kw["D"], "lstm", torch.float32)
    lib = _lib.load()
    rc = lib.rnn_fwd(ctypes.byref(d), 16, 16, 16, None, 16, None, None, 256, 4096, None)
    assert rc == _lib.RNN_EINVAL


def test_null_and_misaligned_pointers_rejected():
    d = _lib.make_dims(2, 3, 1, 8, "lstm", torch.float32)
    lib = _lib.load()
    assert lib.rnn_fwd(ctypes.byref(d), None, 16, 16, None, 16, None, None, 256, 4096, None) == _lib.RNN_EINVAL
    assert lib.rnn_fwd(ctypes.byref(d), 18, 16, 16, None, 16, None, None, 256, 4096, None) == _lib.RNN_EINVAL
    assert lib.rnn_bwd(ctypes.byref(d), 16, 16, 16, None, 16, None, None, None, None, None, None, None,
                       None, 4096, None) == _lib.RNN_EINVAL


def test_workspace_too_small():
    d = _lib.make_dims(2, 3, 1, 8, "lstm", torch.float32)
    lib = _lib.load()
    rc = lib.rnn_fwd(ctypes.byref(d), 256, 256, 256, None, 256, None, None, 256, 16, None)
    assert rc == _lib.RNN_ENOSPC


def test_plan_describe():
    rc, text = _lib.rnn_plan_describe(_lib.make_dims(8, 1024, 3, 256, "lstm", torch.float32))
    assert rc == _lib.RNN_OK and "path=" in text
    assert _lib.rnn_strerror(_lib.RNN_ENOSPC) == "workspace too small"


def test_projection_sizes_and_host_validation():
    """The input projection's size query and argument checks run on the host:
    dims the TMA boxes cannot take size 0 and are rejected, as are null or
    misaligned pointers and a short workspace, before any device work."""
    lib = _lib.load()
    # I and C multiples of 8 and at least 64 (16-byte rows, 64-wide boxes)
    assert _lib.rnn_input_proj_workspace_size(8, 60, 128) == 0
    assert _lib.rnn_input_proj_workspace_size(8, 64, 124) == 0
    assert _lib.rnn_input_proj_workspace_size(8, 64, 56) == 0
    assert _lib.rnn_input_proj_workspace_size(0, 64, 128) == 0
    ok = _lib.rnn_input_proj_workspace_size(8192, 768, 3072)
    # status word + the dbias column-sum partials (at least one row chunk of C fp32)
    assert ok >= 256 + 3072 * 4
    big = _lib.rnn_input_proj_workspace_size(131072, 1024, 4096)
    assert big >= 256 + 4096 * 4
    ws = 4096
    assert lib.rnn_input_proj_fwd(8, 60, 128, 16, 16, None, 16, 256, ws, None) == _lib.RNN_EINVAL
    assert lib.rnn_input_proj_fwd(8, 64, 128, None, 16, None, 16, 256, ws, None) == _lib.RNN_EINVAL
    assert lib.rnn_input_proj_fwd(8, 64, 128, 24, 16, None, 16, 256, ws, None) == _lib.RNN_EINVAL
    assert lib.rnn_input_proj_fwd(8, 64, 128, 16, 16, 40, 16, 256, ws, None) == _lib.RNN_EINVAL
    assert lib.rnn_input_proj_fwd(8192, 768, 3072, 16, 16, None, 16, 256, 256, None) == _lib.RNN_ENOSPC
    assert lib.rnn_input_proj_bwd(8, 64, 128, 16, 16, 16, 24, None, None, 256, ws, None) == _lib.RNN_EINVAL
    assert lib.rnn_input_proj_bwd(8192, 768, 3072, 16, 16, 16, 16, 16, 16, 256, 256, None) == _lib.RNN_ENOSPC


def test_grid_exchange_floor_validates_on_host():
    lib = _lib.load()
    out = ctypes.c_void_p(4096)
    scratch = ctypes.c_void_p(1 << 20)
    # D not a multiple of C, too many rows, a misaligned scratch, a short scratch
    assert lib.rnn_exchange_floor_grid(3, 1, 8, 256, 10, scratch, 1 << 20, out, None) == _lib.RNN_EINVAL
    assert lib.rnn_exchange_floor_grid(16, 1, 33, 256, 10, scratch, 1 << 20, out, None) == _lib.RNN_EINVAL
    assert lib.rnn_exchange_floor_grid(16, 1, 8, 256, 10, ctypes.c_void_p((1 << 20) + 16), 1 << 20, out,
                                       None) == _lib.RNN_EINVAL
    assert lib.rnn_exchange_floor_grid(16, 1, 8, 256, 10, scratch, 1024, out, None) == _lib.RNN_ENOSPC
