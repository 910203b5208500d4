"""Thin ctypes binding of librnn_gb300.so: the C ABI of include/rnn.h, name for
name. Arguments are marshalled from torch tensors (device pointers, the current
CUDA stream); every computation happens in the library's CUDA kernels. There is
no fallback: if the library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import build as _build

RNN_OK, RNN_EINVAL, RNN_EUNSUPPORTED, RNN_ENOSPC, RNN_ETIMEOUT, RNN_ECUDA = range(6)
FUNCTIONS = {"lstm": 0, "gru": 1, "elman": 2, "slstm": 3, "slstm_logsig": 4}
DTYPES = {torch.float32: 0, torch.bfloat16: 1}
PATHS = {"auto": 0, "fused": 1, "alternating": 2, "simt": 3, "grid": 4}
WS_FWD, WS_BWD, WS_BWD_RECOMPUTE = 0, 1, 2

EXPORTS = ["rnn_num_gates", "rnn_num_states", "rnn_tape_size", "rnn_workspace_size", "rnn_fwd",
           "rnn_bwd", "rnn_check_status", "rnn_plan_describe", "rnn_strerror", "rnn_kernel_launches",
           "rnn_profile_events", "rnn_bwd_noalloc", "rnn_bwd_noalloc_status", "rnn_trace",
           "rnn_debug_inject_wait", "rnn_plan_set_limits", "rnn_die_layout", "rnn_die_plan_for"]


class RnnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {rnn_strerror(status)} (status {status})")


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("N", ctypes.c_int), ("D", ctypes.c_int),
                ("function", ctypes.c_int), ("dtype", ctypes.c_int), ("path", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load (building first if needed) the CUDA library; raises if impossible."""
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(path or _build.build())
            vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
            dp = ctypes.POINTER(Dims)
            lib.rnn_num_gates.argtypes = [i]
            lib.rnn_num_states.argtypes = [i]
            lib.rnn_tape_size.argtypes = [dp]
            lib.rnn_tape_size.restype = sz
            lib.rnn_workspace_size.argtypes = [dp, i]
            lib.rnn_workspace_size.restype = sz
            lib.rnn_fwd.argtypes = [dp] + [vp] * 8 + [sz, vp]
            lib.rnn_bwd.argtypes = [dp] + [vp] * 13 + [sz, vp]
            lib.rnn_check_status.argtypes = [vp, vp]
            lib.rnn_plan_describe.argtypes = [dp, i, ctypes.c_char_p, sz]
            lib.rnn_plan_set_limits.argtypes = [i, i, i]
            lib.rnn_die_layout.argtypes = [ctypes.POINTER(i), ctypes.POINTER(i)]
            ull_p = ctypes.POINTER(ctypes.c_ulonglong)
            lib.rnn_die_plan_for.argtypes = [i, i, ull_p, i, ull_p, i] + [ctypes.POINTER(i)] * 4
            lib.rnn_strerror.argtypes = [i]
            lib.rnn_strerror.restype = ctypes.c_char_p
            lib.rnn_kernel_launches.argtypes = []
            lib.rnn_kernel_launches.restype = ctypes.c_ulonglong
            lib.rnn_profile_events.argtypes = [i, vp, vp]
            lib.rnn_bwd_noalloc.argtypes = [dp] + [vp] * 13
            lib.rnn_bwd_noalloc_status.argtypes = [vp]
            lib.rnn_trace.argtypes = [vp, i, i]
            lib.rnn_debug_inject_wait.argtypes = [i, ctypes.c_ulonglong]
            lib.rnn_exchange_floor.argtypes = [i, i, i, vp, vp]
            lib.rnn_exchange_floor_grid.argtypes = [i, i, i, i, i, vp, sz, vp, vp]
            lib.rnn_input_proj_workspace_size.argtypes = [i, i, i]
            lib.rnn_input_proj_workspace_size.restype = sz
            lib.rnn_input_proj_fwd.argtypes = [i, i, i] + [vp] * 5 + [sz, vp]
            lib.rnn_input_proj_bwd.argtypes = [i, i, i] + [vp] * 7 + [sz, vp]
            _lib = lib
    return _lib


def make_dims(B, T, N, D, function="lstm", dtype=torch.bfloat16, path="auto") -> Dims:
    fn = FUNCTIONS[function] if isinstance(function, str) else int(function)
    dt = DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    pa = PATHS[path] if isinstance(path, str) else int(path)
    return Dims(int(B), int(T), int(N), int(D), fn, dt, pa)


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc: int, where: str) -> int:
    if rc != RNN_OK:
        raise RnnError(rc, where)
    return rc


# ---- the C ABI, name for name -------------------------------------------------
def rnn_num_gates(function) -> int:
    return load().rnn_num_gates(FUNCTIONS.get(function, function) if isinstance(function, str) else function)


def rnn_num_states(function) -> int:
    return load().rnn_num_states(FUNCTIONS.get(function, function) if isinstance(function, str) else function)


def rnn_tape_size(dims: Dims) -> int:
    return load().rnn_tape_size(ctypes.byref(dims))


def rnn_workspace_size(dims: Dims, kind: int = WS_FWD) -> int:
    return load().rnn_workspace_size(ctypes.byref(dims), kind)


def rnn_fwd(dims: Dims, Wx, R, b, states0, states, last, tape, workspace, stream=None) -> int:
    rc = load().rnn_fwd(ctypes.byref(dims), _p(Wx), _p(R), _p(b), _p(states0), _p(states), _p(last),
                        _p(tape), _p(workspace), workspace.numel() * workspace.element_size(),
                        _stream(stream))
    return _check(rc, "rnn_fwd")


def rnn_bwd(dims: Dims, Wx, R, b, states0, states, tape, dstates, dlast, dWx, dR, db, dstates0,
            workspace, stream=None) -> int:
    rc = load().rnn_bwd(ctypes.byref(dims), _p(Wx), _p(R), _p(b), _p(states0), _p(states), _p(tape),
                        _p(dstates), _p(dlast), _p(dWx), _p(dR), _p(db), _p(dstates0), _p(workspace),
                        workspace.numel() * workspace.element_size(), _stream(stream))
    return _check(rc, "rnn_bwd")


def rnn_check_status(workspace, stream=None) -> int:
    return _check(load().rnn_check_status(_p(workspace), _stream(stream)), "rnn_check_status")


def rnn_plan_describe(dims: Dims, for_backward: bool = False) -> tuple[int, str]:
    buf = ctypes.create_string_buffer(512)
    rc = load().rnn_plan_describe(ctypes.byref(dims), int(for_backward), buf, 512)
    return rc, buf.value.decode()


def rnn_plan_set_limits(sms: int = 0, smem_per_cta: int = 227 * 1024, max_cluster: int = 16) -> int:
    """Plan for a stated device (sms > 0) or the current one (sms <= 0)."""
    return _check(load().rnn_plan_set_limits(int(sms), int(smem_per_cta), int(max_cluster)),
                  "rnn_plan_set_limits")


def rnn_die_layout():
    """(SMs on die 0, SMs on die 1) as the grid kernels place their groups, or
    None when the device shows no two-die structure (see include/rnn.h)."""
    a, b = ctypes.c_int(0), ctypes.c_int(0)
    rc = load().rnn_die_layout(ctypes.byref(a), ctypes.byref(b))
    if rc == RNN_EUNSUPPORTED:
        return None
    _check(rc, "rnn_die_layout")
    return a.value, b.value


def rnn_die_plan_for(groups: int, C: int, sm_lat, blk_lat):
    """The die placement for stated L2 round trips (no GPU needed): sm_lat from
    the measuring CTA to every CTA (entry 0 itself), blk_lat on each 1 KB
    counter block. Returns (SMs on die 0, SMs on die 1, groups on die 0, each
    group's counter word), or None when the measurements are not trusted or no
    placement fits."""
    sm = (ctypes.c_ulonglong * len(sm_lat))(*[int(v) for v in sm_lat])
    bl = (ctypes.c_ulonglong * len(blk_lat))(*[int(v) for v in blk_lat])
    d0, d1, g0 = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    words = (ctypes.c_int * max(1, int(groups)))()
    rc = load().rnn_die_plan_for(int(groups), int(C), sm, len(sm_lat), bl, len(blk_lat), ctypes.byref(d0),
                                 ctypes.byref(d1), ctypes.byref(g0), words)
    if rc == RNN_EUNSUPPORTED:
        return None
    _check(rc, "rnn_die_plan_for")
    return d0.value, d1.value, g0.value, list(words[:groups])


def rnn_strerror(status: int) -> str:
    return load().rnn_strerror(status).decode()


def rnn_kernel_launches() -> int:
    return int(load().rnn_kernel_launches())


def rnn_profile_events(which: int, before=None, after=None) -> int:
    """which: 0 = forward scan kernel, 1 = backward scan kernel; torch.cuda.Event
    objects (recorded by the library around that kernel) or None to clear."""
    b = ctypes.c_void_p(before.cuda_event) if before is not None else None
    a = ctypes.c_void_p(after.cuda_event) if after is not None else None
    return _check(load().rnn_profile_events(which, b, a), "rnn_profile_events")


def rnn_bwd_noalloc(dims: Dims, Wx, R, b, states0, states, tape, dstates, dlast, dWx, dR, db,
                    dstates0, stream=None) -> int:
    """rnn_bwd without workspace: the library's fixed device scratch is used
    instead (for callers that cannot allocate device memory)."""
    rc = load().rnn_bwd_noalloc(ctypes.byref(dims), _p(Wx), _p(R), _p(b), _p(states0), _p(states),
                                _p(tape), _p(dstates), _p(dlast), _p(dWx), _p(dR), _p(db), _p(dstates0),
                                _stream(stream))
    return _check(rc, "rnn_bwd_noalloc")


def rnn_bwd_noalloc_status(stream=None) -> int:
    """Status of the last rnn_bwd_noalloc call on the current device (synchronises)."""
    return _check(load().rnn_bwd_noalloc_status(_stream(stream)), "rnn_bwd_noalloc_status")


def rnn_trace(buf=None, t0: int = 0, steps: int = 0) -> int:
    """Registers a device tensor of >= 16*steps int64 for the persistent kernels'
    phase trace (clock64 at up to sixteen points of steps [t0, t0+steps)), or None."""
    return _check(load().rnn_trace(_p(buf), int(t0), int(steps)), "rnn_trace")


def rnn_debug_inject_wait(step: int = -1, limit_ns: int = 0) -> int:
    """Test hook: the forward persistent kernels make CTA 0 wait at `step` on a
    barrier nothing signals, for limit_ns; step < 0 switches it off."""
    return _check(load().rnn_debug_inject_wait(int(step), int(limit_ns)), "rnn_debug_inject_wait")


def rnn_exchange_floor(C: int, slice_bytes: int, steps: int, out, stream=None) -> int:
    """Runs the exchange-only kernel (one cluster of C CTAs, bulk copies of
    slice_bytes to every peer per step) for `steps` steps; `out` is a device
    tensor of >= 2 int64: cycles per step of CTA 0, then the status."""
    return _check(load().rnn_exchange_floor(int(C), int(slice_bytes), int(steps), _p(out), _stream(stream)),
                  "rnn_exchange_floor")


def rnn_exchange_floor_grid(C: int, groups: int, rows: int, D: int, steps: int, scratch, out, stream=None) -> int:
    """Runs the grid kernels' L2 exchange alone (groups x C CTAs, `rows` batch
    rows of D units) for `steps` steps; `scratch` is a device uint8 tensor for
    the exchange buffers and counters, `out` >= 2 int64: cycles per step of
    CTA 0, then the status."""
    return _check(load().rnn_exchange_floor_grid(int(C), int(groups), int(rows), int(D), int(steps), _p(scratch),
                                                 scratch.numel() * scratch.element_size(), _p(out), _stream(stream)),
                  "rnn_exchange_floor_grid")


def rnn_input_proj_workspace_size(BT: int, I: int, C: int) -> int:
    return int(load().rnn_input_proj_workspace_size(int(BT), int(I), int(C)))


def rnn_input_proj_fwd(BT: int, I: int, C: int, x, W, bias, Wx, workspace, stream=None) -> int:
    """Wx[BT][C] = x[BT][I] W_x[C][I]^T (+ bias[C]) on the tensor cores (bf16)."""
    rc = load().rnn_input_proj_fwd(int(BT), int(I), int(C), _p(x), _p(W), _p(bias), _p(Wx), _p(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream))
    return _check(rc, "rnn_input_proj_fwd")


def rnn_input_proj_bwd(BT: int, I: int, C: int, x, W, dWx, dx, dW, dbias, workspace, stream=None) -> int:
    """dx = dWx W_x, dW = dWx^T x, dbias = column sums of dWx (each may be None)."""
    rc = load().rnn_input_proj_bwd(int(BT), int(I), int(C), _p(x), _p(W), _p(dWx), _p(dx), _p(dW), _p(dbias),
                                   _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    return _check(rc, "rnn_input_proj_bwd")
