"""Thin ctypes binding of the C ABI in ``include/ssd.h``.

The functions carry the C names (``ssd_workspace_size``, ``ssd_forward``,
``ssd_backward``, ``ssd_status_string``) and only marshal arguments: torch
tensors become device pointers, the torch stream becomes a ``cudaStream_t``,
and a non-OK status becomes an :class:`SSDError`.  Every step of the scan runs
in the library's kernels; there is no fallback of any kind.  If the library
cannot be loaded the call raises.

Convenience wrappers :func:`forward` and :func:`backward` allocate outputs
and the workspace with torch (device memory only) and call the ABI.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

VARIANTS = {"mamba2": 0, "mamba1": 1, "mimo": 2}
DTYPES = {"f32": 0, "bf16": 1}
_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}

SSD_OK = 0


class SSDError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {ssd_status_string(status)} (status {status})")


class ssd_problem(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("io_dtype", ctypes.c_int32), ("batch", ctypes.c_int64),
                ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64), ("headdim", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64), ("chunk", ctypes.c_int64),
                ("mimo_rank", ctypes.c_int64)]


EXPORTS = ("ssd_workspace_size", "ssd_forward", "ssd_backward", "ssd_forward_static", "ssd_profile_start",
           "ssd_profile_stop", "ssd_status_string", "ssd_version", "ssd_states_size", "ssd_forward_stash",
           "ssd_backward_stashed", "ssd_forward_static_status", "ssd_read_status", "ssd_wait_selftest",
           "ssd_checkpoints_size", "ssd_forward_checkpointed", "ssd_backward_checkpointed",
           "ssd_kda_workspace_size", "ssd_kda_forward", "ssd_kda_backward")


class ssd_kda_problem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("value_heads", ctypes.c_int64), ("key_dim", ctypes.c_int64), ("value_dim", ctypes.c_int64)]


class ssd_kernel_time(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_char_p), ("ms", ctypes.c_float)]

_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load (building first if needed) the in-tree shared library."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _build.build()
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library missing: {p}")
        lib = ctypes.CDLL(p)
        vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        lib.ssd_workspace_size.argtypes = [ctypes.POINTER(ssd_problem), i32, ctypes.POINTER(sz)]
        lib.ssd_workspace_size.restype = i32
        lib.ssd_forward.argtypes = [ctypes.POINTER(ssd_problem)] + [vp] * 8 + [vp, sz, vp]
        lib.ssd_forward.restype = i32
        lib.ssd_backward.argtypes = [ctypes.POINTER(ssd_problem)] + [vp] * 14 + [vp, sz, vp]
        lib.ssd_backward.restype = i32
        lib.ssd_status_string.argtypes = [i32]
        lib.ssd_status_string.restype = ctypes.c_char_p
        lib.ssd_forward_static.argtypes = [ctypes.POINTER(ssd_problem)] + [vp] * 8 + [vp]
        lib.ssd_forward_static.restype = i32
        lib.ssd_profile_start.argtypes = [i32]
        lib.ssd_profile_start.restype = i32
        lib.ssd_profile_stop.argtypes = [ctypes.POINTER(ssd_kernel_time), i32, ctypes.POINTER(i32)]
        lib.ssd_profile_stop.restype = i32
        lib.ssd_version.argtypes = []
        lib.ssd_version.restype = i32
        lib.ssd_states_size.argtypes = [ctypes.POINTER(ssd_problem), ctypes.POINTER(sz)]
        lib.ssd_states_size.restype = i32
        lib.ssd_forward_stash.argtypes = [ctypes.POINTER(ssd_problem)] + [vp] * 9 + [sz, vp, sz, vp]
        lib.ssd_forward_stash.restype = i32
        lib.ssd_backward_stashed.argtypes = [ctypes.POINTER(ssd_problem)] + [vp] * 8 + [sz] + [vp] * 7 + [sz, vp]
        lib.ssd_backward_stashed.restype = i32
        lib.ssd_forward_static_status.argtypes = [ctypes.POINTER(ctypes.c_int32), vp]
        lib.ssd_forward_static_status.restype = i32
        lib.ssd_read_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), vp]
        lib.ssd_read_status.restype = i32
        lib.ssd_wait_selftest.argtypes = [vp, ctypes.c_uint32, vp]
        lib.ssd_wait_selftest.restype = i32
        i64 = ctypes.c_int64
        lib.ssd_checkpoints_size.argtypes = [ctypes.POINTER(ssd_problem), i64, ctypes.POINTER(sz)]
        lib.ssd_checkpoints_size.restype = i32
        lib.ssd_forward_checkpointed.argtypes = [ctypes.POINTER(ssd_problem)] + [vp] * 8 + [i64, vp, sz, vp, sz, vp]
        lib.ssd_forward_checkpointed.restype = i32
        lib.ssd_backward_checkpointed.argtypes = ([ctypes.POINTER(ssd_problem)] + [vp] * 7 + [i64, vp, sz] + [vp] * 6 +
                                                 [vp, sz, vp])
        lib.ssd_backward_checkpointed.restype = i32
        kp = ctypes.POINTER(ssd_kda_problem)
        lib.ssd_kda_workspace_size.argtypes = [kp, i32, ctypes.POINTER(sz)]
        lib.ssd_kda_workspace_size.restype = i32
        lib.ssd_kda_forward.argtypes = [kp] + [vp] * 6 + [ctypes.c_float, vp, vp, vp, sz, vp]
        lib.ssd_kda_forward.restype = i32
        lib.ssd_kda_backward.argtypes = [kp] + [vp] * 8 + [ctypes.c_float] + [vp] * 6 + [vp, sz, vp]
        lib.ssd_kda_backward.restype = i32
        _lib = lib
        return lib


def problem(cfg: dict) -> ssd_problem:
    """An ``ssd_problem`` from a config dict (see ``configs.py``)."""
    return ssd_problem(VARIANTS[cfg["variant"]], DTYPES[cfg["dtype"]], cfg["batch"], cfg["seqlen"], cfg["nheads"],
                       cfg["headdim"], cfg["dstate"], cfg["ngroups"], cfg["chunk"], cfg["mimo_rank"])


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def ssd_status_string(status: int) -> str:
    return load().ssd_status_string(int(status)).decode()


def ssd_workspace_size(prob: ssd_problem, backward: bool) -> int:
    out = ctypes.c_size_t(0)
    st = load().ssd_workspace_size(ctypes.byref(prob), int(bool(backward)), ctypes.byref(out))
    if st != SSD_OK:
        raise SSDError(st, "ssd_workspace_size")
    return out.value


def ssd_forward(prob, x, dt_raw, A, B, C, s0, y, s_final, ws, ws_bytes, stream=None) -> None:
    st = load().ssd_forward(ctypes.byref(prob), _ptr(x), _ptr(dt_raw), _ptr(A), _ptr(B), _ptr(C), _ptr(s0),
                            _ptr(y), _ptr(s_final), _ptr(ws), int(ws_bytes), _stream(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_forward")


def ssd_forward_static(prob, x, dt_raw, A, B, C, s0, y, s_final, stream=None) -> None:
    """Forward without a workspace: the library's fixed 32 MiB device array is
    the scratch (see include/ssd.h).  Raises SSDError on a non-OK status."""
    st = load().ssd_forward_static(ctypes.byref(prob), _ptr(x), _ptr(dt_raw), _ptr(A), _ptr(B), _ptr(C), _ptr(s0),
                                   _ptr(y), _ptr(s_final), _stream(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_forward_static")


def ssd_forward_static_status(stream=None, read: bool = True) -> tuple:
    """(status, code) of the fixed array's device status word, read after the work enqueued on `stream`;
    with read=False only the start-up step (module load and address lookup) runs and code is None."""
    if not read:
        return load().ssd_forward_static_status(None, _stream(stream)), None
    code = ctypes.c_int32(-1)
    st = load().ssd_forward_static_status(ctypes.byref(code), _stream(stream))
    return st, code.value


def ssd_read_status(ws, stream=None) -> tuple:
    """(status, code) of the device status word in the first 4 bytes of the workspace `ws`."""
    code = ctypes.c_int32(-1)
    st = load().ssd_read_status(_ptr(ws), ctypes.byref(code), _stream(stream))
    return st, code.value


def ssd_wait_selftest(ws, limit_us: int, stream=None) -> int:
    """Launch the kernel whose bounded wait runs out after limit_us; returns the call's status."""
    return load().ssd_wait_selftest(_ptr(ws), int(limit_us), _stream(stream))


def ssd_backward(prob, dy, ds_final, x, dt_raw, A, B, C, s0, dx, ddt_raw, dA, dB, dC, ds0, ws, ws_bytes,
                 stream=None) -> None:
    st = load().ssd_backward(ctypes.byref(prob), _ptr(dy), _ptr(ds_final), _ptr(x), _ptr(dt_raw), _ptr(A), _ptr(B),
                             _ptr(C), _ptr(s0), _ptr(dx), _ptr(ddt_raw), _ptr(dA), _ptr(dB), _ptr(dC), _ptr(ds0),
                             _ptr(ws), int(ws_bytes), _stream(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_backward")


def ssd_states_size(prob: ssd_problem) -> int:
    out = ctypes.c_size_t(0)
    st = load().ssd_states_size(ctypes.byref(prob), ctypes.byref(out))
    if st != SSD_OK:
        raise SSDError(st, "ssd_states_size")
    return out.value


def ssd_forward_stash(prob, x, dt_raw, A, B, C, s0, y, s_final, states, states_bytes, ws, ws_bytes,
                      stream=None) -> None:
    st = load().ssd_forward_stash(ctypes.byref(prob), _ptr(x), _ptr(dt_raw), _ptr(A), _ptr(B), _ptr(C), _ptr(s0),
                                  _ptr(y), _ptr(s_final), _ptr(states), int(states_bytes), _ptr(ws), int(ws_bytes),
                                  _stream(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_forward_stash")


def ssd_checkpoints_size(prob: ssd_problem, every: int) -> int:
    out = ctypes.c_size_t(0)
    st = load().ssd_checkpoints_size(ctypes.byref(prob), int(every), ctypes.byref(out))
    if st != SSD_OK:
        raise SSDError(st, "ssd_checkpoints_size")
    return out.value


def ssd_forward_checkpointed(prob, x, dt_raw, A, B, C, s0, y, s_final, every, ckpt, ckpt_bytes, ws, ws_bytes,
                             stream=None) -> None:
    st = load().ssd_forward_checkpointed(ctypes.byref(prob), _ptr(x), _ptr(dt_raw), _ptr(A), _ptr(B), _ptr(C),
                                         _ptr(s0), _ptr(y), _ptr(s_final), int(every), _ptr(ckpt), int(ckpt_bytes),
                                         _ptr(ws), int(ws_bytes), _stream(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_forward_checkpointed")


def ssd_backward_checkpointed(prob, dy, ds_final, x, dt_raw, A, B, C, every, ckpt, ckpt_bytes, dx, ddt_raw, dA, dB,
                              dC, ds0, ws, ws_bytes, stream=None) -> None:
    st = load().ssd_backward_checkpointed(ctypes.byref(prob), _ptr(dy), _ptr(ds_final), _ptr(x), _ptr(dt_raw), _ptr(A),
                                          _ptr(B), _ptr(C), int(every), _ptr(ckpt), int(ckpt_bytes), _ptr(dx),
                                          _ptr(ddt_raw), _ptr(dA), _ptr(dB), _ptr(dC), _ptr(ds0), _ptr(ws),
                                          int(ws_bytes), _stream(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_backward_checkpointed")


def ssd_backward_stashed(prob, dy, ds_final, x, dt_raw, A, B, C, states, states_bytes, dx, ddt_raw, dA, dB, dC,
                         ds0, ws, ws_bytes, stream=None) -> None:
    st = load().ssd_backward_stashed(ctypes.byref(prob), _ptr(dy), _ptr(ds_final), _ptr(x), _ptr(dt_raw), _ptr(A),
                                     _ptr(B), _ptr(C), _ptr(states), int(states_bytes), _ptr(dx), _ptr(ddt_raw),
                                     _ptr(dA), _ptr(dB), _ptr(dC), _ptr(ds0), _ptr(ws), int(ws_bytes),
                                     _stream(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_backward_stashed")


def ssd_profile_start(capacity: int) -> None:
    st = load().ssd_profile_start(int(capacity))
    if st != SSD_OK:
        raise SSDError(st, "ssd_profile_start")


def ssd_profile_stop(capacity: int = 1 << 16) -> list:
    """Returns [(kernel name, ms)] for every launch recorded since start."""
    buf = (ssd_kernel_time * capacity)()
    n = ctypes.c_int(0)
    st = load().ssd_profile_stop(buf, int(capacity), ctypes.byref(n))
    if st != SSD_OK:
        raise SSDError(st, "ssd_profile_stop")
    return [(buf[i].kernel.decode(), float(buf[i].ms)) for i in range(n.value)]


# ---------------------------------------------------------------- conveniences
def _workspace(prob, backward, device):
    n = ssd_workspace_size(prob, backward)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device), n


def forward(cfg: dict, x, dt_raw, A, B, C, s0=None, stream=None, workspace=None):
    """Allocate y and s_final, run ``ssd_forward``; returns (y, s_final)."""
    prob = problem(cfg)
    dev = x.device
    y = torch.empty_like(x)
    sf_shape = (cfg["batch"], cfg["nheads"], cfg["dstate"]) if cfg["variant"] == "mamba1" else \
        (cfg["batch"], cfg["nheads"], cfg["headdim"], cfg["dstate"])
    s_final = torch.empty(sf_shape, dtype=torch.float32, device=dev)
    ws, n = workspace if workspace is not None else _workspace(prob, False, dev)
    ssd_forward(prob, x, dt_raw, A, B, C, s0, y, s_final, ws, n, stream)
    return y, s_final


def backward(cfg: dict, dy, ds_final, x, dt_raw, A, B, C, s0=None, stream=None, workspace=None):
    """Allocate the gradients, run ``ssd_backward``; returns a dict with
    dx, ddt_raw, dA (None for MIMO), dB, dC, ds0."""
    prob = problem(cfg)
    dev = x.device
    out = {"dx": torch.empty_like(x), "ddt_raw": torch.empty_like(dt_raw),
           "dA": None if A is None else torch.empty_like(A), "dB": torch.empty_like(B), "dC": torch.empty_like(C),
           "ds0": torch.empty_like(ds_final)}
    ws, n = workspace if workspace is not None else _workspace(prob, True, dev)
    ssd_backward(prob, dy, ds_final, x, dt_raw, A, B, C, s0, out["dx"], out["ddt_raw"], out["dA"], out["dB"],
                 out["dC"], out["ds0"], ws, n, stream)
    return out


def forward_stash(cfg: dict, x, dt_raw, A, B, C, s0=None, stream=None, workspace=None):
    """``forward`` that also keeps the chunk states; returns (y, s_final, states)
    with states a uint8 device tensor for ``backward_stashed``."""
    prob = problem(cfg)
    dev = x.device
    y = torch.empty_like(x)
    s_final = torch.empty((cfg["batch"], cfg["nheads"], cfg["headdim"], cfg["dstate"]), dtype=torch.float32,
                          device=dev)
    nst = ssd_states_size(prob)
    states = torch.empty(nst, dtype=torch.uint8, device=dev)
    ws, n = workspace if workspace is not None else _workspace(prob, False, dev)
    ssd_forward_stash(prob, x, dt_raw, A, B, C, s0, y, s_final, states, nst, ws, n, stream)
    return y, s_final, states


def backward_stashed(cfg: dict, dy, ds_final, x, dt_raw, A, B, C, states, stream=None, workspace=None):
    """``backward`` from the chunk states ``forward_stash`` kept (no s0, no
    forward replay); returns the same dict."""
    prob = problem(cfg)
    dev = x.device
    out = {"dx": torch.empty_like(x), "ddt_raw": torch.empty_like(dt_raw), "dA": torch.empty_like(A),
           "dB": torch.empty_like(B), "dC": torch.empty_like(C), "ds0": torch.empty_like(ds_final)}
    ws, n = workspace if workspace is not None else _workspace(prob, True, dev)
    ssd_backward_stashed(prob, dy, ds_final, x, dt_raw, A, B, C, states, states.numel(), out["dx"], out["ddt_raw"],
                         out["dA"], out["dB"], out["dC"], out["ds0"], ws, n, stream)
    return out


def forward_checkpointed(cfg: dict, x, dt_raw, A, B, C, s0=None, every: int = 8, stream=None, workspace=None):
    """``forward`` that also keeps fp32 checkpoints every ``every`` chunks; returns (y, s_final, ckpt) with ckpt
    a float32 device tensor [b, H, ceil(nc / every), P, N] for ``backward_checkpointed``."""
    prob = problem(cfg)
    dev = x.device
    y = torch.empty_like(x)
    s_final = torch.empty((cfg["batch"], cfg["nheads"], cfg["headdim"], cfg["dstate"]), dtype=torch.float32,
                          device=dev)
    nbytes = ssd_checkpoints_size(prob, every)
    nc = -(-cfg["seqlen"] // cfg["chunk"])
    nk = -(-nc // every)
    ckpt = torch.empty((cfg["batch"], cfg["nheads"], nk, cfg["headdim"], cfg["dstate"]), dtype=torch.float32,
                       device=dev)
    assert ckpt.numel() * 4 == nbytes
    ws, n = workspace if workspace is not None else _workspace(prob, False, dev)
    ssd_forward_checkpointed(prob, x, dt_raw, A, B, C, s0, y, s_final, every, ckpt, nbytes, ws, n, stream)
    return y, s_final, ckpt


def backward_checkpointed(cfg: dict, dy, ds_final, x, dt_raw, A, B, C, ckpt, every: int = 8, stream=None,
                          workspace=None):
    """``backward`` that replays the chunk states from ``forward_checkpointed``'s checkpoints (no s0); returns the
    same dict."""
    prob = problem(cfg)
    dev = x.device
    out = {"dx": torch.empty_like(x), "ddt_raw": torch.empty_like(dt_raw), "dA": torch.empty_like(A),
           "dB": torch.empty_like(B), "dC": torch.empty_like(C), "ds0": torch.empty_like(ds_final)}
    ws, n = workspace if workspace is not None else _workspace(prob, True, dev)
    ssd_backward_checkpointed(prob, dy, ds_final, x, dt_raw, A, B, C, every, ckpt, ckpt.numel() * 4, out["dx"],
                              out["ddt_raw"], out["dA"], out["dB"], out["dC"], out["ds0"], ws, n, stream)
    return out


# ------------------------------------------------------------- KDA (gated delta rule)
def kda_problem(cfg: dict) -> ssd_kda_problem:
    return ssd_kda_problem(cfg["batch"], cfg["seqlen"], cfg["nheads"], cfg["value_heads"], cfg["key_dim"],
                           cfg["value_dim"])


def ssd_kda_workspace_size(prob: ssd_kda_problem, backward: bool) -> int:
    out = ctypes.c_size_t(0)
    st = load().ssd_kda_workspace_size(ctypes.byref(prob), int(bool(backward)), ctypes.byref(out))
    if st != SSD_OK:
        raise SSDError(st, "ssd_kda_workspace_size")
    return out.value


def ssd_kda_forward(prob, q, k, v, g, beta, s0, scale, o, s_final, ws, ws_bytes, stream=None) -> None:
    st = load().ssd_kda_forward(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(s0),
                                float(scale), _ptr(o), _ptr(s_final), _ptr(ws), int(ws_bytes), _stream(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_kda_forward")


def ssd_kda_backward(prob, dout, ds_final, q, k, v, g, beta, s0, scale, dq, dk, dv, dg, dbeta, ds0, ws, ws_bytes,
                     stream=None) -> None:
    st = load().ssd_kda_backward(ctypes.byref(prob), _ptr(dout), _ptr(ds_final), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                 _ptr(beta), _ptr(s0), float(scale), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
                                 _ptr(dbeta), _ptr(ds0), _ptr(ws), int(ws_bytes), _stream(stream))
    if st != SSD_OK:
        raise SSDError(st, "ssd_kda_backward")


def _kda_workspace(prob, backward, device):
    n = ssd_kda_workspace_size(prob, backward)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device), n


def kda_forward(cfg: dict, q, k, v, g, beta, s0=None, scale=None, stream=None, workspace=None):
    """Allocate o, s_final and run ``ssd_kda_forward``; scale defaults to key_dim^-1/2."""
    prob = kda_problem(cfg)
    scale = cfg["key_dim"] ** -0.5 if scale is None else scale
    o = torch.empty_like(v)
    s_final = torch.empty((cfg["batch"], cfg["value_heads"], cfg["key_dim"], cfg["value_dim"]), dtype=torch.float32,
                          device=v.device)
    ws, n = workspace if workspace is not None else _kda_workspace(prob, False, v.device)
    ssd_kda_forward(prob, q, k, v, g, beta, s0, scale, o, s_final, ws, n, stream)
    return o, s_final


def kda_backward(cfg: dict, dout, ds_final, q, k, v, g, beta, s0=None, scale=None, stream=None, workspace=None):
    """Allocate the gradients and run ``ssd_kda_backward``; returns dq, dk, dv, dg, dbeta, ds0."""
    prob = kda_problem(cfg)
    scale = cfg["key_dim"] ** -0.5 if scale is None else scale
    out = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v), "dg": torch.empty_like(g),
           "dbeta": torch.empty_like(beta), "ds0": torch.empty_like(ds_final)}
    ws, n = workspace if workspace is not None else _kda_workspace(prob, True, v.device)
    ssd_kda_backward(prob, dout, ds_final, q, k, v, g, beta, s0, scale, out["dq"], out["dk"], out["dv"], out["dg"],
                     out["dbeta"], out["ds0"], ws, n, stream)
    return out
