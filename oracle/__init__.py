"""Float64 CPU oracle for the selective state-space scan and its VJP.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library and its Python binding never import it, and this
package never imports them: the two implementations share no code.

Two independent float64 implementations live here:

* ``ssd_oracle.c`` -- the serial recurrence and the store-all reverse-time
  VJP (the plain definition, one (batch, head) unit at a time), compiled
  with gcc on first use and called through ctypes.  Functions:
  :func:`mamba2_forward`, :func:`mamba2_backward`, :func:`mamba1_forward`,
  :func:`mamba1_backward`, :func:`mimo_forward`, :func:`mimo_backward`.
* :mod:`oracle.chunkwise` -- the chunkwise (K1..K5) form and its backward,
  written in numpy from the Mamba-3 combined_backward.rs page's algebra.
  It exists to pin the serial oracle (the two must agree to rounding).
* :mod:`oracle.kda` -- the KDA delta-rule recurrence (the notes page
  "sec-10.tex": forward F1-F6 and the reverse loop of steps 1-6, store-all),
  in numpy, a second workload with its own entry points in the library.

Every array argument is converted to contiguous float64; results are new
float64 arrays.  Shapes follow the library's layouts:

* Mamba-2: x [b,T,H,P], dt_raw [b,T,H], A [H], B/C [b,T,G,N], s0 [b,H,P,N]
* Mamba-1: x/dt_raw [b,T,D], A [D,N], B/C [b,T,N], s0 [b,D,N]
* MIMO:    v [b,T,R,H,P], da [b,T,H], B/C [b,T,R,H,N], s0 [b,H,P,N]

``mutation`` (backward only) plants one of the five defects listed on the
"S1-31: SSM_SCAN_BACK" page's verification table; 0 is the correct VJP.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_lib = None

MUTATIONS = {
    0: "none",
    1: "drop the dA path from d(dt)",
    2: "seed the state gradient with zeros",
    3: "drop y's own contribution to dS",
    4: "use s_{t-1} where s_t belongs in dC",
    5: "drop the softplus derivative",
}


def build() -> str:
    """Compile ssd_oracle.c into a shared library (once per source hash)."""
    with open(_SRC, "rb") as f:
        digest = hashlib.sha1(f.read()).hexdigest()[:12]
    os.makedirs(_BUILD, exist_ok=True)
    out = os.path.join(_BUILD, f"libssd_oracle_{digest}.so")
    if not os.path.exists(out):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
               "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dp, ci = ctypes.c_int64, ctypes.POINTER(ctypes.c_double), ctypes.c_int
            lib.oracle_m2_forward.argtypes = [i64] * 6 + [dp] * 8 + [ci]
            lib.oracle_m2_backward.argtypes = [i64] * 6 + [dp] * 14 + [ci, ci]
            lib.oracle_m1_forward.argtypes = [i64] * 4 + [dp] * 8 + [ci]
            lib.oracle_m1_backward.argtypes = [i64] * 4 + [dp] * 14 + [ci, ci]
            lib.oracle_mimo_forward.argtypes = [i64] * 6 + [dp] * 7 + [ci]
            lib.oracle_mimo_backward.argtypes = [i64] * 6 + [dp] * 12 + [ci, ci]
            for fn in ("oracle_m2_forward", "oracle_m2_backward", "oracle_m1_forward",
                       "oracle_m1_backward", "oracle_mimo_forward", "oracle_mimo_backward"):
                getattr(lib, fn).restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _check(rc, name):
    if rc != 0:
        raise RuntimeError(f"{name} failed (rc={rc})")


# ------------------------------------------------------------------ Mamba-2
def mamba2_forward(x, dt_raw, A, B, C, s0=None, nthreads=None):
    x, dt_raw, A, B, C, s0 = map(_f64, (x, dt_raw, A, B, C, s0))
    b, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    assert dt_raw.shape == (b, T, H) and A.shape == (H,)
    assert B.shape == (b, T, G, N) and C.shape == (b, T, G, N)
    assert s0 is None or s0.shape == (b, H, P, N)
    y = np.empty_like(x)
    s_final = np.empty((b, H, P, N))
    rc = _load().oracle_m2_forward(b, T, H, P, N, G, _ptr(x), _ptr(dt_raw), _ptr(A), _ptr(B), _ptr(C),
                                   _ptr(s0), _ptr(y), _ptr(s_final), nthreads or default_threads())
    _check(rc, "oracle_m2_forward")
    return {"y": y, "s_final": s_final}


def mamba2_backward(dy, ds_final, x, dt_raw, A, B, C, s0=None, nthreads=None, mutation=0):
    dy, ds_final, x, dt_raw, A, B, C, s0 = map(_f64, (dy, ds_final, x, dt_raw, A, B, C, s0))
    b, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    assert dy.shape == x.shape and ds_final.shape == (b, H, P, N)
    out = {"dx": np.empty_like(x), "ddt_raw": np.empty_like(dt_raw), "dA": np.empty_like(A),
           "dB": np.empty_like(B), "dC": np.empty_like(C), "ds0": np.empty((b, H, P, N))}
    rc = _load().oracle_m2_backward(b, T, H, P, N, G, _ptr(x), _ptr(dt_raw), _ptr(A), _ptr(B), _ptr(C),
                                    _ptr(s0), _ptr(dy), _ptr(ds_final), _ptr(out["dx"]), _ptr(out["ddt_raw"]),
                                    _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["ds0"]),
                                    nthreads or default_threads(), int(mutation))
    _check(rc, "oracle_m2_backward")
    return out


# ------------------------------------------------------------------ Mamba-1
def mamba1_forward(x, dt_raw, A, B, C, s0=None, nthreads=None):
    x, dt_raw, A, B, C, s0 = map(_f64, (x, dt_raw, A, B, C, s0))
    b, T, D = x.shape
    N = A.shape[1]
    assert dt_raw.shape == (b, T, D) and A.shape == (D, N)
    assert B.shape == (b, T, N) and C.shape == (b, T, N)
    assert s0 is None or s0.shape == (b, D, N)
    y = np.empty_like(x)
    s_final = np.empty((b, D, N))
    rc = _load().oracle_m1_forward(b, T, D, N, _ptr(x), _ptr(dt_raw), _ptr(A), _ptr(B), _ptr(C), _ptr(s0),
                                   _ptr(y), _ptr(s_final), nthreads or default_threads())
    _check(rc, "oracle_m1_forward")
    return {"y": y, "s_final": s_final}


def mamba1_backward(dy, ds_final, x, dt_raw, A, B, C, s0=None, nthreads=None, mutation=0):
    dy, ds_final, x, dt_raw, A, B, C, s0 = map(_f64, (dy, ds_final, x, dt_raw, A, B, C, s0))
    b, T, D = x.shape
    N = A.shape[1]
    assert dy.shape == x.shape and ds_final.shape == (b, D, N)
    out = {"dx": np.empty_like(x), "ddt_raw": np.empty_like(dt_raw), "dA": np.empty_like(A),
           "dB": np.empty_like(B), "dC": np.empty_like(C), "ds0": np.empty((b, D, N))}
    rc = _load().oracle_m1_backward(b, T, D, N, _ptr(x), _ptr(dt_raw), _ptr(A), _ptr(B), _ptr(C), _ptr(s0),
                                    _ptr(dy), _ptr(ds_final), _ptr(out["dx"]), _ptr(out["ddt_raw"]),
                                    _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["ds0"]),
                                    nthreads or default_threads(), int(mutation))
    _check(rc, "oracle_m1_backward")
    return out


# --------------------------------------------------------------------- MIMO
def mimo_forward(v, da, B, C, s0=None, nthreads=None):
    v, da, B, C, s0 = map(_f64, (v, da, B, C, s0))
    b, T, R, H, P = v.shape
    N = B.shape[4]
    assert da.shape == (b, T, H) and B.shape == (b, T, R, H, N) and C.shape == B.shape
    assert s0 is None or s0.shape == (b, H, P, N)
    y = np.empty_like(v)
    s_final = np.empty((b, H, P, N))
    rc = _load().oracle_mimo_forward(b, T, R, H, P, N, _ptr(v), _ptr(da), _ptr(B), _ptr(C), _ptr(s0),
                                     _ptr(y), _ptr(s_final), nthreads or default_threads())
    _check(rc, "oracle_mimo_forward")
    return {"y": y, "s_final": s_final}


def mimo_backward(dy, ds_final, v, da, B, C, s0=None, nthreads=None, mutation=0):
    dy, ds_final, v, da, B, C, s0 = map(_f64, (dy, ds_final, v, da, B, C, s0))
    b, T, R, H, P = v.shape
    N = B.shape[4]
    assert dy.shape == v.shape and ds_final.shape == (b, H, P, N)
    out = {"dv": np.empty_like(v), "dda": np.empty_like(da), "dB": np.empty_like(B),
           "dC": np.empty_like(C), "ds0": np.empty((b, H, P, N))}
    rc = _load().oracle_mimo_backward(b, T, R, H, P, N, _ptr(v), _ptr(da), _ptr(B), _ptr(C), _ptr(s0),
                                      _ptr(dy), _ptr(ds_final), _ptr(out["dv"]), _ptr(out["dda"]),
                                      _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["ds0"]),
                                      nthreads or default_threads(), int(mutation))
    _check(rc, "oracle_mimo_backward")
    return out


# ------------------------------------------------------------- dispatchers
def forward(variant: str, inputs: dict, nthreads=None) -> dict:
    """Run the forward of ``variant`` ('mamba2' | 'mamba1' | 'mimo') on a dict
    of inputs named as in the library (x, dt_raw, A, B, C, s0)."""
    if variant == "mamba2":
        return mamba2_forward(inputs["x"], inputs["dt_raw"], inputs["A"], inputs["B"], inputs["C"],
                              inputs.get("s0"), nthreads)
    if variant == "mamba1":
        return mamba1_forward(inputs["x"], inputs["dt_raw"], inputs["A"], inputs["B"], inputs["C"],
                              inputs.get("s0"), nthreads)
    if variant == "mimo":
        return mimo_forward(inputs["x"], inputs["dt_raw"], inputs["B"], inputs["C"], inputs.get("s0"), nthreads)
    raise ValueError(variant)


def backward(variant: str, inputs: dict, nthreads=None, mutation=0) -> dict:
    """Backward of ``variant``; returns gradients named as the library's
    outputs (dx, ddt_raw, dA, dB, dC, ds0; for MIMO dx is dv, ddt_raw is dda
    and there is no dA)."""
    if variant == "mamba2":
        return mamba2_backward(inputs["dy"], inputs["ds_final"], inputs["x"], inputs["dt_raw"], inputs["A"],
                               inputs["B"], inputs["C"], inputs.get("s0"), nthreads, mutation)
    if variant == "mamba1":
        return mamba1_backward(inputs["dy"], inputs["ds_final"], inputs["x"], inputs["dt_raw"], inputs["A"],
                               inputs["B"], inputs["C"], inputs.get("s0"), nthreads, mutation)
    if variant == "mimo":
        out = mimo_backward(inputs["dy"], inputs["ds_final"], inputs["x"], inputs["dt_raw"], inputs["B"],
                            inputs["C"], inputs.get("s0"), nthreads, mutation)
        return {"dx": out["dv"], "ddt_raw": out["dda"], "dB": out["dB"], "dC": out["dC"], "ds0": out["ds0"]}
    raise ValueError(variant)
