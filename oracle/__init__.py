"""CPU oracle for the chunked gated-delta-rule forward (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this package. The CUDA library never includes,
links or calls anything here; the two share no code. The one thing both sides
use is the seeded input generator module, which holds no arithmetic of the
method.

Contents
--------
* ``gdn_ref.c`` -- the definition: a plain fp64 token-by-token recurrence in
  C (see its header for the equations and the pages they follow), and the
  exact adjoint of each of its steps for the backward pass.
  ``recurrent_forward`` and ``recurrent_backward`` below are their ctypes
  wrappers.
* ``chunked.py`` -- an independent fp64 NumPy/SciPy chunked formulation, used
  only as a pin of the token recurrence (a different algorithm for the same
  function).
* ``chunk_table.py`` -- the CPU builder of the (sequence id, chunk ordinal)
  table with sentinel slots.

Parity status: every function here is pinned by tests in ``tests/`` against
exact rationals, closed forms, invariants and the independent formulation.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_ref.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgdn_ref.so")
_lock = threading.Lock()
_lib = None


def compile_library(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile a C oracle source into a shared library with gcc (fp64, no fast-math)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", *extra_flags, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True)
    return out


def build() -> str:
    """Build the oracle library if it is missing or older than its source."""
    with _lock:
        if (not os.path.exists(_LIB_PATH)
                or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
            compile_library()
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    i64, dbl, ptr = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
    lib.gdn_ref_forward.argtypes = [i64, i64, i64, i64, i64, i64,
                                    ptr, ptr, ptr, ptr, ptr, dbl, ptr, ptr,
                                    ctypes.c_int, dbl, ptr, ptr, ctypes.c_int, ctypes.c_int]
    lib.gdn_ref_forward.restype = ctypes.c_int
    lib.gdn_ref_backward.argtypes = [i64, i64, i64, i64, i64, i64,
                                     ptr, ptr, ptr, ptr, ptr, dbl, ptr, ptr, ptr, ptr,
                                     ptr, ptr, ptr, ptr, ptr, ptr, ctypes.c_int]
    lib.gdn_ref_backward.restype = ctypes.c_int
    lib.gdn_ref_max_threads.argtypes = []
    lib.gdn_ref_max_threads.restype = ctypes.c_int
    return lib


def load_library(path: str | None = None):
    """Return the ctypes handle of the oracle (building the default one if needed)."""
    global _lib
    if path is not None:
        return _bind(path)
    if _lib is None:
        _lib = _bind(build())
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: exact upconversion of its stored dtype
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def recurrent_forward(q, k, v, g, beta, scale=None, initial_state=None,
                      cu_seqlens=None, qk_l2norm=False, eps=1e-6,
                      output_final_state=True, nthreads=0, lib=None,
                      out_init=None):
    """Token-by-token fp64 gated delta rule (the oracle's definition).

    Shapes follow the library boundary: q, k [T, H, dk]; v [T, Hv, dv];
    g, beta [T, Hv] (g may be [T, Hv, dk]: one log-decay per key channel);
    initial_state [N, Hv, dv, dk] (or None for zeros);
    cu_seqlens [N+1] (or None for one sequence of T rows).
    Returns (out [T, Hv, dv], final_state [N, Hv, dv, dk] or None), fp64.
    ``out_init`` fills rows the recurrence does not touch (default zeros).
    """
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    T, H, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    per_channel = g.ndim == 3
    if per_channel and g.shape != (T, Hv, dk):
        raise ValueError("per-channel gates must be [T, Hv, dk]")
    if cu_seqlens is None:
        N, cu = 1, None
    else:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
            dtype=np.int64))
        N = cu.shape[0] - 1
    s0 = _f64(initial_state)
    out = (np.zeros((T, Hv, dv)) if out_init is None
           else np.array(_f64(out_init), dtype=np.float64, copy=True))
    fin = np.zeros((N, Hv, dv, dk)) if output_final_state else None
    if scale is None:
        scale = 0.0  # the oracle maps <= 0 to 1/sqrt(dk)
    lib = lib or load_library()
    rc = lib.gdn_ref_forward(T, N, H, Hv, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                             _ptr(beta), float(scale), _ptr(s0), _ptr(cu),
                             int(bool(qk_l2norm)), float(eps), _ptr(out), _ptr(fin),
                             int(nthreads), int(per_channel))
    if rc != 0:
        raise ValueError(f"gdn_ref_forward rejected its arguments (rc={rc})")
    return out, fin


def recurrent_backward(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None,
                       d_out=None, d_final=None, nthreads=0, lib=None):
    """Gradients of the token recurrence (scalar gates, no L2 norm) in fp64.

    d_out [T, Hv, dv] is the gradient with respect to out, d_final [N, Hv, dv, dk]
    (or None) with respect to final_state. Returns a dict with dq, dk [T, H, dk],
    dv [T, Hv, dv], dg, dbeta [T, Hv] and d_initial [N, Hv, dv, dk]; rows outside
    the sequences get zeros."""
    q, k, v, g, beta, d_out = (_f64(a) for a in (q, k, v, g, beta, d_out))
    T, H, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    if g.ndim != 2:
        raise ValueError("the backward takes one gate per token and value head")
    if cu_seqlens is None:
        N, cu = 1, None
    else:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
            dtype=np.int64))
        N = cu.shape[0] - 1
    s0, dfin = _f64(initial_state), _f64(d_final)
    out = dict(dq=np.zeros((T, H, dk)), dk=np.zeros((T, H, dk)), dv=np.zeros((T, Hv, dv)),
               dg=np.zeros((T, Hv)), dbeta=np.zeros((T, Hv)), d_initial=np.zeros((N, Hv, dv, dk)))
    lib = lib or load_library()
    rc = lib.gdn_ref_backward(T, N, H, Hv, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                              _ptr(beta), float(scale or 0.0), _ptr(s0), _ptr(cu), _ptr(d_out),
                              _ptr(dfin), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
                              _ptr(out["dg"]), _ptr(out["dbeta"]), _ptr(out["d_initial"]),
                              int(nthreads))
    if rc != 0:
        raise ValueError(f"gdn_ref_backward rejected its arguments (rc={rc})")
    return out


def max_threads(lib=None) -> int:
    return int((lib or load_library()).gdn_ref_max_threads())
