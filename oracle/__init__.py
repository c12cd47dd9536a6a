"""fp64 CPU oracle for the gated temporal scan layer and the bias-gradient
column sum (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The CUDA library never calls it and shares no
code with it.

The arithmetic lives in ``m2scan_oracle.c`` (plain C loops in float64, one
OpenMP-parallel loop over samples). This module only compiles that file with
gcc, loads it with ctypes and converts numpy arrays to float64 (an exact
up-cast of the float32 inputs the GPU sees).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "m2scan_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """Compile an oracle C source file into the shared library ``out``."""
    tmp = out + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` and return its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def open_library(path: str):
    """Load an oracle shared library and declare its entry points."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.m2o_scan_state.argtypes = [dp] * 5 + [i64, i32, i32, i32, dbl] + [dp] * 5
    lib.m2o_forward.argtypes = [dp] * 6 + [dbl, i64, i32, i32, i32, dbl, i32, dp, dp, i32]
    lib.m2o_backward.argtypes = ([dp] * 6 + [dbl, dp, i64, i32, i32, i32, dbl, i32]
                                 + [dp] * 9 + [i32])
    lib.m2o_bias_grad.argtypes = [dp, i64, i32, dp, i32, dp]
    for f in (lib.m2o_scan_state, lib.m2o_forward, lib.m2o_backward, lib.m2o_bias_grad):
        f.restype = ctypes.c_int
    return lib


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _dims(h_history, W_A):
    B, K, SH2 = h_history.shape
    D = W_A.shape[1]
    return B, K, SH2, D


def scan_state(h_history, h_s2, W_A, W_B, W_C, lib=None, gate_scale=1.0):
    """Per-sample intermediates: A, Bv, x (all [B,K,D]) and C, ctx ([B,D]).
    ``gate_scale`` multiplies every gate (the pages' optional gate multiplier)."""
    h, hs, wa, wb, wc = map(_f64, (h_history, h_s2, W_A, W_B, W_C))
    B, K, SH2, D = _dims(h, wa)
    A = np.empty((B, K, D)); Bv = np.empty((B, K, D)); x = np.empty((B, K, D))
    C = np.empty((B, D)); ctx = np.empty((B, D))
    rc = _load(lib).m2o_scan_state(_ptr(h), _ptr(hs), _ptr(wa), _ptr(wb), _ptr(wc),
                                B, K, SH2, D, float(gate_scale), _ptr(A), _ptr(Bv), _ptr(x),
                                _ptr(C), _ptr(ctx))
    if rc:
        raise RuntimeError("oracle scan_state failed (%d)" % rc)
    return A, Bv, x, C, ctx


def forward(h_history, h_s2, W_A, W_B, W_C, W_O, tw, n_threads=None, lib=None, gate_scale=1.0,
            blend=False, abs_terms=False):
    """h_enriched [B,SH2] in float64; ``gate_scale`` multiplies every gate.
    ``blend``: the pages' output step, W_O is then the per-feature weight
    vector w [SH2] (None: ones) and tw is ignored.
    ``abs_terms``: return (h_enriched, the per-element sum of the absolute
    values of the terms h_enriched adds up)."""
    h, hs, wa, wb, wc = map(_f64, (h_history, h_s2, W_A, W_B, W_C))
    B, K, SH2, D = _dims(h, wa)
    wo = _f64(np.ones(SH2) if W_O is None else W_O)
    out = np.empty((B, SH2))
    aout = np.empty((B, SH2)) if abs_terms else None
    rc = _load(lib).m2o_forward(_ptr(h), _ptr(hs), _ptr(wa), _ptr(wb), _ptr(wc), _ptr(wo),
                             float(tw), B, K, SH2, D, float(gate_scale), 1 if blend else 0,
                             _ptr(out), _ptr(aout) if abs_terms else None,
                             n_threads or default_threads())
    if rc:
        raise RuntimeError("oracle forward failed (%d)" % rc)
    return (out, aout) if abs_terms else out


def backward(h_history, h_s2, W_A, W_B, W_C, W_O, tw, d_h_enriched, n_threads=None,
             lib=None, gate_scale=1.0, blend=False, abs_terms=False):
    """Returns dict of float64 arrays: d_h_history, d_h_s2, dW_A, dW_B, dW_C, dW_O.
    ``gate_scale`` multiplies every gate (a constant: it gets no gradient).
    ``blend``: the pages' output step (see ``forward``); dW_O is then the
    gradient of the per-feature weights, [SH2].
    ``abs_terms``: also return, under the keys ``dW_A_abs`` ... ``dW_O_abs``,
    ``d_h_history_abs`` and ``d_h_s2_abs``, the per-element sums of the
    absolute values of the terms each output adds up (the scale that bounds
    the rounding error of an fp32 evaluation of those sums)."""
    h, hs, wa, wb, wc, g = map(_f64, (h_history, h_s2, W_A, W_B, W_C, d_h_enriched))
    B, K, SH2, D = _dims(h, wa)
    wo = _f64(np.ones(SH2) if W_O is None else W_O)
    out = {
        "d_h_history": np.empty((B, K, SH2)), "d_h_s2": np.empty((B, SH2)),
        "dW_A": np.empty((SH2, D)), "dW_B": np.empty((SH2, D)),
        "dW_C": np.empty((SH2, D)), "dW_O": np.empty((SH2,) if blend else (D, SH2)),
    }
    terms = np.zeros((4, SH2 * D)) if abs_terms else None
    adh = np.empty((B, K, SH2)) if abs_terms else None
    adhs = np.empty((B, SH2)) if abs_terms else None
    rc = _load(lib).m2o_backward(
        _ptr(h), _ptr(hs), _ptr(wa), _ptr(wb), _ptr(wc), _ptr(wo), float(tw), _ptr(g),
        B, K, SH2, D, float(gate_scale), 1 if blend else 0, _ptr(out["d_h_history"]), _ptr(out["d_h_s2"]), _ptr(out["dW_A"]),
        _ptr(out["dW_B"]), _ptr(out["dW_C"]), _ptr(out["dW_O"]),
        _ptr(terms) if abs_terms else None, _ptr(adh) if abs_terms else None,
        _ptr(adhs) if abs_terms else None, n_threads or default_threads())
    if rc:
        raise RuntimeError("oracle backward failed (%d)" % rc)
    if abs_terms:
        for i, k in enumerate(("dW_A", "dW_B", "dW_C", "dW_O")):
            out[k + "_abs"] = terms[i][:out[k].size].reshape(out[k].shape).copy()
        out["d_h_history_abs"] = adh
        out["d_h_s2_abs"] = adhs
    return out


def bias_grad(dy, db=None, accumulate=False, lib=None):
    """Column sums of dy [N, C] in float64 (plus db when accumulating): the
    bias gradient of a fully connected layer."""
    d = _f64(dy)
    if d.ndim != 2:
        raise ValueError("dy must be [N, C]")
    N, C = d.shape
    out = np.empty(C)
    dbi = _f64(db) if accumulate else np.zeros(C)
    rc = _load(lib).m2o_bias_grad(_ptr(d), N, C, _ptr(dbi), 1 if accumulate else 0, _ptr(out))
    if rc:
        raise RuntimeError("oracle bias_grad failed (%d)" % rc)
    return out
