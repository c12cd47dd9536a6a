"""ctypes binding of libm2scan.so (argument marshalling only).

The functions named like the C ABI (``m2scan_fwd`` ...) take raw device
addresses as Python ints. ``fwd``/``bwd`` accept torch CUDA tensors, allocate
outputs with torch when none are given and pass ``data_ptr()`` values and the
current torch stream to the library; every step of the layer runs in the
library's kernels. There is no fallback: if the library is missing or the
call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import build as _build

M2SCAN_OK = 0
STATUS_NAMES = {0: "M2SCAN_OK", 1: "M2SCAN_ERR_NULL", 2: "M2SCAN_ERR_SHAPE", 3: "M2SCAN_ERR_ALIGN",
                4: "M2SCAN_ERR_ALIAS", 5: "M2SCAN_ERR_WORKSPACE", 6: "M2SCAN_ERR_UNSUPPORTED",
                7: "M2SCAN_ERR_CUDA", 8: "M2SCAN_ERR_DEVICE"}

_lock = threading.Lock()
_lib = None


class M2ScanError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load_library()
        msg = lib.m2scan_status_str(status).decode()
        if status == 7:
            msg += " (cudaError %d)" % lib.m2scan_last_cuda_error()
        super().__init__("%s: %s (%s)" % (where, STATUS_NAMES.get(status, status), msg))
        self.status = status


def header_functions() -> list:
    """Names of the functions declared in include/m2scan.h."""
    text = open(os.path.join(_build.INCLUDE, "m2scan.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(m2scan_\w+)\s*\(", text)))


def load_library(path: str | None = None):
    """Load libm2scan.so (built in-tree by ``gated_ssm_temporal_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError("libm2scan.so not found at %s: build it first with "
                               "gated_ssm_temporal_gb300.build.build()" % path)
        lib = ctypes.CDLL(path)
        vp, i64, i32, f32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                 ctypes.c_float, ctypes.c_size_t)
        lib.m2scan_fwd.argtypes = [vp] * 6 + [f32, i64, i32, i32, i32, vp, vp]
        lib.m2scan_fwd.restype = ctypes.c_int
        lib.m2scan_fwd_ex.argtypes = [vp] * 6 + [f32, vp, i64, i32, i32, i32, vp, vp]
        lib.m2scan_fwd_ex.restype = ctypes.c_int
        lib.m2scan_bwd_ex.argtypes = ([vp] * 6 + [f32, vp, vp, i64, i32, i32, i32] + [vp] * 6
                                      + [vp, sz, vp])
        lib.m2scan_bwd_ex.restype = ctypes.c_int
        lib.m2scan_bwd.argtypes = ([vp] * 6 + [f32, vp, i64, i32, i32, i32] + [vp] * 6
                                   + [vp, sz, vp])
        lib.m2scan_bwd.restype = ctypes.c_int
        lib.m2scan_bwd_noalloc.argtypes = ([vp] * 6 + [f32, vp, i64, i32, i32, i32] + [vp] * 6
                                           + [vp])
        lib.m2scan_bwd_noalloc.restype = ctypes.c_int
        lib.m2scan_bwd_workspace_bytes.argtypes = [i64, i32, i32, i32]
        lib.m2scan_bwd_workspace_bytes.restype = sz
        lib.m2scan_status_str.argtypes = [ctypes.c_int]
        lib.m2scan_status_str.restype = ctypes.c_char_p
        lib.m2scan_last_cuda_error.argtypes = []
        lib.m2scan_last_cuda_error.restype = ctypes.c_int
        lib.m2scan_set_force_generic.argtypes = [ctypes.c_int]
        lib.m2scan_set_force_generic.restype = ctypes.c_int
        lib.m2scan_path_for.argtypes = [i32, i32, i32]
        lib.m2scan_path_for.restype = ctypes.c_int
        lib.m2scan_fwd_path_for.argtypes = [i32, i32, i32]
        lib.m2scan_fwd_path_for.restype = ctypes.c_int
        lib.m2scan_read_device_flags.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
        lib.m2scan_read_device_flags.restype = ctypes.c_int
        lib.m2scan_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp, vp]
        lib.m2scan_selftest_wait_timeout.restype = ctypes.c_int
        lib.m2scan_last_launch_count.argtypes = []
        lib.m2scan_last_launch_count.restype = ctypes.c_int
        lib.m2scan_bias_grad_workspace_bytes.argtypes = [i64, i32]
        lib.m2scan_bias_grad_workspace_bytes.restype = sz
        lib.m2scan_bias_grad.argtypes = [vp, i64, i32, vp, i32, vp, sz, vp]
        lib.m2scan_bias_grad.restype = ctypes.c_int
        lib.m2scan_fwd_bf16.argtypes = [vp] * 6 + [f32, vp, i64, i32, i32, i32, vp, vp]
        lib.m2scan_fwd_bf16.restype = ctypes.c_int
        lib.m2scan_bwd_bf16.argtypes = ([vp] * 6 + [f32, vp, vp, i64, i32, i32, i32] + [vp] * 6
                                        + [vp, sz, vp])
        lib.m2scan_bwd_bf16.restype = ctypes.c_int
        lib.m2scan_blend_fwd_workspace_bytes.argtypes = [i32, i32]
        lib.m2scan_blend_fwd_workspace_bytes.restype = sz
        lib.m2scan_blend_bwd_workspace_bytes.argtypes = [i64, i32, i32, i32]
        lib.m2scan_blend_bwd_workspace_bytes.restype = sz
        lib.m2scan_fwd_blend.argtypes = [vp] * 7 + [i64, i32, i32, i32, vp, vp, sz, vp]
        lib.m2scan_fwd_blend.restype = ctypes.c_int
        lib.m2scan_bwd_blend.argtypes = ([vp] * 8 + [i64, i32, i32, i32] + [vp] * 6
                                         + [vp, sz, vp])
        lib.m2scan_bwd_blend.restype = ctypes.c_int
        _lib = lib
        return lib


# ---------------------------------------------------------------- raw C ABI

def m2scan_fwd(h_history, h_s2, W_A, W_B, W_C, W_O, tw, B, K, SH2, D, h_enriched, stream=0):
    return load_library().m2scan_fwd(h_history, h_s2, W_A, W_B, W_C, W_O, float(tw), B, K, SH2,
                                     D, h_enriched, stream)


def m2scan_bwd(h_history, h_s2, W_A, W_B, W_C, W_O, tw, d_h_enriched, B, K, SH2, D,
               d_h_history, d_h_s2, dW_A, dW_B, dW_C, dW_O, workspace, workspace_bytes,
               stream=0):
    return load_library().m2scan_bwd(h_history, h_s2, W_A, W_B, W_C, W_O, float(tw),
                                     d_h_enriched, B, K, SH2, D, d_h_history, d_h_s2, dW_A,
                                     dW_B, dW_C, dW_O, workspace, workspace_bytes, stream)


def m2scan_fwd_ex(h_history, h_s2, W_A, W_B, W_C, W_O, tw, gate_scale, B, K, SH2, D, h_enriched,
                  stream=0):
    return load_library().m2scan_fwd_ex(h_history, h_s2, W_A, W_B, W_C, W_O, float(tw), gate_scale,
                                        B, K, SH2, D, h_enriched, stream)


def m2scan_bwd_ex(h_history, h_s2, W_A, W_B, W_C, W_O, tw, gate_scale, d_h_enriched, B, K, SH2,
                  D, d_h_history, d_h_s2, dW_A, dW_B, dW_C, dW_O, workspace, workspace_bytes,
                  stream=0):
    return load_library().m2scan_bwd_ex(h_history, h_s2, W_A, W_B, W_C, W_O, float(tw),
                                        gate_scale, d_h_enriched, B, K, SH2, D, d_h_history,
                                        d_h_s2, dW_A, dW_B, dW_C, dW_O, workspace,
                                        workspace_bytes, stream)


def m2scan_bwd_noalloc(h_history, h_s2, W_A, W_B, W_C, W_O, tw, d_h_enriched, B, K, SH2, D,
                       d_h_history, d_h_s2, dW_A, dW_B, dW_C, dW_O, stream=0):
    """m2scan_bwd for callers that cannot allocate: scratch is the library's static array."""
    return load_library().m2scan_bwd_noalloc(h_history, h_s2, W_A, W_B, W_C, W_O, float(tw),
                                             d_h_enriched, B, K, SH2, D, d_h_history, d_h_s2,
                                             dW_A, dW_B, dW_C, dW_O, stream)


NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


def m2scan_bwd_workspace_bytes(B, K, SH2, D):
    return load_library().m2scan_bwd_workspace_bytes(B, K, SH2, D)


def m2scan_bias_grad_workspace_bytes(N, C):
    return load_library().m2scan_bias_grad_workspace_bytes(N, C)


def m2scan_bias_grad(dy, N, C, db, accumulate, workspace, workspace_bytes, stream=0):
    return load_library().m2scan_bias_grad(dy, N, C, db, int(accumulate), workspace,
                                           workspace_bytes, stream)


def m2scan_status_str(status):
    return load_library().m2scan_status_str(status).decode()


def m2scan_last_cuda_error():
    return load_library().m2scan_last_cuda_error()


def m2scan_set_force_generic(force):
    return load_library().m2scan_set_force_generic(int(force))


def m2scan_path_for(K, SH2, D):
    return load_library().m2scan_path_for(K, SH2, D)


def m2scan_fwd_path_for(K, SH2, D):
    return load_library().m2scan_fwd_path_for(K, SH2, D)


def m2scan_read_device_flags():
    flags = ctypes.c_uint32(0)
    st = load_library().m2scan_read_device_flags(ctypes.byref(flags))
    if st != M2SCAN_OK:
        raise M2ScanError(st, "m2scan_read_device_flags")
    return flags.value


def m2scan_selftest_wait_timeout(limit_ns, out, stream=0):
    """Launches the wait-limit self-test; ``out`` is a device pointer to three uint64."""
    return load_library().m2scan_selftest_wait_timeout(limit_ns, out, stream)


def m2scan_last_launch_count():
    return load_library().m2scan_last_launch_count()


# ------------------------------------------------------- torch conveniences

def _check(t, name, shape):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32:
        raise TypeError("%s must be a float32 CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    return t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def dims_of(h_history, W_A):
    B, K, SH2 = (int(v) for v in h_history.shape)
    return B, K, SH2, int(W_A.shape[1])


def _gate_ptr(gate_scale):
    return 0 if gate_scale is None else _check(gate_scale, "gate_scale", (1,))


def fwd(h_history, h_s2, W_A, W_B, W_C, W_O, tw, out=None, stream=None, gate_scale=None):
    """h_enriched [B,SH2] = layer forward; all tensors float32 CUDA, contiguous.
    ``gate_scale``: optional one-element tensor g multiplying every gate."""
    import torch
    B, K, SH2, D = dims_of(h_history, W_A)
    if out is None:
        out = torch.empty((B, SH2), device=h_history.device, dtype=torch.float32)
    st = m2scan_fwd_ex(_check(h_history, "h_history", (B, K, SH2)), _check(h_s2, "h_s2", (B, SH2)),
                       _check(W_A, "W_A", (SH2, D)), _check(W_B, "W_B", (SH2, D)),
                       _check(W_C, "W_C", (SH2, D)), _check(W_O, "W_O", (D, SH2)), tw,
                       _gate_ptr(gate_scale), B, K, SH2, D, _check(out, "h_enriched", (B, SH2)),
                       _stream(stream))
    if st != M2SCAN_OK:
        raise M2ScanError(st, "m2scan_fwd")
    return out


def alloc_bwd_outputs(B, K, SH2, D, device):
    import torch
    f = dict(device=device, dtype=torch.float32)
    return {"d_h_history": torch.empty((B, K, SH2), **f), "d_h_s2": torch.empty((B, SH2), **f),
            "dW_A": torch.empty((SH2, D), **f), "dW_B": torch.empty((SH2, D), **f),
            "dW_C": torch.empty((SH2, D), **f), "dW_O": torch.empty((D, SH2), **f)}


def alloc_workspace(B, K, SH2, D, device):
    import torch
    n = m2scan_bwd_workspace_bytes(B, K, SH2, D)
    return torch.empty((max(n, 16) + 3) // 4, device=device, dtype=torch.float32)


def bwd(h_history, h_s2, W_A, W_B, W_C, W_O, tw, d_h_enriched, outs=None, workspace=None,
        stream=None, gate_scale=None):
    """Layer backward; returns dict d_h_history, d_h_s2, dW_A, dW_B, dW_C, dW_O.
    ``gate_scale``: optional one-element tensor g multiplying every gate."""
    B, K, SH2, D = dims_of(h_history, W_A)
    if outs is None:
        outs = alloc_bwd_outputs(B, K, SH2, D, h_history.device)
    if workspace is None:
        workspace = alloc_workspace(B, K, SH2, D, h_history.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = m2scan_bwd_ex(
        _check(h_history, "h_history", (B, K, SH2)), _check(h_s2, "h_s2", (B, SH2)),
        _check(W_A, "W_A", (SH2, D)), _check(W_B, "W_B", (SH2, D)),
        _check(W_C, "W_C", (SH2, D)), _check(W_O, "W_O", (D, SH2)), tw, _gate_ptr(gate_scale),
        _check(d_h_enriched, "d_h_enriched", (B, SH2)), B, K, SH2, D,
        _check(outs["d_h_history"], "d_h_history", (B, K, SH2)),
        _check(outs["d_h_s2"], "d_h_s2", (B, SH2)), _check(outs["dW_A"], "dW_A", (SH2, D)),
        _check(outs["dW_B"], "dW_B", (SH2, D)), _check(outs["dW_C"], "dW_C", (SH2, D)),
        _check(outs["dW_O"], "dW_O", (D, SH2)), workspace.data_ptr(), ws_bytes, _stream(stream))
    if st != M2SCAN_OK:
        raise M2ScanError(st, "m2scan_bwd")
    return outs


def bias_grad(dy, db=None, accumulate=False, workspace=None, stream=None):
    """db [C] = column sums of dy [N, C] (added into db when ``accumulate``);
    float32 CUDA tensors, contiguous. Returns db."""
    import torch
    if dy.dim() != 2:
        raise ValueError("dy must be [N, C]")
    N, C = (int(v) for v in dy.shape)
    if db is None:
        if accumulate:
            raise ValueError("accumulate needs db")
        db = torch.empty((C,), device=dy.device, dtype=torch.float32)
    need = m2scan_bias_grad_workspace_bytes(N, C)
    if workspace is None:
        workspace = torch.empty((max(1, need // 4),), device=dy.device, dtype=torch.float32)
    st = m2scan_bias_grad(_check(dy, "dy", (N, C)), N, C, _check(db, "db", (C,)),
                          accumulate, workspace.data_ptr(), workspace.numel() * 4,
                          _stream(stream))
    if st != M2SCAN_OK:
        raise M2ScanError(st, "m2scan_bias_grad")
    return db


def m2scan_blend_fwd_workspace_bytes(SH2, D):
    return load_library().m2scan_blend_fwd_workspace_bytes(SH2, D)


def m2scan_blend_bwd_workspace_bytes(B, K, SH2, D):
    return load_library().m2scan_blend_bwd_workspace_bytes(B, K, SH2, D)


def m2scan_fwd_blend(h_history, h_s2, W_A, W_B, W_C, temporal_weight, gate_scale, B, K, SH2, D,
                     h_enriched, workspace, workspace_bytes, stream=0):
    return load_library().m2scan_fwd_blend(h_history, h_s2, W_A, W_B, W_C, temporal_weight,
                                           gate_scale, B, K, SH2, D, h_enriched, workspace,
                                           workspace_bytes, stream)


def m2scan_bwd_blend(h_history, h_s2, W_A, W_B, W_C, temporal_weight, gate_scale, d_h_enriched,
                     B, K, SH2, D, d_h_history, d_h_s2, dW_A, dW_B, dW_C, d_temporal_weight,
                     workspace, workspace_bytes, stream=0):
    return load_library().m2scan_bwd_blend(h_history, h_s2, W_A, W_B, W_C, temporal_weight,
                                           gate_scale, d_h_enriched, B, K, SH2, D, d_h_history,
                                           d_h_s2, dW_A, dW_B, dW_C, d_temporal_weight,
                                           workspace, workspace_bytes, stream)


def fwd_blend(h_history, h_s2, W_A, W_B, W_C, temporal_weight=None, gate_scale=None, out=None,
              stream=None):
    """The layer with the pages' per-feature blend output step:
    h_enriched = h_s2 + w[j] * (sum_s ctx_s) / D, w = ``temporal_weight`` [SH2] (None: ones)."""
    import torch
    B, K, SH2, D = dims_of(h_history, W_A)
    if out is None:
        out = torch.empty((B, SH2), device=h_history.device, dtype=torch.float32)
    need = m2scan_blend_fwd_workspace_bytes(SH2, D)
    ws = torch.empty((max(1, need // 4),), device=h_history.device, dtype=torch.float32)
    tw = 0 if temporal_weight is None else _check(temporal_weight, "temporal_weight", (SH2,))
    st = m2scan_fwd_blend(_check(h_history, "h_history", (B, K, SH2)), _check(h_s2, "h_s2", (B, SH2)),
                          _check(W_A, "W_A", (SH2, D)), _check(W_B, "W_B", (SH2, D)),
                          _check(W_C, "W_C", (SH2, D)), tw, _gate_ptr(gate_scale), B, K, SH2, D,
                          _check(out, "h_enriched", (B, SH2)), ws.data_ptr(), ws.numel() * 4,
                          _stream(stream))
    if st != M2SCAN_OK:
        raise M2ScanError(st, "m2scan_fwd_blend")
    return out


def bwd_blend(h_history, h_s2, W_A, W_B, W_C, d_h_enriched, temporal_weight=None, gate_scale=None,
              stream=None):
    """Backward of ``fwd_blend``: dict d_h_history, d_h_s2, dW_A, dW_B, dW_C and, when
    ``temporal_weight`` is given, d_temporal_weight [SH2]."""
    import torch
    B, K, SH2, D = dims_of(h_history, W_A)
    dev = h_history.device
    outs = {"d_h_history": torch.empty((B, K, SH2), device=dev), "d_h_s2": torch.empty((B, SH2), device=dev),
            "dW_A": torch.empty((SH2, D), device=dev), "dW_B": torch.empty((SH2, D), device=dev),
            "dW_C": torch.empty((SH2, D), device=dev)}
    dtw = 0
    if temporal_weight is not None:
        outs["d_temporal_weight"] = torch.empty((SH2,), device=dev)
        dtw = outs["d_temporal_weight"].data_ptr()
    need = m2scan_blend_bwd_workspace_bytes(B, K, SH2, D)
    ws = torch.empty((max(1, need // 4),), device=dev, dtype=torch.float32)
    tw = 0 if temporal_weight is None else _check(temporal_weight, "temporal_weight", (SH2,))
    st = m2scan_bwd_blend(
        _check(h_history, "h_history", (B, K, SH2)), _check(h_s2, "h_s2", (B, SH2)),
        _check(W_A, "W_A", (SH2, D)), _check(W_B, "W_B", (SH2, D)), _check(W_C, "W_C", (SH2, D)),
        tw, _gate_ptr(gate_scale), _check(d_h_enriched, "d_h_enriched", (B, SH2)), B, K, SH2, D,
        outs["d_h_history"].data_ptr(), outs["d_h_s2"].data_ptr(), outs["dW_A"].data_ptr(),
        outs["dW_B"].data_ptr(), outs["dW_C"].data_ptr(), dtw, ws.data_ptr(), ws.numel() * 4,
        _stream(stream))
    if st != M2SCAN_OK:
        raise M2ScanError(st, "m2scan_bwd_blend")
    return outs


def m2scan_fwd_bf16(h_history, h_s2, W_A, W_B, W_C, W_O, tw, gate_scale, B, K, SH2, D, h_enriched,
                    stream=0):
    return load_library().m2scan_fwd_bf16(h_history, h_s2, W_A, W_B, W_C, W_O, float(tw),
                                          gate_scale, B, K, SH2, D, h_enriched, stream)


def m2scan_bwd_bf16(h_history, h_s2, W_A, W_B, W_C, W_O, tw, gate_scale, d_h_enriched, B, K, SH2,
                    D, d_h_history, d_h_s2, dW_A, dW_B, dW_C, dW_O, workspace, workspace_bytes,
                    stream=0):
    return load_library().m2scan_bwd_bf16(h_history, h_s2, W_A, W_B, W_C, W_O, float(tw),
                                          gate_scale, d_h_enriched, B, K, SH2, D, d_h_history,
                                          d_h_s2, dW_A, dW_B, dW_C, dW_O, workspace,
                                          workspace_bytes, stream)


def _check_bf16(t, name, shape):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16:
        raise TypeError("%s must be a bfloat16 CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    return t.data_ptr()


def fwd_bf16(h_history, h_s2, W_A, W_B, W_C, W_O, tw, out=None, stream=None, gate_scale=None):
    """Layer forward with bfloat16 h_history, h_s2 and h_enriched (fp32 weights and sums)."""
    import torch
    B, K, SH2, D = dims_of(h_history, W_A)
    if out is None:
        out = torch.empty((B, SH2), device=h_history.device, dtype=torch.bfloat16)
    st = m2scan_fwd_bf16(_check_bf16(h_history, "h_history", (B, K, SH2)),
                         _check_bf16(h_s2, "h_s2", (B, SH2)), _check(W_A, "W_A", (SH2, D)),
                         _check(W_B, "W_B", (SH2, D)), _check(W_C, "W_C", (SH2, D)),
                         _check(W_O, "W_O", (D, SH2)), tw, _gate_ptr(gate_scale), B, K, SH2, D,
                         _check_bf16(out, "h_enriched", (B, SH2)), _stream(stream))
    if st != M2SCAN_OK:
        raise M2ScanError(st, "m2scan_fwd_bf16")
    return out


def bwd_bf16(h_history, h_s2, W_A, W_B, W_C, W_O, tw, d_h_enriched, outs=None, workspace=None,
             stream=None, gate_scale=None):
    """Layer backward with bfloat16 h_history, h_s2, d_h_enriched in and bfloat16
    d_h_history, d_h_s2 out; fp32 weights, weight gradients and sums. Returns
    the dict of ``bwd``."""
    import torch
    B, K, SH2, D = dims_of(h_history, W_A)
    if outs is None:
        f = dict(device=h_history.device, dtype=torch.float32)
        b = dict(device=h_history.device, dtype=torch.bfloat16)
        outs = {"d_h_history": torch.empty((B, K, SH2), **b), "d_h_s2": torch.empty((B, SH2), **b),
                "dW_A": torch.empty((SH2, D), **f), "dW_B": torch.empty((SH2, D), **f),
                "dW_C": torch.empty((SH2, D), **f), "dW_O": torch.empty((D, SH2), **f)}
    if workspace is None:
        workspace = alloc_workspace(B, K, SH2, D, h_history.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = m2scan_bwd_bf16(
        _check_bf16(h_history, "h_history", (B, K, SH2)), _check_bf16(h_s2, "h_s2", (B, SH2)),
        _check(W_A, "W_A", (SH2, D)), _check(W_B, "W_B", (SH2, D)),
        _check(W_C, "W_C", (SH2, D)), _check(W_O, "W_O", (D, SH2)), tw, _gate_ptr(gate_scale),
        _check_bf16(d_h_enriched, "d_h_enriched", (B, SH2)), B, K, SH2, D,
        _check_bf16(outs["d_h_history"], "d_h_history", (B, K, SH2)),
        _check_bf16(outs["d_h_s2"], "d_h_s2", (B, SH2)), _check(outs["dW_A"], "dW_A", (SH2, D)),
        _check(outs["dW_B"], "dW_B", (SH2, D)), _check(outs["dW_C"], "dW_C", (SH2, D)),
        _check(outs["dW_O"], "dW_O", (D, SH2)), workspace.data_ptr(), ws_bytes, _stream(stream))
    if st != M2SCAN_OK:
        raise M2ScanError(st, "m2scan_bwd_bf16")
    return outs
