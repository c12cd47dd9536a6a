"""Runs the CUDA path on numpy inputs (through the C ABI) and returns numpy results."""
import numpy as np

import gated_ssm_temporal_gb300 as g
from gated_ssm_temporal_gb300 import build as gbuild

OUTPUTS = ("d_h_history", "d_h_s2", "dW_A", "dW_B", "dW_C", "dW_O")
NAMES_ALL = ("h_enriched",) + OUTPUTS


def ensure_built():
    gbuild.build()
    g.load_library()


def to_dev(x):
    import torch
    return {k: (torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).cuda()
                if isinstance(v, np.ndarray) else v) for k, v in x.items()}


def run_fwd(d):
    return g.fwd(d["h_history"], d["h_s2"], d["W_A"], d["W_B"], d["W_C"], d["W_O"], d["tw"])


def run_bwd(d, outs=None, workspace=None, stream=None):
    return g.bwd(d["h_history"], d["h_s2"], d["W_A"], d["W_B"], d["W_C"], d["W_O"], d["tw"],
                 d["d_h_enriched"], outs=outs, workspace=workspace, stream=stream)


def run_all(x, force_generic=False):
    import torch
    ensure_built()
    prev = g.m2scan_set_force_generic(1 if force_generic else 0)
    try:
        d = to_dev(x)
        y = run_fwd(d)
        gr = run_bwd(d)
        torch.cuda.synchronize()
        out = {"h_enriched": y.cpu().numpy()}
        out.update({k: gr[k].cpu().numpy() for k in OUTPUTS})
    finally:
        g.m2scan_set_force_generic(prev)
    return out


def oracle_all(x, **kw):
    """The oracle's outputs and, under ``<name>_abs``, the sums of the absolute
    values of each output's terms (the error scale of the parity bound)."""
    import oracle
    y, ya = oracle.forward(x["h_history"], x["h_s2"], x["W_A"], x["W_B"], x["W_C"], x["W_O"],
                           x["tw"], abs_terms=True, **kw)
    ref = {"h_enriched": y, "h_enriched_abs": ya}
    ref.update(oracle.backward(x["h_history"], x["h_s2"], x["W_A"], x["W_B"], x["W_C"],
                               x["W_O"], x["tw"], x["d_h_enriched"], abs_terms=True, **kw))
    return ref


def shape_of(x):
    B, K, SH2 = x["h_history"].shape
    return int(B), int(K), int(SH2), int(x["W_A"].shape[1])


def runs_wide(x, force_generic=False):
    """Whether the backward of these shapes runs the wide-state family (its
    own sample ranges for the weight gradients, as many as the slots)."""
    ensure_built()
    B, K, SH2, D = shape_of(x)
    return not force_generic and g.m2scan_path_for(K, SH2, D) == 3
