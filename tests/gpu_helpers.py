"""Runs the CUDA path on numpy inputs (through the C ABI) and returns numpy results."""
import numpy as np

import gated_ssm_temporal_gb300 as g
from gated_ssm_temporal_gb300 import build as gbuild

OUTPUTS = ("d_h_history", "d_h_s2", "dW_A", "dW_B", "dW_C", "dW_O")


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


def oracle_all(x):
    import oracle
    ref = {"h_enriched": oracle.forward(x["h_history"], x["h_s2"], x["W_A"], x["W_B"],
                                        x["W_C"], x["W_O"], x["tw"])}
    ref.update(oracle.backward(x["h_history"], x["h_s2"], x["W_A"], x["W_B"], x["W_C"],
                               x["W_O"], x["tw"], x["d_h_enriched"]))
    return ref
