"""The layer with the pages' optional gate multiplier (m2scan_fwd_ex /
m2scan_bwd_ex, every gate g * sigmoid(A_t)) against the fp64 oracle, on a
shape of every kernel family (needs a GB300)."""
import numpy as np
import pytest

import gated_ssm_temporal_gb300 as g
from gated_ssm_temporal_gb300.workloads import Workload, make_inputs
from gpu_helpers import OUTPUTS, ensure_built, oracle_all, runs_wide, shape_of, to_dev
from tolerance import assert_outputs

pytestmark = pytest.mark.gpu

SHAPES = [
    (300, 8, 256, 16, False),   # tensor-core kernels, K % 8 == 0
    (120, 5, 256, 16, False),   # tensor-core kernels, K % 8 != 0
    (40, 64, 256, 16, False),   # long history
    (200, 8, 128, 8, False),    # D = 8: tensor-core forward, FP32 backward
    (100, 8, 32, 4, False),     # D = 4: FP32 kernels
    (300, 16, 512, 64, False),  # wide states
    (50, 8, 64, 16, True),      # generic kernels
]


def run(x, gs, force_generic=False):
    import torch
    ensure_built()
    prev = g.m2scan_set_force_generic(1 if force_generic else 0)
    try:
        d = to_dev(x)
        gt = None if gs is None else torch.tensor([gs], dtype=torch.float32, device="cuda")
        y = g.fwd(d["h_history"], d["h_s2"], d["W_A"], d["W_B"], d["W_C"], d["W_O"], d["tw"],
                  gate_scale=gt)
        gr = g.bwd(d["h_history"], d["h_s2"], d["W_A"], d["W_B"], d["W_C"], d["W_O"], d["tw"],
                   d["d_h_enriched"], gate_scale=gt)
        torch.cuda.synchronize()
    finally:
        g.m2scan_set_force_generic(prev)
    out = {"h_enriched": y.cpu().numpy()}
    out.update({k: gr[k].cpu().numpy() for k in OUTPUTS})
    return out


def reference(x, gs):
    return oracle_all(x, gate_scale=gs)


NAMES = ("h_enriched",) + OUTPUTS


@pytest.mark.parametrize("B,K,SH2,D,generic", SHAPES)
def test_gate_multiplier_parity(B, K, SH2, D, generic):
    x = make_inputs(Workload("gate", B, K, SH2, D, 0.3, B + K + D))
    got, ref = run(x, 0.85, generic), reference(x, 0.85)
    assert_outputs(got, ref, shape_of(x), NAMES, wide=runs_wide(x, generic))


def test_gate_multiplier_zero_keeps_only_the_last_step():
    # g = 0: x_{K-1} = B_{K-1}; W_A then gets no gradient at all
    x = make_inputs(Workload("gate0", 64, 8, 256, 16, 0.3, 5))
    got, ref = run(x, 0.0), reference(x, 0.0)
    assert_outputs(got, ref, shape_of(x), NAMES)
    assert np.all(got["dW_A"] == 0.0)


def test_gate_multiplier_one_is_the_plain_layer():
    x = make_inputs(Workload("gate1", 200, 8, 256, 16, 0.3, 6))
    a, b = run(x, 1.0), run(x, None)
    for n in a:
        assert np.array_equal(a[n], b[n]), n
