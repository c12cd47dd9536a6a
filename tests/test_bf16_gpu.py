"""Forward with bf16 activations (m2scan_fwd_bf16) against the fp64 oracle on
the same bf16 inputs (needs a GB300).

Tolerance: the result is the fp32 computation rounded once to bfloat16 (8
significant bits), so |got - exact| <= 2^-8 |exact| (the rounding, with room
for the fp32 error before it) + 1e-5 absolute.
"""
import numpy as np
import pytest

import oracle
import gated_ssm_temporal_gb300 as g
from gated_ssm_temporal_gb300.workloads import WORKLOADS, Workload, make_inputs
from gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu


def run_and_check(x, gs=None):
    import torch
    ensure_built()
    hh = torch.from_numpy(x["h_history"]).cuda().to(torch.bfloat16)
    hs = torch.from_numpy(x["h_s2"]).cuda().to(torch.bfloat16)
    w = {k: torch.from_numpy(x[k]).cuda() for k in ("W_A", "W_B", "W_C", "W_O")}
    gt = None if gs is None else torch.tensor([gs], dtype=torch.float32, device="cuda")
    y = g.fwd_bf16(hh, hs, w["W_A"], w["W_B"], w["W_C"], w["W_O"], x["tw"], gate_scale=gt)
    torch.cuda.synchronize()
    got = y.float().cpu().numpy().astype(np.float64)
    ref = oracle.forward(hh.float().cpu().numpy(), hs.float().cpu().numpy(), x["W_A"], x["W_B"],
                         x["W_C"], x["W_O"], x["tw"], gate_scale=1.0 if gs is None else gs)
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-5
    bad = int((err > bound).sum())
    assert bad == 0, "%d elements beyond the bf16 bound, worst %.3e" % (bad, float(err.max()))
    return got, ref


def test_pages_workload():
    run_and_check(make_inputs(WORKLOADS["pages"]))


@pytest.mark.parametrize("B,K,SH2", [(1, 8, 256), (17, 8, 256), (153, 8, 64), (1000, 5, 128),
                                     (300, 64, 256), (40, 128, 192)])
def test_shapes(B, K, SH2):
    run_and_check(make_inputs(Workload("bf16", B, K, SH2, 16, 0.3, B + K)))


def test_gate_multiplier():
    run_and_check(make_inputs(Workload("bf16g", 500, 8, 256, 16, 0.3, 3)), gs=0.85)


def test_unsupported_shapes_are_rejected():
    import torch
    ensure_built()
    z = lambda *s: torch.zeros(s, device="cuda", dtype=torch.bfloat16)
    f = lambda *s: torch.zeros(s, device="cuda")
    with pytest.raises(g.M2ScanError):
        g.fwd_bf16(z(4, 8, 96), z(4, 96), f(96, 16), f(96, 16), f(96, 16), f(16, 96), 0.1)
    with pytest.raises(g.M2ScanError):
        g.fwd_bf16(z(4, 8, 64), z(4, 64), f(64, 8), f(64, 8), f(64, 8), f(8, 64), 0.1)
