"""The layer with the pages' per-feature blend output step (m2scan_fwd_blend /
m2scan_bwd_blend) against the fp64 oracle, on a shape of every kernel family
(needs a GB300)."""
import numpy as np
import pytest

import oracle
import gated_ssm_temporal_gb300 as g
from gated_ssm_temporal_gb300.workloads import Workload, make_inputs
from gpu_helpers import ensure_built, runs_wide, shape_of, to_dev
from tolerance import assert_outputs

pytestmark = pytest.mark.gpu

SHAPES = [
    (300, 8, 256, 16, False, True, None),
    (120, 5, 256, 16, False, True, 0.9),
    (200, 8, 128, 8, False, True, None),
    (100, 8, 32, 4, False, False, None),
    (300, 16, 512, 64, False, True, 0.9),
    (50, 8, 64, 16, True, True, None),
]


def run(x, w, gs, force_generic=False):
    import torch
    ensure_built()
    prev = g.m2scan_set_force_generic(1 if force_generic else 0)
    try:
        d = to_dev(x)
        wt = None if w is None else torch.from_numpy(w.astype(np.float32)).cuda()
        gt = None if gs is None else torch.tensor([gs], dtype=torch.float32, device="cuda")
        y = g.fwd_blend(d["h_history"], d["h_s2"], d["W_A"], d["W_B"], d["W_C"], wt, gt)
        gr = g.bwd_blend(d["h_history"], d["h_s2"], d["W_A"], d["W_B"], d["W_C"],
                         d["d_h_enriched"], wt, gt)
        torch.cuda.synchronize()
    finally:
        g.m2scan_set_force_generic(prev)
    out = {"h_enriched": y.cpu().numpy()}
    out.update({k: v.cpu().numpy() for k, v in gr.items()})
    return out


@pytest.mark.parametrize("B,K,SH2,D,generic,with_w,gs", SHAPES)
def test_blend_parity(B, K, SH2, D, generic, with_w, gs):
    x = make_inputs(Workload("blend", B, K, SH2, D, 1.0, B + 3 * K + D))
    w = np.random.default_rng(B).standard_normal(SH2) if with_w else None
    got = run(x, w, gs, generic)
    kw = dict(blend=True, gate_scale=1.0 if gs is None else gs, abs_terms=True)
    y, ya = oracle.forward(x["h_history"], x["h_s2"], x["W_A"], x["W_B"], x["W_C"], w, 1.0, **kw)
    ref = {"h_enriched": y, "h_enriched_abs": ya}
    ref.update(oracle.backward(x["h_history"], x["h_s2"], x["W_A"], x["W_B"], x["W_C"], w, 1.0,
                               x["d_h_enriched"], **kw))
    names = ["h_enriched", "d_h_history", "d_h_s2", "dW_A", "dW_B", "dW_C"]
    if with_w:
        # the weights' gradient is a sum over the batch, like dW_O, folded over the states
        got["dw"] = got["d_temporal_weight"]
        names.append("dw")
    else:
        assert "d_temporal_weight" not in got
    assert_outputs(got, ref, shape_of(x), names, wide=runs_wide(x, generic),
                   key_map={"dw": "dW_O"})


def test_blend_empty_batch_zero_fills_the_weight_gradient():
    import torch
    ensure_built()
    K, SH2, D = 8, 64, 16
    e = lambda *s: torch.zeros(s, device="cuda")
    w = torch.ones(SH2, device="cuda")
    gr = g.bwd_blend(e(0, K, SH2), e(0, SH2), e(SH2, D), e(SH2, D), e(SH2, D), e(0, SH2), w)
    torch.cuda.synchronize()
    assert torch.all(gr["d_temporal_weight"] == 0) and torch.all(gr["dW_A"] == 0)
