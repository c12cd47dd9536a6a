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


# ------------------------------------------------------------------ backward
# d_h_history and d_h_s2 are rounded once to bfloat16: the bound of the
# forward. The weight gradients stay fp32 sums of products of exact fp32
# values (a bf16 input is exact in fp32): the fp32 criteria of the layer.

def run_bwd_and_check(x, gs=None):
    import torch
    from tolerance import assert_outputs
    ensure_built()
    bf = lambda k: torch.from_numpy(x[k]).cuda().to(torch.bfloat16)
    hh, hs, dy = bf("h_history"), bf("h_s2"), bf("d_h_enriched")
    w = {k: torch.from_numpy(x[k]).cuda() for k in ("W_A", "W_B", "W_C", "W_O")}
    gt = None if gs is None else torch.tensor([gs], dtype=torch.float32, device="cuda")
    out = g.bwd_bf16(hh, hs, w["W_A"], w["W_B"], w["W_C"], w["W_O"], x["tw"], dy, gate_scale=gt)
    torch.cuda.synchronize()
    assert g.m2scan_last_launch_count() == (2 if x["h_history"].shape[0] else 0)
    assert out["d_h_history"].dtype == torch.bfloat16 and out["dW_A"].dtype == torch.float32
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)
    ref = oracle.backward(f64(hh), f64(hs), x["W_A"], x["W_B"], x["W_C"], x["W_O"], x["tw"],
                          f64(dy), gate_scale=1.0 if gs is None else gs, abs_terms=True)
    for name in ("d_h_history", "d_h_s2"):
        got = f64(out[name])
        err = np.abs(got - ref[name])
        bound = 2.0 ** -8 * np.abs(ref[name]) + 1e-5
        bad = int((err > bound).sum())
        assert bad == 0, "%s: %d elements beyond the bf16 bound, worst %.3e" % (
            name, bad, float(err.max()) if err.size else 0.0)
    B, K, SH2 = x["h_history"].shape
    got = {k: out[k].cpu().numpy() for k in ("dW_A", "dW_B", "dW_C", "dW_O")}
    assert_outputs(got, ref, (B, K, SH2, x["W_A"].shape[1]), list(got), context={"test": "bf16"})
    return out


def test_bwd_pages_workload():
    run_bwd_and_check(make_inputs(WORKLOADS["pages"]))


@pytest.mark.parametrize("B,K,SH2,D", [(1, 8, 256, 16), (17, 8, 256, 16), (153, 3, 96, 8),
                                       (1000, 5, 128, 16), (300, 64, 256, 16), (40, 128, 64, 4),
                                       (37, 8, 512, 64), (5, 1, 36, 3)])
def test_bwd_shapes(B, K, SH2, D):
    run_bwd_and_check(make_inputs(Workload("bf16b", B, K, SH2, D, 0.3, B + K + D, 2.0)))


@pytest.mark.parametrize("B,K,SH2", [(2000, 8, 64), (3000, 3, 192), (777, 128, 128),
                                     (461, 8, 256), (5000, 1, 256), (1234, 24, 128)])
def test_bwd_tensor_core_shapes(B, K, SH2):
    # D = 16 runs the tensor-core kernel: one to four 64-column blocks, tiles
    # of 1 to 16 samples (K = 128 down to 1), K % 8 == 0 (the packed dA|dB
    # stores) and not, ragged tile splits (B = 461: three or four tiles per CTA)
    run_bwd_and_check(make_inputs(Workload("bf16tc", B, K, SH2, 16, 0.3, B + K + SH2, 2.0)))


@pytest.mark.parametrize("sign", [-1.0, 1.0])
def test_bwd_saturated_gates(sign):
    x = make_inputs(Workload("bf16sat", 300, 8, 256, 16, 0.3, 31))
    x["h_history"][:, :, 0] = 1.0
    x["W_A"][0, :] = 50.0 * sign
    run_bwd_and_check(x)


def test_bwd_heavy_tailed_history():
    run_bwd_and_check(make_inputs(Workload("bf16ht", 500, 8, 256, 16, 0.1, 32, 1.0, 10.0)))


def test_bwd_gate_multiplier():
    run_bwd_and_check(make_inputs(Workload("bf16bg", 500, 8, 256, 16, 0.3, 5)), gs=0.85)


def test_bwd_weight_gradients_are_reproducible():
    x = make_inputs(Workload("bf16br", 2000, 8, 256, 16, 0.3, 9))
    a = run_bwd_and_check(x)
    b = run_bwd_and_check(x)
    for name in ("dW_A", "dW_B", "dW_C", "dW_O", "d_h_history", "d_h_s2"):
        assert bool((a[name] == b[name]).all()), name


def test_bwd_empty_batch_zeroes_weight_gradients():
    import torch
    ensure_built()
    z = lambda *s: torch.zeros(s, device="cuda", dtype=torch.bfloat16)
    f = lambda *s: torch.ones(s, device="cuda")
    out = g.bwd_bf16(z(0, 8, 256), z(0, 256), f(256, 16), f(256, 16), f(256, 16), f(16, 256), 0.1,
                     z(0, 256))
    torch.cuda.synchronize()
    assert g.m2scan_last_launch_count() == 0
    for name in ("dW_A", "dW_B", "dW_C", "dW_O"):
        assert float(out[name].abs().max()) == 0.0
