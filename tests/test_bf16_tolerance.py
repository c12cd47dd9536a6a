"""Calibration of the bf16 parity bound |got - exact| <= 2^-8 |exact| + 1e-5.

A bf16 result is the fp32 result rounded once to nearest even: 8
significant bits, so the rounding alone is at most 2^-9 relative, and the
fp32 error before it is far smaller. The bound must admit that, and must
reject a conversion that truncates instead of rounding (error up to 2^-7
relative), the plausible mistake in a hand-written bf16 store. Checked on
the oracle's own outputs for the layer's inputs, forward and backward.
"""
import numpy as np

import oracle
from gated_ssm_temporal_gb300.workloads import Workload, make_inputs


def bf16_rne(x):
    """fp32 -> bf16 (round to nearest, ties to even), returned as fp32."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32)


def bf16_trunc(x):
    u = np.asarray(x, dtype=np.float32).view(np.uint32)
    return (u >> 16 << 16).view(np.float32)


def n_outside(got, ref):
    got = np.asarray(got, dtype=np.float64)
    return int((np.abs(got - ref) > 2.0 ** -8 * np.abs(ref) + 1e-5).sum())


def layer_outputs():
    x = make_inputs(Workload("bf16cal", 64, 8, 256, 16, 0.3, 11))
    acts = {k: bf16_rne(x[k]).astype(np.float64) for k in ("h_history", "h_s2", "d_h_enriched")}
    y = oracle.forward(acts["h_history"], acts["h_s2"], x["W_A"], x["W_B"], x["W_C"], x["W_O"],
                       x["tw"])
    gr = oracle.backward(acts["h_history"], acts["h_s2"], x["W_A"], x["W_B"], x["W_C"], x["W_O"],
                         x["tw"], acts["d_h_enriched"])
    return {"h_enriched": y, "d_h_history": gr["d_h_history"], "d_h_s2": gr["d_h_s2"]}


def test_bf16_rounding_lies_inside_the_bound():
    for name, ref in layer_outputs().items():
        # the fp32 value (as a stand-in for the fp32 arithmetic), then one rounding
        assert n_outside(bf16_rne(ref.astype(np.float32)), ref) == 0, name


def test_truncating_conversion_is_rejected():
    for name, ref in layer_outputs().items():
        bad = n_outside(bf16_trunc(ref.astype(np.float32)), ref)
        assert bad > ref.size // 20, (name, bad, ref.size)  # 14-27% here


def test_rounding_helper_matches_torch():
    import torch
    v = np.random.default_rng(5).standard_normal(4096).astype(np.float32) * 7
    ties = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -1.0 - 2.0 ** -8], dtype=np.float32)
    v = np.concatenate([v, ties])
    ours = bf16_rne(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    assert np.array_equal(ours, ref)
