"""How many weight-gradient entries a plain fp32 evaluation misses under the
strict elementwise criterion (|err| > max(1e-4 |exact|, 1e-5)), per workload.

The layer is evaluated with numpy float32 operations (BLAS matrix products,
elementwise scan) on the same seeded inputs, and compared with the fp64
oracle. The counts show which strict misses of the GPU path are a property of
fp32 summation itself. Also printed: the largest error in units of
2^-24 * sum|terms| (the scale of the parity bound in tests/tolerance.py).

    python tests/fp32_numpy_reference.py [workload ...]
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from gated_ssm_temporal_gb300.workloads import WORKLOADS, make_inputs  # noqa: E402

F = np.float32
U = 2.0 ** -24


def numpy_fp32_weight_gradients(x):
    h, hs, WA, WB, WC, WO, g = (np.asarray(x[k], F) for k in
                                ("h_history", "h_s2", "W_A", "W_B", "W_C", "W_O", "d_h_enriched"))
    tw = F(x["tw"])
    B, K, SH2 = h.shape
    D = WA.shape[1]
    A, Bv, C = h @ WA, h @ WB, hs @ WC
    sig = (F(1) / (F(1) + np.exp(-A))).astype(F)
    xs = np.zeros((B, K, D), F)
    xc = np.zeros((B, D), F)
    for t in range(K):
        xc = sig[:, t] * xc + Bv[:, t]
        xs[:, t] = xc
    ctx = C * xc
    dctx = tw * (g @ WO.T)
    dC = dctx * xc
    dx = dctx * C
    dA = np.zeros((B, K, D), F)
    dB = np.zeros((B, K, D), F)
    for t in range(K - 1, -1, -1):
        xp = xs[:, t - 1] if t > 0 else np.zeros((B, D), F)
        dB[:, t] = dx
        dA[:, t] = dx * xp * sig[:, t] * (F(1) - sig[:, t])
        dx = dx * sig[:, t]
    hf = h.reshape(-1, SH2)
    return {"dW_A": hf.T @ dA.reshape(-1, D), "dW_B": hf.T @ dB.reshape(-1, D),
            "dW_C": hs.T @ dC, "dW_O": tw * (ctx.T @ g)}


def counts(name):
    x = make_inputs(WORKLOADS[name])
    ref = oracle.backward(x["h_history"], x["h_s2"], x["W_A"], x["W_B"], x["W_C"], x["W_O"],
                          x["tw"], x["d_h_enriched"], abs_terms=True)
    got = numpy_fp32_weight_gradients(x)
    out = {}
    for k, v in got.items():
        err = np.abs(v.astype(np.float64) - ref[k])
        strict = np.maximum(1e-4 * np.abs(ref[k]), 1e-5)
        out[k] = (int((err > strict).sum()), float((err / (U * ref[k + "_abs"])).max()))
    return out


if __name__ == "__main__":
    for name in sys.argv[1:] or ["pages", "long_history", "wide_state", "stress"]:
        for k, (n, r) in counts(name).items():
            print("%-13s %s  strict misses %4d   max err / (2^-24 sum|terms|) %.2f" % (name, k, n, r))
