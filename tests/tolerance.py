"""Parity criteria between the CUDA path (fp32) and the fp64 oracle.

The layer's tolerance is a relative error of 1e-4 with an absolute floor of
1e-5. For h_enriched, d_h_history and d_h_s2 this is applied element by
element: |gpu - ref| <= max(1e-4 * |ref|, 1e-5).

The four weight gradients (and the blend's dw) are sums over B or B*K sample
terms whose signs cancel; some entries land arbitrarily close to 0 while each
term is O(1), and no fp32 evaluation reaches a 1e-4 relative error on those
entries (a numpy float32 evaluation misses 1-15 of 4096 entries per tensor on
the 8192-sample and long-history workloads). What bounds the error of a
floating-point sum is not the sum but the sum of the absolute values of its
terms: the oracle returns T = sum |term| per element, and an element passes
when

    |gpu - ref| <= max(1e-4 * |ref|,  c * 2^-24 * T,  1e-5).

c is derived, not fitted: c = L + E where
  L  the longest chain of fp32 roundings between a term and the result in
     any of the kernels: at most one rounding per term added to a slot's
     running sum (a tensor-core step adds 8 terms with a few roundings, a
     fused multiply-add one), R terms per slot with R = ceil(B / P) samples
     (times K rows for dW_A, dW_B), then the slot sum (P slots added as eight
     interleaved chains of ceil(P / 8) and the eight in order) and the final
     adds;
  E  the term's own error relative to the term: 64 units for the product
     itself (3 x TF32 represents each operand product to 2^-19 = 32 units)
     and the fp32 roundings that form its factors, 4 per step of the K-step
     scan that dA, dB, dC and ctx come out of, and 8 sqrt(SH2) for the error
     those factors inherit from the projections (sums of SH2 products, each
     represented to about 8 units, whose errors are independent):
     E = 64 + 4 K + 8 sqrt(SH2).
The oracle's T is pinned on the CPU (tests/oracle_pins.py). A single dropped
sample moves some element of each weight gradient by more than 9000 units of
2^-24 T on the 8192-sample workload, so the gate still catches it.

Every tensor whose entries exceed 100x the floor must also meet a normwise
relative error <= 1e-5 (<= 1e-4 for the ill-conditioned inputs below).

Stress inputs outside the layer's workloads (history activations x30 on odd
samples) make every output ill-conditioned: outputs are small differences of
large terms, and a numpy float32 evaluation misses the elementwise bound on
18-45 entries of h_enriched, d_h_history and d_h_s2. Those tests apply the
same T-based bound to every output (``ill_conditioned=True``), with the
chain of each per-sample output's own sum in L.

``compare`` also reports the strict elementwise count (|err| > max(1e-4 |ref|,
1e-5)) and the largest err / (2^-24 T); when the environment variable
M2SCAN_PARITY_RECORD names a file, every comparison is appended to it as one
JSON line.
"""
import json
import math
import os

import numpy as np

RTOL = 1e-4
ATOL = 1e-5
NORMWISE = 1e-5
U = 2.0 ** -24
MAX_SLOTS = 152      # weight-gradient slots of the fused kernels (one per SM of a GB300)
WIDE_SLOTS = 152     # sample ranges of the wide-state dW products
REDUCTIONS = ("dW_A", "dW_B", "dW_C", "dW_O", "dw")


def term_budget(K, SH2):
    """E: the error of one term relative to the term, in units of 2^-24."""
    return 64 + 4 * K + 8 * math.ceil(math.sqrt(SH2))


def chain_length(name, B, K, SH2, D, wide=False):
    """L: the longest chain of fp32 roundings from a term of output ``name`` to
    its result, for any kernel family (``wide``: the wide-state family's
    sample ranges in place of the slots; both number 152)."""
    if name in ("h_enriched", "d_h_s2"):
        return D + 2
    if name == "d_h_history":
        return 2 * D + 4
    if B <= 0:
        return 1
    P = min(B, WIDE_SLOTS if wide else MAX_SLOTS)
    R = -(-B // P) * (K if name in ("dW_A", "dW_B") else 1)
    L = R + 1 + (-(-P // 8)) + 8 + 1
    if name == "dw":  # the blend's fold of dW_O over the D states
        L += D + 1
    return L


def coefficient(name, B, K, SH2, D, wide=False):
    return chain_length(name, B, K, SH2, D, wide) + term_budget(K, SH2)


def compare(name, got, ref, terms=None, c=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite values" % name
    err = np.abs(got - ref)
    strict = np.maximum(RTOL * np.abs(ref), ATOL)
    out = {"name": name, "n": int(err.size)}
    if terms is not None:
        terms = np.asarray(terms, dtype=np.float64)
        assert terms.shape == ref.shape, (name, terms.shape)
        bound = np.maximum(strict, c * U * terms)
        with np.errstate(divide="ignore", invalid="ignore"):
            ratio = np.where(terms > 0, err / (U * terms), 0.0)
        out.update(c=float(c), max_err_over_u_terms=float(ratio.max()) if err.size else 0.0)
    else:
        bound = strict
    nref = float(np.linalg.norm(ref))
    normwise = float(np.linalg.norm(got - ref)) / nref if nref > 0 else float(np.linalg.norm(got))
    out.update({
        "max_err_over_bound": float(np.max(err / bound)) if err.size else 0.0,
        "n_fail": int(np.sum(err > bound)),
        "n_fail_strict_elementwise": int(np.sum(err > strict)),
        "normwise": normwise,
        "max_abs_err": float(err.max()) if err.size else 0.0,
    })
    return out


def _record(r, context):
    path = os.environ.get("M2SCAN_PARITY_RECORD")
    if path:
        rec = dict(r)
        rec.update(context or {})
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")


def _above_floor(ref):
    """The normwise limit applies to tensors with entries well above the absolute floor;
    a tensor that is ~0 everywhere (e.g. dW_A with every gate closed) is governed by
    the elementwise floor alone."""
    ref = np.asarray(ref, dtype=np.float64)
    return ref.size > 0 and float(np.abs(ref).max()) > 100 * ATOL


def assert_parity(name, got, ref, terms=None, c=None, normwise_limit=NORMWISE, context=None):
    """Weight gradients need ``terms`` (the oracle's sum of |terms|) and ``c``;
    other outputs are compared strictly unless ``terms`` is given."""
    if name in REDUCTIONS:
        assert terms is not None and c is not None, "%s: a reduction needs its |terms| and c" % name
    r = compare(name, got, ref, terms, c)
    _record(r, context)
    assert r["n_fail"] == 0, "%s: %d elements outside tolerance (worst ratio %.3f)" % (
        name, r["n_fail"], r["max_err_over_bound"])
    if _above_floor(ref):
        assert r["normwise"] <= normwise_limit, "%s: normwise error %.3e" % (name, r["normwise"])
    return r


def assert_outputs(got, ref, shape, names, ill_conditioned=False, wide=False, context=None,
                   key_map=None):
    """Every output in ``names`` against the oracle dict ``ref`` (which holds
    the ``<name>_abs`` sums); ``shape`` = (B, K, SH2, D). ``key_map`` maps a
    name of ``got`` to the oracle's name (e.g. the blend's dw is the oracle's
    dW_O)."""
    B, K, SH2, D = shape
    res = {}
    for n in names:
        rn = (key_map or {}).get(n, n)
        ctx = dict(context or {}, B=B, K=K, SH2=SH2, D=D)
        if rn in ("dW_A", "dW_B", "dW_C", "dW_O") or ill_conditioned:
            cn = "dw" if n == "dw" else rn
            c = coefficient(cn, B, K, SH2, D, wide)
            res[n] = assert_parity(n, got[n], ref[rn], terms=ref[rn + "_abs"], c=c,
                                   normwise_limit=1e-4 if ill_conditioned else NORMWISE,
                                   context=ctx)
        else:
            res[n] = assert_parity(n, got[n], ref[rn], context=ctx)
    return res
