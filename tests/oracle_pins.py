"""Checks that pin the oracle to facts outside itself.

Every pin takes an oracle library handle (``None`` = the real oracle) and
raises AssertionError when the oracle disagrees with:
  * central finite differences of L = <d_h_enriched, h_enriched> (all six
    gradients),
  * the unrolled closed form of the scan, x_{K-1} = sum_t (prod_{u>t} sig_u) B_t,
    and of the reverse scan, dB_t = d_ctx * C * prod_{u>t} sig_u,
  * the special cases K=1, K=2, saturated gates (A -> -inf gives x = B_{K-1},
    A -> +inf gives x = sum_t B_t), tw = 0,
  * linearity of h_enriched - h_s2 in tw, W_O, W_C and W_B,
  * float64 autograd of the same layer written with torch operators,
  * the hand-derived example in tests/golden/hand_k2.txt,
  * independence from the number of threads,
  * for the optional gate multiplier g (every gate g * sig(A_t), the pages'
    isv_signals[11]): the closed form with g, central differences and torch
    autograd with g, and g = 1 giving the plain layer bit for bit,
  * for the pages' own output step (one scalar context per sample blended
    into every feature with a weight w[j] and 1/D): central differences and
    torch autograd of all gradients including dw, the K=1 closed form, and
    w = 0 giving the identity on h_s2.
  * for the per-element error scales (sums of the absolute values of the
    terms each output adds up, which bound the rounding error of an fp32
    evaluation): the same sums formed from torch float64 autograd's dA, dB,
    dC, ctx, equality with the signed result when every term is
    non-negative or there is a single term, additivity over samples,
    invariance under a sign flip of dY and under a permutation of samples,
    and the triangle inequality.
``tests/test_oracle_mutants.py`` plants mistakes in copies of the oracle and
checks that these pins catch each one.
"""
import numpy as np

import oracle
from golden_io import hand_k2

PARAMS = ["h_history", "h_s2", "W_A", "W_B", "W_C", "W_O"]
GRADS = {"h_history": "d_h_history", "h_s2": "d_h_s2", "W_A": "dW_A", "W_B": "dW_B",
         "W_C": "dW_C", "W_O": "dW_O"}


def rand_inputs(B, K, SH2, D, seed, tw=0.7, wscale=1.0):
    rng = np.random.default_rng(1000 + seed)
    x = {
        "h_history": rng.standard_normal((B, K, SH2)),
        "h_s2": rng.standard_normal((B, SH2)),
        "W_A": rng.standard_normal((SH2, D)) * wscale / np.sqrt(SH2),
        "W_B": rng.standard_normal((SH2, D)) / np.sqrt(SH2),
        "W_C": rng.standard_normal((SH2, D)) / np.sqrt(SH2),
        "W_O": rng.standard_normal((D, SH2)) / np.sqrt(D),
        "d_h_enriched": rng.standard_normal((B, SH2)),
        "tw": tw,
    }
    return x


def fwd(x, lib, **kw):
    return oracle.forward(x["h_history"], x["h_s2"], x["W_A"], x["W_B"], x["W_C"],
                          x["W_O"], x["tw"], lib=lib, **kw)


def bwd(x, lib, **kw):
    return oracle.backward(x["h_history"], x["h_s2"], x["W_A"], x["W_B"], x["W_C"],
                           x["W_O"], x["tw"], x["d_h_enriched"], lib=lib, **kw)


def sigmoid(a):
    return 1.0 / (1.0 + np.exp(-a))


def close(a, b, rtol, atol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    err = np.abs(a - b)
    bound = rtol * np.abs(b) + atol
    bad = err > bound
    assert not bad.any(), "%s: %d mismatches, worst %.3e (bound %.3e)" % (
        what, int(bad.sum()), float(err.max()), float(bound.flat[np.argmax(err - bound)]))


# ---------------------------------------------------------------------------

def pin_finite_differences(lib=None):
    """All six gradients against central differences of <dY, h_enriched>."""
    for (B, K, SH2, D, seed) in [(3, 4, 6, 3, 0), (2, 1, 5, 2, 1), (2, 3, 4, 4, 2)]:
        x = rand_inputs(B, K, SH2, D, seed, wscale=2.0)
        g = bwd(x, lib)
        dy = x["d_h_enriched"]

        def loss(xx):
            return float(np.sum(dy * fwd(xx, lib)))

        eps = 1e-6
        for p in PARAMS:
            num = np.zeros_like(x[p])
            flat = num.reshape(-1)
            for i in range(flat.size):
                xp = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in x.items()}
                xm = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in x.items()}
                xp[p].reshape(-1)[i] += eps
                xm[p].reshape(-1)[i] -= eps
                flat[i] = (loss(xp) - loss(xm)) / (2 * eps)
            close(g[GRADS[p]], num, 1e-6, 1e-8, "finite differences d%s (K=%d)" % (p, K))


def pin_closed_form_scan(lib=None):
    """x_{K-1} = sum_t (prod_{u>t} sig(A_u)) B_t, ctx = C x_{K-1}, output step."""
    x = rand_inputs(5, 6, 8, 3, 3, wscale=3.0)
    h, hs = x["h_history"], x["h_s2"]
    A = h @ x["W_A"]
    Bv = h @ x["W_B"]
    C = hs @ x["W_C"]
    sig = sigmoid(A)
    K = h.shape[1]
    xk = np.zeros_like(C)
    for t in range(K):
        xk += np.prod(sig[:, t + 1:, :], axis=1) * Bv[:, t, :]
    oA, oB, ox, oC, octx = oracle.scan_state(h, hs, x["W_A"], x["W_B"], x["W_C"], lib=lib)
    close(oA, A, 1e-12, 1e-13, "A projection")
    close(oB, Bv, 1e-12, 1e-13, "B projection")
    close(oC, C, 1e-12, 1e-13, "C projection")
    close(ox[:, K - 1, :], xk, 1e-12, 1e-13, "closed-form x_{K-1}")
    close(octx, C * xk, 1e-12, 1e-13, "ctx = C x_{K-1}")
    y = hs + x["tw"] * ((C * xk) @ x["W_O"])
    close(fwd(x, lib), y, 1e-12, 1e-13, "output step")
    # every intermediate state, not only the last
    for t in range(K):
        xt = np.zeros_like(C)
        for u in range(t + 1):
            xt += np.prod(sig[:, u + 1:t + 1, :], axis=1) * Bv[:, u, :]
        close(ox[:, t, :], xt, 1e-12, 1e-13, "closed-form x_%d" % t)


def pin_reverse_closed_form(lib=None):
    """dB_t = d_ctx*C*prod_{u>t} sig_u; dA_0 = 0 so d_h_history[:,0] = dB_0 W_B^T."""
    x = rand_inputs(4, 5, 7, 3, 4, wscale=2.0)
    h, hs, W_B, W_O = x["h_history"], x["h_s2"], x["W_B"], x["W_O"]
    A = h @ x["W_A"]
    C = hs @ x["W_C"]
    sig = sigmoid(A)
    dctx = x["tw"] * (x["d_h_enriched"] @ W_O.T)
    dB0 = dctx * C * np.prod(sig[:, 1:, :], axis=1)
    g = bwd(x, lib)
    close(g["d_h_history"][:, 0, :], dB0 @ W_B.T, 1e-11, 1e-13, "d_h_history at t=0")


def pin_k1(lib=None):
    """K=1: x = B_0, so h_enriched ignores W_A and dW_A is exactly zero."""
    x = rand_inputs(3, 1, 6, 3, 5)
    y1 = fwd(x, lib)
    x2 = dict(x)
    x2["W_A"] = x["W_A"] * -7.0 + 1.0
    y2 = fwd(x2, lib)
    assert np.array_equal(y1, y2), "K=1 output depends on W_A"
    Bv = x["h_history"][:, 0, :] @ x["W_B"]
    C = x["h_s2"] @ x["W_C"]
    close(y1, x["h_s2"] + x["tw"] * ((C * Bv) @ x["W_O"]), 1e-12, 1e-13, "K=1 closed form")
    g = bwd(x, lib)
    assert np.all(g["dW_A"] == 0.0), "K=1 dW_A not zero"


def pin_k2(lib=None):
    """K=2: x = sig(A_1) B_0 + B_1."""
    x = rand_inputs(3, 2, 5, 2, 6, wscale=2.0)
    A = x["h_history"] @ x["W_A"]
    Bv = x["h_history"] @ x["W_B"]
    xk = sigmoid(A[:, 1]) * Bv[:, 0] + Bv[:, 1]
    _, _, ox, _, _ = oracle.scan_state(x["h_history"], x["h_s2"], x["W_A"], x["W_B"],
                                       x["W_C"], lib=lib)
    close(ox[:, 1], xk, 1e-12, 1e-13, "K=2 closed form")


def pin_saturated_gates(lib=None):
    """A -> -inf gives x_{K-1} = B_{K-1}; A -> +inf gives x_{K-1} = sum_t B_t."""
    for sign, expect in ((-1.0, "last"), (1.0, "sum")):
        x = rand_inputs(3, 6, 5, 3, 7)
        x["h_history"][:, :, 0] = 1.0          # constant feature
        x["W_A"][:] = 0.0
        x["W_A"][0, :] = 50.0 * sign           # A = +-50 everywhere
        Bv = x["h_history"] @ x["W_B"]
        xk = Bv[:, -1] if expect == "last" else Bv.sum(axis=1)
        _, _, ox, _, _ = oracle.scan_state(x["h_history"], x["h_s2"], x["W_A"], x["W_B"],
                                           x["W_C"], lib=lib)
        close(ox[:, -1], xk, 1e-12, 1e-13, "saturated gate (%s)" % expect)
        g = bwd(x, lib)
        assert np.abs(g["dW_A"]).max() < 1e-15, "saturated gate: dW_A not ~0"


def pin_tw_zero(lib=None):
    """tw = 0: the layer is the identity on h_s2 and every other gradient vanishes."""
    x = rand_inputs(3, 4, 6, 3, 8, tw=0.0)
    assert np.array_equal(fwd(x, lib), x["h_s2"]), "tw=0 output != h_s2"
    g = bwd(x, lib)
    assert np.array_equal(g["d_h_s2"], x["d_h_enriched"]), "tw=0 d_h_s2 != dY"
    for k in ("d_h_history", "dW_A", "dW_B", "dW_C", "dW_O"):
        assert np.all(g[k] == 0.0), "tw=0 %s not zero" % k


def pin_linearity(lib=None):
    """h_enriched - h_s2 is linear in tw, in W_O, in W_C and in W_B."""
    x = rand_inputs(3, 5, 6, 3, 9, wscale=2.0)
    base = fwd(x, lib) - x["h_s2"]
    for alpha in (-1.5, 3.0):
        for key in ("tw", "W_O", "W_C", "W_B"):
            xs = dict(x)
            xs[key] = x[key] * alpha
            close(fwd(xs, lib) - x["h_s2"], alpha * base, 1e-11, 1e-13,
                  "linearity in %s" % key)


def pin_torch_autograd(lib=None):
    """Output and all gradients against torch float64 autograd."""
    import torch
    for (B, K, SH2, D, seed) in [(4, 7, 9, 3, 10), (2, 3, 16, 5, 11)]:
        x = rand_inputs(B, K, SH2, D, seed, wscale=3.0)
        t = {k: torch.tensor(x[k], dtype=torch.float64, requires_grad=True) for k in PARAMS}
        A = t["h_history"] @ t["W_A"]
        Bv = t["h_history"] @ t["W_B"]
        C = t["h_s2"] @ t["W_C"]
        state = torch.zeros(B, D, dtype=torch.float64)
        for k in range(K):
            state = torch.sigmoid(A[:, k]) * state + Bv[:, k]
        y = t["h_s2"] + x["tw"] * ((C * state) @ t["W_O"])
        (y * torch.tensor(x["d_h_enriched"])).sum().backward()
        close(fwd(x, lib), y.detach().numpy(), 1e-12, 1e-13, "autograd output")
        g = bwd(x, lib)
        for p in PARAMS:
            close(g[GRADS[p]], t[p].grad.numpy(), 1e-10, 1e-12, "autograd d%s" % p)


def pin_golden_hand_example(lib=None):
    """The hand-derived example in tests/golden/hand_k2.txt (exact values)."""
    x = hand_k2()
    close(fwd(x, lib), x["h_enriched"], 0.0, 1e-15, "golden h_enriched")
    g = bwd(x, lib)
    for k in ("d_h_history", "d_h_s2", "dW_A", "dW_B", "dW_C", "dW_O"):
        close(g[k], x[k], 0.0, 1e-15, "golden %s" % k)


def pin_thread_count_invariance(lib=None):
    """Outputs do not depend on the number of threads (fixed block order)."""
    x = rand_inputs(37, 3, 8, 2, 12)
    g1 = bwd(x, lib, n_threads=1)
    g3 = bwd(x, lib, n_threads=3)
    for k in g1:
        assert np.array_equal(g1[k], g3[k]), "thread count changed %s" % k
    assert np.array_equal(fwd(x, lib, n_threads=1), fwd(x, lib, n_threads=4))


def pin_gate_scale_closed_form(lib=None):
    """x_{K-1} = sum_t (prod_{u>t} g sig(A_u)) B_t with a gate multiplier g."""
    gs = 0.6
    x = rand_inputs(4, 5, 7, 3, 13, wscale=2.0)
    h, hs = x["h_history"], x["h_s2"]
    sig = sigmoid(h @ x["W_A"])
    Bv = h @ x["W_B"]
    K = h.shape[1]
    xk = np.zeros((h.shape[0], x["W_A"].shape[1]))
    for t in range(K):
        xk += np.prod(gs * sig[:, t + 1:, :], axis=1) * Bv[:, t, :]
    _, _, ox, oC, _ = oracle.scan_state(h, hs, x["W_A"], x["W_B"], x["W_C"], lib=lib,
                                        gate_scale=gs)
    close(ox[:, K - 1, :], xk, 1e-12, 1e-13, "closed-form x_{K-1} with a gate multiplier")
    y = hs + x["tw"] * ((oC * xk) @ x["W_O"])
    close(fwd(x, lib, gate_scale=gs), y, 1e-12, 1e-13, "output with a gate multiplier")
    # g = 1 is the plain layer, bit for bit
    assert np.array_equal(fwd(x, lib, gate_scale=1.0), fwd(x, lib))
    g1, g0 = bwd(x, lib, gate_scale=1.0), bwd(x, lib)
    for k in g0:
        assert np.array_equal(g1[k], g0[k]), "gate multiplier 1 changed %s" % k


def pin_gate_scale_gradients(lib=None):
    """All six gradients with a gate multiplier: central differences and torch autograd."""
    import torch
    gs = 0.7
    x = rand_inputs(2, 3, 4, 3, 14, wscale=2.0)
    g = bwd(x, lib, gate_scale=gs)
    dy = x["d_h_enriched"]

    def loss(xx):
        return float(np.sum(dy * fwd(xx, lib, gate_scale=gs)))

    eps = 1e-6
    for p in PARAMS:
        num = np.zeros_like(x[p])
        flat = num.reshape(-1)
        for i in range(flat.size):
            xp = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in x.items()}
            xm = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in x.items()}
            xp[p].reshape(-1)[i] += eps
            xm[p].reshape(-1)[i] -= eps
            flat[i] = (loss(xp) - loss(xm)) / (2 * eps)
        close(g[GRADS[p]], num, 1e-6, 1e-8, "finite differences d%s with a gate multiplier" % p)
    x = rand_inputs(3, 6, 9, 4, 15, wscale=3.0)
    t = {k: torch.tensor(x[k], dtype=torch.float64, requires_grad=True) for k in PARAMS}
    A = t["h_history"] @ t["W_A"]
    Bv = t["h_history"] @ t["W_B"]
    C = t["h_s2"] @ t["W_C"]
    state = torch.zeros(3, 4, dtype=torch.float64)
    for k in range(6):
        state = gs * torch.sigmoid(A[:, k]) * state + Bv[:, k]
    y = t["h_s2"] + x["tw"] * ((C * state) @ t["W_O"])
    (y * torch.tensor(x["d_h_enriched"])).sum().backward()
    close(fwd(x, lib, gate_scale=gs), y.detach().numpy(), 1e-12, 1e-13,
          "autograd output with a gate multiplier")
    g = bwd(x, lib, gate_scale=gs)
    for p in PARAMS:
        close(g[GRADS[p]], t[p].grad.numpy(), 1e-10, 1e-12,
              "autograd d%s with a gate multiplier" % p)


def pin_blend(lib=None):
    """The pages' output step h + w[j] * (sum_s ctx_s) / D: closed form, w = 0,
    central differences and torch autograd of every gradient (dw included)."""
    import torch
    x = rand_inputs(3, 1, 6, 4, 16)
    w = np.random.default_rng(17).standard_normal(6)
    Bv = x["h_history"][:, 0, :] @ x["W_B"]
    C = x["h_s2"] @ x["W_C"]
    want = x["h_s2"] + np.outer((C * Bv).sum(axis=1) / 4.0, w)
    close(fwd(dict(x, W_O=w), lib, blend=True), want, 1e-12, 1e-13, "blend K=1 closed form")
    x0 = dict(x, W_O=np.zeros(6))
    assert np.array_equal(fwd(x0, lib, blend=True), x["h_s2"]), "blend w=0 != h_s2"
    g0 = bwd(x0, lib, blend=True)
    assert np.array_equal(g0["d_h_s2"], x["d_h_enriched"])
    assert np.all(g0["dW_A"] == 0.0) and np.all(g0["d_h_history"] == 0.0)
    ones = fwd(dict(x, W_O=None), lib, blend=True)
    assert np.array_equal(ones, fwd(dict(x, W_O=np.ones(6)), lib, blend=True))
    # every gradient by central differences (dw is the gradient of W_O = w)
    x = rand_inputs(2, 3, 5, 3, 18, wscale=2.0)
    x["W_O"] = np.random.default_rng(19).standard_normal(5)
    gr = bwd(x, lib, blend=True)
    dy = x["d_h_enriched"]

    def loss(xx):
        return float(np.sum(dy * fwd(xx, lib, blend=True)))

    eps = 1e-6
    for p in PARAMS:
        num = np.zeros_like(x[p])
        flat = num.reshape(-1)
        for i in range(flat.size):
            xp = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in x.items()}
            xm = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in x.items()}
            xp[p].reshape(-1)[i] += eps
            xm[p].reshape(-1)[i] -= eps
            flat[i] = (loss(xp) - loss(xm)) / (2 * eps)
        close(gr[GRADS[p]], num, 1e-6, 1e-8, "blend finite differences d%s" % p)
    # torch float64 autograd, with a gate multiplier as well
    gs = 0.9
    x = rand_inputs(3, 5, 7, 4, 20, wscale=3.0)
    x["W_O"] = np.random.default_rng(21).standard_normal(7)
    t = {k: torch.tensor(x[k], dtype=torch.float64, requires_grad=True) for k in PARAMS}
    A = t["h_history"] @ t["W_A"]
    Bv = t["h_history"] @ t["W_B"]
    C = t["h_s2"] @ t["W_C"]
    state = torch.zeros(3, 4, dtype=torch.float64)
    for k in range(5):
        state = gs * torch.sigmoid(A[:, k]) * state + Bv[:, k]
    context = (C * state).sum(dim=1, keepdim=True)
    y = t["h_s2"] + t["W_O"][None, :] * context / 4.0
    (y * torch.tensor(x["d_h_enriched"])).sum().backward()
    close(fwd(x, lib, blend=True, gate_scale=gs), y.detach().numpy(), 1e-12, 1e-13,
          "blend autograd output")
    gr = bwd(x, lib, blend=True, gate_scale=gs)
    for p in PARAMS:
        close(gr[GRADS[p]], t[p].grad.numpy(), 1e-10, 1e-12, "blend autograd d%s" % p)


ABS_KEYS = ("dW_A", "dW_B", "dW_C", "dW_O", "d_h_history", "d_h_s2")


def bwd_abs(x, lib, **kw):
    return bwd(x, lib, abs_terms=True, **kw)


def pin_abs_terms_autograd(lib=None):
    """Absolute-term sums against the same sums built from torch float64
    autograd's intermediate gradients (dA, dB = dL/dB_t, dC = dL/dC) and
    forward values (ctx)."""
    import torch
    for (B, K, SH2, D, seed) in [(4, 5, 7, 3, 20), (3, 1, 6, 2, 21)]:
        x = rand_inputs(B, K, SH2, D, seed, wscale=3.0)
        t = {k: torch.tensor(x[k], dtype=torch.float64, requires_grad=True) for k in PARAMS}
        A = t["h_history"] @ t["W_A"]
        Bv = t["h_history"] @ t["W_B"]
        C = t["h_s2"] @ t["W_C"]
        for v in (A, Bv, C):
            v.retain_grad()
        state = torch.zeros(B, D, dtype=torch.float64)
        for k in range(K):
            state = torch.sigmoid(A[:, k]) * state + Bv[:, k]
        ctx = C * state
        y = t["h_s2"] + x["tw"] * (ctx @ t["W_O"])
        (y * torch.tensor(x["d_h_enriched"])).sum().backward()
        h, hs, g = x["h_history"], x["h_s2"], x["d_h_enriched"]
        dA, dB, dC = A.grad.numpy(), Bv.grad.numpy(), C.grad.numpy()
        cx = ctx.detach().numpy()
        exp = {
            "dW_A": np.abs(h[:, :, :, None] * dA[:, :, None, :]).sum(axis=(0, 1)),
            "dW_B": np.abs(h[:, :, :, None] * dB[:, :, None, :]).sum(axis=(0, 1)),
            "dW_C": np.abs(hs[:, :, None] * dC[:, None, :]).sum(axis=0),
            "dW_O": np.abs(x["tw"] * cx[:, :, None] * g[:, None, :]).sum(axis=0),
            "d_h_history": (np.abs(dA[:, :, None, :] * x["W_A"][None, None]).sum(axis=3)
                            + np.abs(dB[:, :, None, :] * x["W_B"][None, None]).sum(axis=3)),
            "d_h_s2": np.abs(g) + np.abs(dC[:, None, :] * x["W_C"][None]).sum(axis=2),
        }
        r = bwd_abs(x, lib)
        for k in ABS_KEYS:
            close(r[k + "_abs"], exp[k], 1e-10, 1e-13, "autograd |terms| of %s" % k)
        out, aout = fwd(x, lib, abs_terms=True)
        close(aout, np.abs(hs) + abs(x["tw"]) * np.abs(cx[:, :, None] * x["W_O"][None]).sum(axis=1),
              1e-10, 1e-13, "autograd |terms| of h_enriched")


def pin_abs_terms_invariants(lib=None):
    """Equalities and invariances every absolute-term sum must satisfy."""
    # every term non-negative: inputs >= 0 and tw > 0 make every projection,
    # state, gradient and product non-negative, so |sum| = sum of |terms|
    x = rand_inputs(5, 4, 6, 3, 30)
    for k in PARAMS + ["d_h_enriched"]:
        x[k] = np.abs(x[k])
    r = bwd_abs(x, lib)
    for k in ABS_KEYS:
        close(r[k + "_abs"], np.abs(r[k]), 1e-12, 0.0, "non-negative terms %s" % k)
    out, aout = fwd(x, lib, abs_terms=True)
    close(aout, np.abs(out), 1e-12, 0.0, "non-negative terms h_enriched")
    # one sample, one step, one state, no residual: every sum has one term
    x = rand_inputs(1, 1, 5, 1, 31)
    r = bwd_abs(x, lib)
    for k in ("dW_A", "dW_B", "dW_C", "dW_O", "d_h_history"):
        close(r[k + "_abs"], np.abs(r[k]), 1e-14, 0.0, "single term %s" % k)
    xz = dict(x)
    xz["h_s2"] = np.zeros_like(x["h_s2"])
    out, aout = fwd(xz, lib, abs_terms=True)
    close(aout, np.abs(out), 1e-14, 0.0, "single term h_enriched")
    # mixed signs: triangle inequality, additivity over samples, sign flip of
    # dY, permutation of samples
    x = rand_inputs(6, 5, 7, 3, 32, wscale=2.0)
    r = bwd_abs(x, lib)
    for k in ABS_KEYS:
        assert np.all(np.abs(r[k]) <= r[k + "_abs"] * (1 + 1e-12) + 1e-300), "triangle %s" % k
    part = []
    for sl in (slice(0, 2), slice(2, 6)):
        xs = {k: (v[sl] if k in ("h_history", "h_s2", "d_h_enriched") else v) for k, v in x.items()}
        part.append(bwd_abs(xs, lib))
    for k in ("dW_A", "dW_B", "dW_C", "dW_O"):
        close(r[k + "_abs"], part[0][k + "_abs"] + part[1][k + "_abs"], 1e-12, 0.0,
              "additivity over samples %s" % k)
    for k in ("d_h_history", "d_h_s2"):
        close(r[k + "_abs"], np.concatenate([part[0][k + "_abs"], part[1][k + "_abs"]]), 0.0, 0.0,
              "per-sample %s" % k)
    xf = dict(x)
    xf["d_h_enriched"] = -x["d_h_enriched"]
    rf = bwd_abs(xf, lib)
    for k in ABS_KEYS:
        close(rf[k + "_abs"], r[k + "_abs"], 1e-14, 0.0, "sign flip of dY %s" % k)
    perm = np.array([3, 0, 5, 1, 4, 2])
    xp = {k: (v[perm] if k in ("h_history", "h_s2", "d_h_enriched") else v) for k, v in x.items()}
    rp = bwd_abs(xp, lib)
    for k in ("dW_A", "dW_B", "dW_C", "dW_O"):
        close(rp[k + "_abs"], r[k + "_abs"], 1e-12, 0.0, "sample permutation %s" % k)


ALL_PINS = [pin_finite_differences, pin_closed_form_scan, pin_reverse_closed_form, pin_k1,
            pin_k2, pin_saturated_gates, pin_tw_zero, pin_linearity, pin_torch_autograd,
            pin_golden_hand_example, pin_thread_count_invariance, pin_gate_scale_closed_form,
            pin_gate_scale_gradients, pin_blend, pin_abs_terms_autograd,
            pin_abs_terms_invariants]
