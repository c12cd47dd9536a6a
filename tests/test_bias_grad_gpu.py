"""CUDA column sum (m2scan_bias_grad) against the fp64 oracle (needs a GB300).

Tolerance: the kernels add fp32 values; every input reaches its column's
result through at most L additions (its position in a thread's row sum, the
pairwise tree over the row phases of its column, the range partials of one
lane, the lane combine, and the add into db), so
|got - exact| <= L * 2^-24 * (sum |dy| + |db|) to first order. L is computed
from the shapes with the kernels' row split.
"""
import math

import numpy as np
import pytest

import oracle
from gated_ssm_temporal_gb300.workloads import BIAS_WORKLOADS, make_bias_input
from gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def depth(N, C, accumulate):
    """Largest number of fp32 additions between an input and its column's result."""
    if N == 0:
        return 1
    P = min(152, max(1, -(-N // 16)))
    rows = -(-N // P)  # rows of the largest range
    L = C // 4 if C % 4 == 0 else C  # lanes per row: column quads or columns
    worst = 0
    for l0 in range(0, L, 256):
        cb = min(256, L - l0)
        RY = 256 // cb
        worst = max(worst, -(-rows // RY) + math.ceil(math.log2(RY)))
    return worst + -(-P // 8) + 7 + (1 if accumulate else 0)


def run(dy, db=None, accumulate=False, stream=None):
    import torch
    import gated_ssm_temporal_gb300 as g
    ensure_built()
    d = torch.from_numpy(dy).cuda()
    b = None if db is None else torch.from_numpy(np.asarray(db, dtype=np.float32)).cuda()
    out = g.bias_grad(d, b, accumulate=accumulate, stream=stream)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def check(dy, db=None, accumulate=False):
    got = run(dy, db, accumulate)
    ref = oracle.bias_grad(dy, db, accumulate=accumulate)
    N, C = dy.shape
    scale = np.abs(dy.astype(np.float64)).sum(axis=0)
    if accumulate:
        scale = scale + np.abs(np.asarray(db, dtype=np.float64))
    bound = depth(N, C, accumulate) * U * scale * 1.0001 + 1e-30
    err = np.abs(got.astype(np.float64) - ref)
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, "columns %s: err %s > bound %s" % (bad[:5], err[bad[:5]], bound[bad[:5]])
    return got, ref


@pytest.mark.parametrize("name", sorted(BIAS_WORKLOADS))
def test_workloads(name):
    w = BIAS_WORKLOADS[name]
    check(make_bias_input(w.N, w.C, w.seed))


@pytest.mark.parametrize("N,C", [(1, 1), (1, 256), (2, 3), (63, 5), (64, 256), (65, 256),
                                 (1000, 257), (777, 1000), (9731, 42), (65537, 128),
                                 (200000, 3)])
def test_shapes(N, C):
    check(make_bias_input(N, C, seed=N + C))


def test_accumulate_adds_into_db():
    dy = make_bias_input(5000, 130, seed=7)
    db = np.random.default_rng(8).standard_normal(130).astype(np.float32) * 100
    check(dy, db, accumulate=True)


def test_empty_batch():
    import torch
    import gated_ssm_temporal_gb300 as g
    ensure_built()
    db = torch.full((9,), 3.5, device="cuda")
    dy = torch.empty((0, 9), device="cuda")
    g.bias_grad(dy, db, accumulate=True)
    torch.cuda.synchronize()
    assert torch.all(db == 3.5)
    g.bias_grad(dy, db)
    torch.cuda.synchronize()
    assert torch.all(db == 0)


def test_exact_on_small_integers():
    # sums of small integers are exact in fp32 whatever the order
    N, C = 4099, 77
    r = np.arange(N)[:, None]
    c = np.arange(C)[None, :]
    dy = (((7 * r + 3 * c) % 11) - 5).astype(np.float32)
    got = run(dy)
    assert np.array_equal(got.astype(np.float64), oracle.bias_grad(dy))


def test_bitwise_reproducible_and_stream_independent():
    import torch
    dy = make_bias_input(12345, 200, seed=9)
    a = run(dy)
    s = torch.cuda.Stream()
    b = run(dy, stream=s)
    c = run(dy)
    assert np.array_equal(a, b) and np.array_equal(a, c)


def test_guard_bands_and_launch_count():
    import torch
    import gated_ssm_temporal_gb300 as g
    ensure_built()
    N, C, pad, sentinel = 3000, 45, 64, 777.25
    dy = torch.from_numpy(make_bias_input(N, C, seed=10)).cuda()
    buf = torch.full((C + 2 * pad,), sentinel, device="cuda")
    db = buf[pad:pad + C]
    wsn = g.m2scan_bias_grad_workspace_bytes(N, C) // 4
    wsbuf = torch.full((wsn + 2 * pad,), sentinel, device="cuda")
    g.bias_grad(dy, db, workspace=wsbuf[pad:pad + wsn])
    assert g.m2scan_last_launch_count() == 2
    torch.cuda.synchronize()
    for b in (buf, wsbuf):
        assert torch.all(b[:pad] == sentinel) and torch.all(b[-pad:] == sentinel)
    ref = oracle.bias_grad(dy.cpu().numpy())
    assert np.allclose(db.cpu().numpy(), ref, rtol=0, atol=1e-3)
