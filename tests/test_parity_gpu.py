"""CUDA path against the fp64 oracle, element by element (needs a GB300)."""
import numpy as np
import pytest

from gated_ssm_temporal_gb300.workloads import WORKLOADS, Workload, make_inputs
from golden_io import hand_k2
from gpu_helpers import (OUTPUTS, ensure_built, oracle_all, run_all, run_bwd, run_fwd, runs_wide,
                         shape_of, to_dev)
from tolerance import assert_outputs

pytestmark = pytest.mark.gpu

NAMES = ("h_enriched",) + OUTPUTS


def check(x, force_generic=False, ill_conditioned=False, label=None):
    got = run_all(x, force_generic=force_generic)
    ref = oracle_all(x)
    return assert_outputs(got, ref, shape_of(x), NAMES, ill_conditioned=ill_conditioned,
                          wide=runs_wide(x, force_generic),
                          context={"test": label or "", "generic": force_generic})


def custom(B, K, SH2, D, seed, tw=0.3, wa_scale=1.0, odd=1.0):
    return make_inputs(Workload("custom", B, K, SH2, D, tw, seed, wa_scale, odd))


@pytest.mark.parametrize("seed", range(5))
def test_tiny_workload(seed):
    check(make_inputs(WORKLOADS["tiny"].with_batch(4, seed)), label="tiny seed %d" % seed)


@pytest.mark.parametrize("name", ["pages", "long_history", "wide_state", "stress"])
def test_full_size_workloads(name):
    """Every output of the full workload, in the launch configuration the benchmark times."""
    check(make_inputs(WORKLOADS[name]), label=name)


@pytest.mark.parametrize("B", [1, 2, 5, 17, 151, 152, 153, 1000, 8191])
def test_ragged_batches(B):
    check(custom(B, 8, 256, 16, seed=100 + B, tw=0.1))


@pytest.mark.parametrize("K,SH2,D", [
    (1, 256, 16), (2, 64, 16), (3, 96, 8), (5, 160, 16), (7, 32, 4), (16, 128, 8),
    (33, 64, 16), (100, 256, 16), (128, 64, 4), (8, 256, 8), (8, 512, 8)])
def test_fast_path_shapes(K, SH2, D):
    check(custom(37, K, SH2, D, seed=K * 1000 + SH2 + D, wa_scale=2.0))


@pytest.mark.parametrize("B,K,SH2", [
    (3503, 1, 256), (2999, 3, 96), (4000, 5, 160), (2000, 12, 32), (1217, 33, 256), (900, 128, 64)])
def test_tensor_core_multi_tile_shapes(B, K, SH2):
    # D = 16 runs the tensor-core kernels; B > 152 gives every CTA several
    # tiles of unequal size (S_t from 16 down to 1 sample, 1 or 2 sample
    # items, 1 to 8 row items) and SH2 / 32 chunks per tile
    check(custom(B, K, SH2, 16, seed=B + K + SH2, wa_scale=2.0))


# samples per tile 16, 8, 6, 4 and 1 cover the three dot layouts of the
# wide-state tile kernels (8, 4 and 2 chunk columns per thread); SH2 from 128
# to 1024 (4 to 32 chunks and 1 to 8 column blocks per tile)
@pytest.mark.parametrize("B,K,SH2", [
    (1, 1, 128), (5, 16, 512), (37, 3, 128), (1000, 7, 384), (300, 128, 256), (2047, 16, 512),
    (700, 20, 128), (333, 32, 256), (300, 4, 1024), (155, 2, 640)])
def test_wide_state_shapes(B, K, SH2):
    # D = 64 runs the wide-state tensor-core kernels: 128-row tiles of up to
    # 16 samples, a partial last tile, and up to 152 sample ranges for the dW
    # products (fewer when B < 152)
    import gated_ssm_temporal_gb300 as g
    ensure_built()
    assert g.m2scan_path_for(K, SH2, 64) == 3
    check(custom(B, K, SH2, 64, seed=B * 7 + K + SH2, wa_scale=2.0))


@pytest.mark.parametrize("K,SH2,D", [
    (8, 36, 16), (129, 64, 4), (4, 4, 1), (6, 20, 3), (8, 256, 16), (16, 512, 64), (3, 64, 24)])
def test_generic_path_shapes(K, SH2, D):
    force = (K, SH2, D) == (8, 256, 16)
    check(custom(23, K, SH2, D, seed=7 + K + SH2 + D, wa_scale=2.0), force_generic=force)


def test_generic_path_matches_on_pages_dims():
    check(custom(600, 8, 256, 16, seed=5, tw=0.1), force_generic=True)


@pytest.mark.parametrize("sign", [-1.0, 1.0])
def test_saturated_gates(sign):
    """A constant feature with W_A row 0 = +-50 drives every gate to sigmoid(+-50): fully
    open (x_{K-1} = sum_t B_t) or closed (x_{K-1} = B_{K-1}); no NaN may appear."""
    for force in (False, True):
        x = custom(64, 8, 256, 16, seed=11)
        x["h_history"][:, :, 0] = 1.0
        x["W_A"][0, :] = 50.0 * sign
        check(x, force_generic=force)


def test_heavy_tailed_history():
    """Every odd sample's history x30. Ill-conditioned outputs: every output on the
    bound from its sum of |terms|."""
    for force in (False, True):
        check(custom(300, 8, 256, 16, seed=12, odd=30.0), force_generic=force,
              ill_conditioned=True, label="history x30")


def _padded_golden(SH2, D):
    """The hand-derived example embedded in SH2 features and D states with zero padding."""
    x = hand_k2()
    f = np.float32
    out = {"tw": x["tw"]}
    h = np.zeros((1, 2, SH2), f); h[:, :, :2] = x["h_history"]
    hs = np.zeros((1, SH2), f); hs[:, :2] = x["h_s2"]
    g = np.zeros((1, SH2), f); g[:, :2] = x["d_h_enriched"]
    out.update(h_history=h, h_s2=hs, d_h_enriched=g)
    for k in ("W_A", "W_B", "W_C"):
        w = np.zeros((SH2, D), f); w[:2, :1] = x[k]; out[k] = w
    wo = np.zeros((D, SH2), f); wo[:1, :2] = x["W_O"]; out["W_O"] = wo
    exp = {}
    y = hs.copy(); y[:, :2] = x["h_enriched"]; exp["h_enriched"] = y
    dh = np.zeros((1, 2, SH2)); dh[:, :, :2] = x["d_h_history"]; exp["d_h_history"] = dh
    dhs = g.astype(np.float64).copy(); dhs[:, :2] = x["d_h_s2"]; exp["d_h_s2"] = dhs
    for k in ("dW_A", "dW_B", "dW_C"):
        w = np.zeros((SH2, D)); w[:2, :1] = x[k]; exp[k] = w
    wo = np.zeros((D, SH2)); wo[:1, :2] = x["dW_O"]; exp["dW_O"] = wo
    return out, exp


@pytest.mark.parametrize("SH2,D,force", [(32, 4, False), (4, 1, False), (32, 4, True)])
def test_golden_hand_example(SH2, D, force):
    x, exp = _padded_golden(SH2, D)
    got = run_all(x, force_generic=force)
    for n in NAMES:
        np.testing.assert_allclose(got[n], exp[n], rtol=0, atol=1e-6, err_msg=n)


def test_bwd_bitwise_reproducible_and_stream_independent():
    import torch
    ensure_built()
    x = make_inputs(WORKLOADS["pages"])
    d = to_dev(x)
    r1 = {k: v.clone() for k, v in run_bwd(d).items()}
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        r2 = run_bwd(d, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    r3 = run_bwd(d)
    torch.cuda.synchronize()
    for k in OUTPUTS:
        assert torch.equal(r1[k], r2[k]), k
        assert torch.equal(r1[k], r3[k]), k
    y1 = run_fwd(d).clone()
    y2 = run_fwd(d)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("B,K,SH2,D", [(8192, 8, 256, 16), (4096, 16, 512, 64)])
def test_concurrent_calls_on_two_streams(B, K, SH2, D):
    """Forward and backward calls on two streams at once, each with its own
    inputs, outputs and workspace, give the results of the same calls made
    one after another: the calls share no state."""
    import torch
    import gated_ssm_temporal_gb300 as g
    ensure_built()
    ds = [to_dev(custom(B, K, SH2, D, seed=s, tw=0.1)) for s in (31, 32)]
    wss = [g.alloc_workspace(B, K, SH2, D, "cuda") for _ in ds]

    def call(d, ws, stream=None):
        y = g.fwd(d["h_history"], d["h_s2"], d["W_A"], d["W_B"], d["W_C"], d["W_O"], d["tw"],
                  stream=stream)
        r = run_bwd(d, workspace=ws, stream=stream)
        r["h_enriched"] = y
        return r

    serial = [call(d, ws) for d, ws in zip(ds, wss)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for rep in range(5):
        outs = [None, None]
        for i in (0, 1):
            with torch.cuda.stream(streams[i]):
                outs[i] = call(ds[i], wss[i], stream=streams[i])
        torch.cuda.synchronize()
        for i in (0, 1):
            for k, v in outs[i].items():
                assert torch.equal(v, serial[i][k]), (rep, i, k)
    assert g.m2scan_read_device_flags() == 0


# one shape per kernel family: the D = 16, 4 and 8 tensor-core kernels, the
# wide-state kernels and the generic kernels, each with a ragged last tile
GUARD_SHAPES = [(153, 8, 256, 16), (153, 8, 256, 4), (153, 8, 256, 8), (155, 4, 512, 64),
                (23, 8, 36, 16)]


@pytest.mark.parametrize("B,K,SH2,D", GUARD_SHAPES)
def test_guard_bands_untouched(B, K, SH2, D):
    """Outputs and the workspace sit inside larger buffers filled with a
    sentinel (16 KB on each side); nothing outside them is written."""
    import torch
    import gated_ssm_temporal_gb300 as g
    ensure_built()
    x = custom(B, K, SH2, D, seed=3, tw=0.1)
    d = to_dev(x)
    pad = 4096
    sentinel = 12345.5

    def guarded(shape, dtype=torch.float32):
        n = int(np.prod(shape))
        buf = torch.full((n + 2 * pad,), sentinel, device="cuda", dtype=dtype)
        return buf, buf[pad:pad + n].view(*shape)

    bufs = {}
    outs = {}
    shapes = {"d_h_history": (B, K, SH2), "d_h_s2": (B, SH2), "dW_A": (SH2, D), "dW_B": (SH2, D),
              "dW_C": (SH2, D), "dW_O": (D, SH2)}
    for k, sh in shapes.items():
        bufs[k], outs[k] = guarded(sh)
    ybuf, y = guarded((B, SH2))
    wsn = g.m2scan_bwd_workspace_bytes(B, K, SH2, D) // 4
    wsbuf, ws = guarded((wsn,))
    g.fwd(d["h_history"], d["h_s2"], d["W_A"], d["W_B"], d["W_C"], d["W_O"], d["tw"], out=y)
    run_bwd(d, outs=outs, workspace=ws)
    torch.cuda.synchronize()
    for buf in list(bufs.values()) + [ybuf, wsbuf]:
        assert torch.all(buf[:pad] == sentinel) and torch.all(buf[-pad:] == sentinel)
    ref = oracle_all(x)
    got = {k: v.cpu().numpy() for k, v in outs.items()}
    got["h_enriched"] = y.cpu().numpy()
    assert_outputs(got, ref, shape_of(x), NAMES, wide=runs_wide(x, False))
    assert g.m2scan_read_device_flags() == 0


def test_guard_bands_untouched_bf16():
    """The same for the bf16 kernels: bf16 activation outputs, fp32 weight
    gradients and workspace, each inside sentinel-filled buffers."""
    import torch
    import gated_ssm_temporal_gb300 as g
    ensure_built()
    B, K, SH2, D = 153, 8, 256, 16
    d = to_dev(custom(B, K, SH2, D, seed=4, tw=0.1))
    for k in ("h_history", "h_s2", "d_h_enriched"):
        d[k] = d[k].to(torch.bfloat16)
    pad = 4096
    sentinel = 1234.0  # exact in bf16

    def guarded(shape, dtype):
        n = int(np.prod(shape))
        buf = torch.full((n + 2 * pad,), sentinel, device="cuda", dtype=dtype)
        return buf, buf[pad:pad + n].view(*shape)

    bf, f32 = torch.bfloat16, torch.float32
    shapes = {"d_h_history": ((B, K, SH2), bf), "d_h_s2": ((B, SH2), bf), "dW_A": ((SH2, D), f32),
              "dW_B": ((SH2, D), f32), "dW_C": ((SH2, D), f32), "dW_O": ((D, SH2), f32)}
    bufs, outs = {}, {}
    for k, (sh, dt) in shapes.items():
        bufs[k], outs[k] = guarded(sh, dt)
    ybuf, y = guarded((B, SH2), bf)
    wsbuf, ws = guarded((g.m2scan_bwd_workspace_bytes(B, K, SH2, D) // 4,), f32)
    args = (d["h_history"], d["h_s2"], d["W_A"], d["W_B"], d["W_C"], d["W_O"], d["tw"])
    g.fwd_bf16(*args, out=y)
    g.bwd_bf16(*args, d["d_h_enriched"], outs=outs, workspace=ws)
    torch.cuda.synchronize()
    for buf in list(bufs.values()) + [ybuf, wsbuf]:
        assert torch.all(buf[:pad] == sentinel) and torch.all(buf[-pad:] == sentinel)
    for k, v in list(outs.items()) + [("h_enriched", y)]:
        assert torch.isfinite(v.float()).all(), k
    assert g.m2scan_read_device_flags() == 0


def test_empty_batch():
    import torch
    import gated_ssm_temporal_gb300 as g
    ensure_built()
    x = custom(0, 8, 256, 16, seed=1)
    d = to_dev(x)
    y = run_fwd(d)
    assert y.shape == (0, 256)
    outs = g.alloc_bwd_outputs(0, 8, 256, 16, "cuda")
    for k in ("dW_A", "dW_B", "dW_C", "dW_O"):
        outs[k].fill_(7.0)
    run_bwd(d, outs=outs)
    torch.cuda.synchronize()
    for k in ("dW_A", "dW_B", "dW_C", "dW_O"):
        assert torch.all(outs[k] == 0)


def test_launch_counts():
    import gated_ssm_temporal_gb300 as g
    ensure_built()
    d = to_dev(custom(64, 8, 256, 16, seed=2))
    run_fwd(d)
    assert g.m2scan_last_launch_count() == 1
    run_bwd(d)
    assert g.m2scan_last_launch_count() == 2
    # wide-state family: the weights' split, tile kernel, d_h_s2,
    # weight-gradient products, slot sum
    d = to_dev(custom(70, 4, 256, 64, seed=2))
    run_bwd(d)
    assert g.m2scan_last_launch_count() == 5


def test_no_device_wait_timeouts():
    import gated_ssm_temporal_gb300 as g
    ensure_built()
    run_all(custom(64, 8, 256, 16, seed=4))
    assert g.m2scan_read_device_flags() == 0


def test_calls_from_a_new_host_thread():
    # a host thread that has made no CUDA runtime call yet (autograd's backward
    # runs on one): the library makes the device's context current itself
    import threading
    x = custom(300, 8, 256, 16, seed=21)
    ref = oracle_all(x)
    res = {}

    def work():
        try:
            res["got"] = run_all(x)
        except Exception as e:  # reported below, on the test's thread
            res["err"] = e

    th = threading.Thread(target=work)
    th.start()
    th.join()
    assert "err" not in res, res.get("err")
    assert_outputs(res["got"], ref, shape_of(x), NAMES)
