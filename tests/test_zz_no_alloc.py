"""m2scan_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: code whose device memory belongs to a
host framework's pool, latency-critical paths that cannot take cudaMalloc's
implicit synchronisation, minimal C hosts that only own their tensors. For
them the library keeps the backward's weight-gradient scratch in a static
device array. These tests call that entry point through the C ABI, twice in a
row. It runs the same kernels with the same sample-to-slot assignment as
m2scan_bwd, so each call's six outputs must equal m2scan_bwd's bit for bit; on
the 8192-sample workload they are also checked against the fp64 oracle with
the parity criteria the other tests use, and no kernel may have given up on a
barrier wait. This file is collected last on purpose.
"""
import numpy as np
import pytest

import gated_ssm_temporal_gb300 as g
from gated_ssm_temporal_gb300.workloads import WORKLOADS, make_inputs
from gpu_helpers import OUTPUTS, ensure_built, oracle_all, run_bwd, shape_of, to_dev
from tolerance import assert_outputs

pytestmark = pytest.mark.gpu


def _noalloc(d, outs):
    B, K, SH2 = (int(v) for v in d["h_history"].shape)
    D = int(d["W_A"].shape[1])
    import torch
    st = g.m2scan_bwd_noalloc(
        d["h_history"].data_ptr(), d["h_s2"].data_ptr(), d["W_A"].data_ptr(), d["W_B"].data_ptr(),
        d["W_C"].data_ptr(), d["W_O"].data_ptr(), d["tw"], d["d_h_enriched"].data_ptr(),
        B, K, SH2, D, outs["d_h_history"].data_ptr(), outs["d_h_s2"].data_ptr(),
        outs["dW_A"].data_ptr(), outs["dW_B"].data_ptr(), outs["dW_C"].data_ptr(),
        outs["dW_O"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    return st


@pytest.mark.parametrize("name", ["pages", "long_history"])
def test_noalloc_matches_bwd_on_two_calls(name):
    import torch
    ensure_built()
    x = make_inputs(WORKLOADS[name])
    d = to_dev(x)
    g.m2scan_read_device_flags()  # start from clear flags
    ref = {k: v.clone() for k, v in run_bwd(d).items()}
    B, K, SH2, D = shape_of(x)
    for _ in range(2):
        outs = g.alloc_bwd_outputs(B, K, SH2, D, "cuda")
        for v in outs.values():
            v.fill_(float("nan"))
        assert _noalloc(d, outs) == g.M2SCAN_OK
        torch.cuda.synchronize()
        for k in OUTPUTS:
            assert torch.equal(outs[k], ref[k]), k
    if name == "pages":
        exact = oracle_all(x)
        assert_outputs({k: outs[k].cpu().numpy() for k in OUTPUTS}, exact, (B, K, SH2, D),
                       OUTPUTS, context={"test": "noalloc"})
    assert g.m2scan_read_device_flags() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """The wide-state shapes need 182 MB of workspace, above the 16 MiB array: the call
    returns M2SCAN_ERR_WORKSPACE before anything is launched."""
    import torch
    ensure_built()
    B, K, SH2, D = 16384, 16, 512, 64
    assert g.m2scan_bwd_workspace_bytes(B, K, SH2, D) > g.NOALLOC_SCRATCH_BYTES
    small = torch.zeros(16, device="cuda")
    p = small.data_ptr()
    st = g.m2scan_bwd_noalloc(p, p, p, p, p, p, 0.1, p, B, K, SH2, D, p, p, p, p, p, p, 0)
    assert st == 5  # M2SCAN_ERR_WORKSPACE
