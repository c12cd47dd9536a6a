"""The weight-gradient slot sum runs as a programmatic dependent of the kernel
that writes the slots and waits for that kernel's completion before it reads
them. Here the workspace is filled with NaN before each call and the inputs
change between calls, so a sum that read a slot before its writer finished
would show NaN or the previous call's partial sums. Every backward family
that feeds the slot sum is covered (needs a GB300)."""
import numpy as np
import pytest

import gated_ssm_temporal_gb300 as g
from gated_ssm_temporal_gb300.workloads import Workload, make_inputs
from gpu_helpers import ensure_built, to_dev

pytestmark = pytest.mark.gpu

DW = ("dW_A", "dW_B", "dW_C", "dW_O")

# (B, K, SH2, D, bf16, force_generic): the fp32 and bf16 tensor-core
# backwards on the layer's shape, the wide-state family, the tensor-core
# backward with D = 8 zero-padded to 16 states, and the generic per-sample
# kernel
CASES = [(8192, 8, 256, 16, False, False), (8192, 8, 256, 16, True, False),
         (1000, 4, 512, 64, False, False), (3000, 8, 128, 8, False, False),
         (500, 8, 256, 16, False, True)]


def _inputs(B, K, SH2, D, seed, bf16):
    import torch
    d = to_dev(make_inputs(Workload("custom", B, K, SH2, D, 0.3, seed, 1.0, 1.0)))
    if bf16:
        for k in ("h_history", "h_s2", "d_h_enriched"):
            d[k] = d[k].to(torch.bfloat16)
    return d


def _bwd(d, ws, bf16):
    call = g.bwd_bf16 if bf16 else g.bwd
    r = call(d["h_history"], d["h_s2"], d["W_A"], d["W_B"], d["W_C"], d["W_O"], d["tw"],
             d["d_h_enriched"], workspace=ws)
    return {k: r[k].clone() for k in DW}


@pytest.mark.parametrize("B,K,SH2,D,bf16,force_generic", CASES)
def test_slot_sum_reads_only_finished_slots(B, K, SH2, D, bf16, force_generic):
    import torch
    ensure_built()
    prev = g.m2scan_set_force_generic(1 if force_generic else 0)
    try:
        d1, d2 = _inputs(B, K, SH2, D, 11, bf16), _inputs(B, K, SH2, D, 12, bf16)
        ws = g.alloc_workspace(B, K, SH2, D, "cuda")
        fresh = _bwd(d2, torch.zeros_like(ws), bf16)
        first = None
        for rep in range(3):
            ws.fill_(float("nan"))
            a = _bwd(d1, ws, bf16)
            ws.fill_(float("nan"))
            b = _bwd(d2, ws, bf16)
            torch.cuda.synchronize()
            if first is None:
                first = a
            for k in DW:
                assert torch.isfinite(b[k]).all(), (k, rep)
                assert torch.equal(b[k], fresh[k]), (k, rep)
                assert torch.equal(a[k], first[k]), (k, rep)
                assert not torch.equal(a[k], b[k]), k
        assert g.m2scan_read_device_flags() == 0
    finally:
        g.m2scan_set_force_generic(prev)
