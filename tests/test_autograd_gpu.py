"""The layer as a torch autograd operation, eagerly and inside a CUDA graph."""
import numpy as np
import pytest

from gated_ssm_temporal_gb300.workloads import Workload, make_inputs
from gpu_helpers import ensure_built, oracle_all, runs_wide, shape_of, to_dev
from tolerance import assert_outputs

pytestmark = pytest.mark.gpu

GRADS = {"h_history": "d_h_history", "h_s2": "d_h_s2", "W_A": "dW_A", "W_B": "dW_B",
         "W_C": "dW_C", "W_O": "dW_O"}


def _leaves(d):
    return {k: d[k].detach().clone().requires_grad_(True) for k in GRADS}


@pytest.mark.parametrize("B,K,SH2,D", [(300, 8, 256, 16), (64, 16, 512, 64), (37, 5, 64, 8)])
def test_autograd_matches_oracle(B, K, SH2, D):
    import torch
    from gated_ssm_temporal_gb300.autograd import gated_temporal_scan
    ensure_built()
    x = make_inputs(Workload("custom", B, K, SH2, D, 0.3, B + K, 1.0, 1.0))
    d = to_dev(x)
    leaves = _leaves(d)
    y = gated_temporal_scan(*(leaves[k] for k in GRADS), d["tw"])
    y.backward(d["d_h_enriched"])
    ref = oracle_all(x)
    got = {name: leaves[k].grad.cpu().numpy() for k, name in GRADS.items()}
    got["h_enriched"] = y.detach().cpu().numpy()
    assert_outputs(got, ref, shape_of(x), list(got), wide=runs_wide(x))


def test_autograd_with_gate_multiplier():
    import torch
    from gated_ssm_temporal_gb300.autograd import gated_temporal_scan
    ensure_built()
    x = make_inputs(Workload("custom", 200, 8, 256, 16, 0.3, 9, 1.0, 1.0))
    d = to_dev(x)
    leaves = _leaves(d)
    gs = torch.tensor([0.8], device="cuda")
    y = gated_temporal_scan(*(leaves[k] for k in GRADS), d["tw"], gs)
    y.backward(d["d_h_enriched"])
    ref = oracle_all(x, gate_scale=0.8)
    got = {name: leaves[k].grad.cpu().numpy() for k, name in GRADS.items()}
    got["h_enriched"] = y.detach().cpu().numpy()
    assert_outputs(got, ref, shape_of(x), list(got))


def test_cuda_graph_replays_the_eager_step():
    import torch
    from gated_ssm_temporal_gb300.autograd import gated_temporal_scan
    ensure_built()
    x = make_inputs(Workload("custom", 1000, 8, 256, 16, 0.1, 11, 1.0, 1.0))
    d = to_dev(x)
    leaves = _leaves(d)

    def step():
        for t in leaves.values():
            t.grad = None
        y = gated_temporal_scan(*(leaves[k] for k in GRADS), d["tw"])
        y.backward(d["d_h_enriched"])
        return y

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):  # loads the library and its kernels outside the capture
            y_eager = step().detach().clone()
    torch.cuda.current_stream().wait_stream(s)
    eager = {k: v.grad.detach().clone() for k, v in leaves.items()}
    for t in leaves.values():
        t.grad = None
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        y_graph = gated_temporal_scan(*(leaves[k] for k in GRADS), d["tw"])
        y_graph.backward(d["d_h_enriched"])
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(y_graph, y_eager)
    for k, v in leaves.items():
        # the weight gradients are summed in a fixed order: bit-identical
        assert torch.equal(v.grad, eager[k]), k
