"""The layer as a differentiable torch operation.

``gated_temporal_scan(h_history, h_s2, W_A, W_B, W_C, W_O, tw)`` returns
h_enriched = h_s2 + tw * ((C * x_{K-1}) @ W_O), with A = h_history @ W_A,
B = h_history @ W_B, C = h_s2 @ W_C and x_t = sigmoid(A_t) * x_{t-1} + B_t
from x_{-1} = 0 (the layer of "Custom Kernel Optimization Implementation
Plan", Tasks 1 and 2; the output step as the layer fixes it). Its backward
calls the library's fused backward, which recomputes the projections and the
scan from the saved inputs (nothing else is kept between the two passes) and
returns the gradients of all six tensor inputs; ``tw`` is a Python float and
gets no gradient.

An optional ``gate_scale`` (a one-element CUDA tensor g) multiplies every
gate, g * sigmoid(A_t), as the pages' optional gate multiplier does
("Custom Kernel Optimization Implementation Plan", Tasks 1 and 2); it is a
constant of the step and gets no gradient.

Both passes are single stream-ordered library calls on the current stream,
with no host synchronisation and no allocation outside torch's caching
allocator, so a training step that uses the operation can be captured in a
CUDA graph (``torch.cuda.graph``) once the library has been loaded and
called outside the capture.
"""
import torch

from .binding import bwd, fwd


class GatedTemporalScan(torch.autograd.Function):
    """Forward and backward of the layer through the C-ABI library."""

    @staticmethod
    def forward(ctx, h_history, h_s2, W_A, W_B, W_C, W_O, tw, gate_scale=None):
        ins = [t.contiguous() for t in (h_history, h_s2, W_A, W_B, W_C, W_O)]
        out = fwd(*ins, float(tw), stream=torch.cuda.current_stream(h_history.device),
                  gate_scale=gate_scale)
        ctx.save_for_backward(*ins)
        ctx.tw = float(tw)
        ctx.gate_scale = gate_scale
        return out

    @staticmethod
    def backward(ctx, d_h_enriched):
        h_history, h_s2, W_A, W_B, W_C, W_O = ctx.saved_tensors
        g = bwd(h_history, h_s2, W_A, W_B, W_C, W_O, ctx.tw, d_h_enriched.contiguous(),
                stream=torch.cuda.current_stream(h_history.device), gate_scale=ctx.gate_scale)
        return (g["d_h_history"], g["d_h_s2"], g["dW_A"], g["dW_B"], g["dW_C"], g["dW_O"], None,
                None)


def gated_temporal_scan(h_history, h_s2, W_A, W_B, W_C, W_O, tw, gate_scale=None):
    """h_enriched [B, SH2] of the layer, differentiable in its six tensor inputs."""
    return GatedTemporalScan.apply(h_history, h_s2, W_A, W_B, W_C, W_O, tw, gate_scale)
