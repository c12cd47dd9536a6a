"""Seeded synthetic inputs for the gated temporal scan layer.

This module holds no arithmetic of the layer itself: it only draws random
numbers and applies the scalings that define each workload. Both the oracle
tests and the CUDA path take their inputs from here.

Recipe (numpy PCG64, ``default_rng(seed)``, float32 standard normals, drawn in
this order): h_history [B,K,SH2], h_s2 [B,SH2], W_A, W_B, W_C [SH2,D],
W_O [D,SH2], d_h_enriched [B,SH2]. Weights are then multiplied by
1/sqrt(fan_in) (fan_in = SH2 for W_A, W_B, W_C and D for W_O). Per-workload
extras: ``long_history`` multiplies W_A by 4 (gate pre-activations of about
+-6, a mix of saturated and open gates); ``stress`` multiplies h_history of
every odd sample by 10 (heavy-tailed activations for half of the batch).

The pages' workload is the hidden state of a futures-trading DQN trunk
(SH2=256, STATE_D=16, K=8, batch 8192); that data is not available, so
Gaussian stand-ins with the same shapes are used.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    K: int
    SH2: int
    D: int
    tw: float
    seed: int
    wa_scale: float = 1.0
    odd_history_scale: float = 1.0

    def shapes(self):
        return dict(B=self.B, K=self.K, SH2=self.SH2, D=self.D)

    def with_batch(self, B: int, seed: int | None = None) -> "Workload":
        return Workload(self.name, B, self.K, self.SH2, self.D, self.tw,
                        self.seed if seed is None else seed, self.wa_scale,
                        self.odd_history_scale)


# The five workloads of the layer, by what they are.
WORKLOADS = {
    "tiny": Workload("tiny", B=4, K=8, SH2=32, D=4, tw=0.5, seed=0),
    "pages": Workload("pages", B=8192, K=8, SH2=256, D=16, tw=0.1, seed=1),
    "long_history": Workload("long_history", B=2048, K=64, SH2=256, D=16, tw=0.1,
                             seed=2, wa_scale=4.0),
    "wide_state": Workload("wide_state", B=16384, K=16, SH2=512, D=64, tw=0.1, seed=3),
    "stress": Workload("stress", B=65536, K=8, SH2=256, D=16, tw=0.1, seed=4,
                       odd_history_scale=10.0),
}

WORKLOAD_ORDER = ["tiny", "pages", "long_history", "wide_state", "stress"]


def make_inputs(w: Workload) -> dict:
    """Draw the float32 inputs of workload ``w`` (all C-contiguous numpy arrays)."""
    rng = np.random.default_rng(w.seed)
    B, K, SH2, D = w.B, w.K, w.SH2, w.D
    f32 = np.float32
    h_history = rng.standard_normal((B, K, SH2), dtype=f32)
    h_s2 = rng.standard_normal((B, SH2), dtype=f32)
    W_A = rng.standard_normal((SH2, D), dtype=f32)
    W_B = rng.standard_normal((SH2, D), dtype=f32)
    W_C = rng.standard_normal((SH2, D), dtype=f32)
    W_O = rng.standard_normal((D, SH2), dtype=f32)
    d_h_enriched = rng.standard_normal((B, SH2), dtype=f32)
    s_in = f32(1.0 / np.sqrt(SH2))
    W_A *= s_in
    W_B *= s_in
    W_C *= s_in
    W_O *= f32(1.0 / np.sqrt(D))
    if w.wa_scale != 1.0:
        W_A *= f32(w.wa_scale)
    if w.odd_history_scale != 1.0:
        h_history[1::2] *= f32(w.odd_history_scale)
    return dict(h_history=h_history, h_s2=h_s2, W_A=W_A, W_B=W_B, W_C=W_C, W_O=W_O,
                d_h_enriched=d_h_enriched, tw=float(w.tw))


def algorithmic_bytes(B: int, K: int, SH2: int, elem: int = 4) -> dict:
    """HBM bytes the layer must move per call (weights excluded), with
    activations of ``elem`` bytes (4: fp32, 2: bf16).

    forward reads h_history and h_s2 and writes h_enriched: elem*SH2*(K+2) per
    sample; backward reads h_history, h_s2 and d_h_enriched and writes
    d_h_history and d_h_s2: elem*SH2*(2K+3) per sample.
    """
    fwd = elem * SH2 * (K + 2) * B
    bwd = elem * SH2 * (2 * K + 3) * B
    return dict(fwd=fwd, bwd=bwd, total=fwd + bwd)


def algorithmic_flops(B: int, K: int, SH2: int, D: int) -> dict:
    """Floating-point operations of the method per call (a multiply-add
    counts 2): forward 4*SH2*D*(K+1) per sample (the A|B projections over K
    steps and C, then context . W_O), backward with the projections
    recomputed 2*SH2*D*(6K+5) per sample (A|B again, d_h_history, dW_A|dW_B,
    d_ctx, dW_O, dW_C, d_h_s2). The scan's O(K*D) work is left out."""
    fwd = 4 * SH2 * D * (K + 1) * B
    bwd = 2 * SH2 * D * (6 * K + 5) * B
    return dict(fwd=fwd, bwd=bwd, total=fwd + bwd)


# The bias-gradient column sum: the per-output-feature gradient dy [N, C] of
# a fully connected layer of the pages' network ("Phase 3 Kernel Optimization
# Implementation Plan": batch 8192, out_dim from 3 to 256 for the main
# network, 42 and 128 for the curiosity module). Same generator: PCG64
# ``default_rng(seed)`` float32 standard normals, one [N, C] draw.
@dataclass(frozen=True)
class BiasWorkload:
    name: str
    N: int
    C: int
    seed: int


BIAS_WORKLOADS = {
    "bias_fc": BiasWorkload("bias_fc", N=8192, C=256, seed=11),
    "bias_narrow": BiasWorkload("bias_narrow", N=8192, C=3, seed=12),
    "bias_curiosity_out": BiasWorkload("bias_curiosity_out", N=8192, C=42, seed=13),
    "bias_curiosity_hidden": BiasWorkload("bias_curiosity_hidden", N=8192, C=128, seed=14),
}


def make_bias_input(N: int, C: int, seed: int):
    """dy [N, C] float32 standard normals (C-contiguous)."""
    return np.random.default_rng(seed).standard_normal((N, C), dtype=np.float32)
