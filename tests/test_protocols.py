"""The barrier protocols of the tensor-core kernels, checked on executable
models (``protocol_models``): random interleavings of every role over the
kernels' tile splits, ring depths and item counts must finish without a
deadlock, a parity alias or a buffer hazard, and each planted protocol
mistake must be caught."""
import itertools
import os
import re

import pytest

import protocol_models as pm

P = 152
CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "gated_ssm_temporal_gb300", "csrc")
# every copy-ring depth a kernel can run with: the fused kernels' plans pick
# 2 .. kMaxStages stages from the shared memory they need, the wide-state and
# bf16 kernels have fixed depths
DEPTHS = (2, 3, 4, 5, 6)
# (B, K): the layer's workload, ragged splits, a CTA with one or no sample,
# the narrowest and widest histories
SHAPES = [(8192, 8), (65536, 8), (1000, 8), (300, 16), (152, 8), (20, 8), (700, 1), (400, 128), (333, 3)]
WIDTHS = {"fwd_tc16": (256, 64, 32), "fwd_bf16": (256, 128, 64), "bwd_tc": (256, 64, 32),
          "fwd_tc": (256, 64, 32), "wide_tc_fwd": (512, 256, 128), "wide_tc_bwd": (512, 384, 128),
          "wide_tc_dw": (512, 128), "bwd_bf16": (256, 192, 64)}


@pytest.mark.parametrize("model", sorted(pm.MODELS))
def test_protocol_runs_clean(model):
    f = pm.MODELS[model]
    for (B, K), SH2, NST, cta in itertools.product(SHAPES, WIDTHS[model], DEPTHS, (0, 77, P - 1)):
        for seed in range(6):
            f(B, P, cta, K, SH2, NST, seed)


def _kernel_constant(fname, name):
    src = open(os.path.join(CSRC, fname)).read()
    found = re.findall(r"constexpr int %s = (\d+);" % name, src)
    assert len(found) == 1, (fname, name)
    return int(found[0])


def test_models_use_the_kernels_constants():
    # item sizes, hand-off rings and remainder buffers as the kernels define them
    assert pm.kRowItem == _kernel_constant("m2scan_bwd_tc.cu", "kRowItem")
    assert pm.kBwdSampleItem == _kernel_constant("m2scan_bwd_tc.cu", "kBwdSampleItem")
    for f in ("m2scan_bwd_tc.cu", "m2scan_fwd_tc16.cu"):
        assert pm.kChunkRing == _kernel_constant(f, "kChunkRing")
        assert pm.kLoBufs == _kernel_constant(f, "kLoBufs")
    # every copy-ring depth a kernel can run with is one the models run
    assert max(DEPTHS) == _kernel_constant("m2scan_internal.h", "kMaxStages")
    assert pm.kChunkRing >= max(DEPTHS)
    for f, name in (("m2scan_wide_tc.cu", "kNst"), ("m2scan_wide_tc.cu", "kDwNst"),
                    ("m2scan_bwd_bf16.cu", "kNst"), ("m2scan_fwd_bf16.cu", "kBfStages")):
        assert _kernel_constant(f, name) in DEPTHS, (f, name)


def test_tile_split_covers_the_slice():
    for B, K in SHAPES:
        S_max = min(128 // K, 16)
        total = 0
        for cta in range(P):
            sizes = pm.tiles(B, P, cta, K)
            assert all(1 <= s <= S_max for s in sizes)
            assert not sizes or max(sizes) - min(sizes) <= 1
            total += sum(sizes)
        assert total == B


def test_post_item_order_is_a_permutation():
    for nsi, nri in itertools.product(range(0, 4), range(0, 10)):
        seen = [pm.post_item(p, nsi, nri) for p in range(nsi + nri)]
        assert sorted(seen) == sorted([(1, i) for i in range(nsi)] + [(2, i) for i in range(nri)])
        if nsi and nri:
            assert seen[0] == (1, 0) and seen[1] == (2, 0)


MUTATIONS = [
    ("fwd_tc16", "no_lofree_wait"),
    ("fwd_tc16", "no_last_lofree_wait"),
    ("fwd_tc16", "no_accempty_wait"),
    ("fwd_tc16", "one_full_barrier"),
    ("fwd_bf16", "no_accempty_wait"),
    ("fwd_bf16", "no_mdone_wait"),
    ("fwd_bf16", "early_empty"),
    ("fwd_bf16", "one_full_barrier"),
    ("bwd_tc", "no_htfree_wait"),
    ("bwd_tc", "no_dhfree1_wait"),
    ("bwd_tc", "early_row_empty"),
    ("fwd_tc", "no_afree_wait"),
    ("fwd_tc", "no_accfull_wait"),
    ("fwd_tc", "early_empty"),
    ("wide_tc_fwd", "no_lo_wait"),
    ("wide_tc_fwd", "no_acc_full_wait"),
    ("wide_tc_fwd", "early_split"),
    ("wide_tc_bwd", "no_lo_wait"),
    ("wide_tc_bwd", "early_split"),
    ("wide_tc_bwd", "no_dh_full_wait"),
    ("wide_tc_bwd", "no_wlo_wait"),
    ("wide_tc_bwd", "no_wlo_free_wait"),
    ("wide_tc_bwd", "skip_dh_waits"),
    ("wide_tc_dw", "no_split_wait"),
    ("wide_tc_dw", "early_split"),
    ("wide_tc_dw", "no_done_wait"),
    ("bwd_bf16", "no_dh_free_wait"),
    ("bwd_bf16", "no_t_ready_wait"),
    ("bwd_bf16", "early_empty"),
    ("bwd_bf16", "no_dh_full_wait"),
]


@pytest.mark.parametrize("model,mutation", MUTATIONS)
def test_planted_protocol_mistake_is_caught(model, mutation):
    f = pm.MODELS[model]
    for (B, K), SH2, NST in itertools.product(SHAPES[:3], WIDTHS[model], (6, 4, 3)):
        for seed in range(4):
            try:
                f(B, P, 0, K, SH2, NST, seed, mutation=mutation)
            except (AssertionError, RuntimeError):
                return
    pytest.fail("%s: %s not detected" % (model, mutation))


# Waits the kernels keep as second guards although another wait implies
# them: dropping one must stay harmless on the whole grid. In the wide-state
# tile kernels the compute warps split the next stage only after reading the
# accumulators back (forward acc_free), after writing dA|dB into TMEM
# (dab_ready) and after reading the previous d_h block back (dh_free), and
# the MMA thread waits for every split.
IMPLIED = [("wide_tc_fwd", "no_acc_free_wait"), ("wide_tc_bwd", "no_dab_ready_wait"),
           ("wide_tc_bwd", "no_dh_free_wait")]


@pytest.mark.parametrize("model,mutation", IMPLIED)
def test_implied_wait_is_redundant(model, mutation):
    f = pm.MODELS[model]
    for (B, K), SH2, NST, cta in itertools.product(SHAPES, WIDTHS[model], (2, 4), (0, 77)):
        for seed in range(3):
            f(B, P, cta, K, SH2, NST, seed, mutation=mutation)

