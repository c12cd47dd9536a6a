"""Seeded random shapes through every kernel family against the oracle.

The shapes are drawn once from a fixed seed: D from the fused family's
states (4, 8, 16), the wide-state family's 64 and the generic kernels' other
sizes; SH2 a multiple of 32 (fused), of 128 (wide state) or of 4 (generic);
K from 1 to 128; B from 1 to a size that keeps the oracle's work small. Each
case runs the forward and the backward on the GPU and compares all seven
outputs with the oracle element by element (needs a GB300)."""
import random

import pytest

import gated_ssm_temporal_gb300 as g
from gated_ssm_temporal_gb300.workloads import Workload, make_inputs
from gpu_helpers import ensure_built, oracle_all, run_all, runs_wide, shape_of
from test_parity_gpu import NAMES
from tolerance import assert_outputs

pytestmark = pytest.mark.gpu

WORK_LIMIT = 2.5e7  # B * K * SH2 * D of one case: the oracle stays well under a second


def _draw(rng):
    family = rng.choice(["fused", "fused", "fused", "wide", "generic"])
    if family == "fused":
        D, SH2 = rng.choice([4, 8, 16]), 32 * rng.randint(1, 8)
    elif family == "wide":
        D, SH2 = 64, 128 * rng.randint(1, 4)
    else:
        D, SH2 = rng.choice([1, 2, 3, 5, 12, 24, 32]), 4 * rng.randint(1, 80)
    K = rng.choice([1, 2, 3, 5, 7, 8, 9, 16, 31, 33, 64, 100, 128])
    b_max = max(1, min(400, int(WORK_LIMIT // (K * SH2 * D))))
    B = rng.randint(1, b_max)
    return family, B, K, SH2, D


_rng = random.Random(20261202)
CASES = [_draw(_rng) for _ in range(24)]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_random_shape_matches_oracle(case):
    family, B, K, SH2, D = CASES[case]
    ensure_built()
    expect = {"fused": 1, "wide": 3, "generic": 2}[family]
    assert g.m2scan_path_for(K, SH2, D) == expect, CASES[case]
    assert g.m2scan_fwd_path_for(K, SH2, D) == expect, CASES[case]
    x = make_inputs(Workload("fuzz", B, K, SH2, D, 0.3, 1000 + case, 2.0, 1.0))
    got = run_all(x)
    ref = oracle_all(x)
    assert_outputs(got, ref, shape_of(x), NAMES, wide=runs_wide(x),
                   context={"test": "fuzz %s B=%d K=%d SH2=%d D=%d" % (family, B, K, SH2, D),
                            "generic": False})
    assert g.m2scan_read_device_flags() == 0
