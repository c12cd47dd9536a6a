"""The C-ABI library loads, exports what include/m2scan.h declares, and rejects
bad arguments on the host (no GPU needed)."""
import json
import os
import subprocess
import sys

import pytest

import gated_ssm_temporal_gb300 as g
from gated_ssm_temporal_gb300 import build as gbuild

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return g.load_library()


def test_exports_every_header_function(lib):
    names = g.header_functions()
    assert "m2scan_fwd" in names and "m2scan_bwd" in names
    for n in names:
        assert hasattr(lib, n), "libm2scan.so does not export %s" % n


def test_library_built_for_sm103a(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", gbuild.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    for n in g.header_functions():
        assert (" T %s" % n) in out


@pytest.fixture(scope="module")
def probe(lib):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(HERE, "abi_host_probe.py")], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    return json.loads(r.stdout.strip().splitlines()[-1])


NULL, SHAPE, ALIGN, ALIAS, WORKSPACE = 1, 2, 3, 4, 5


@pytest.mark.parametrize("key,expect", [
    ("fwd_null_WA", NULL), ("fwd_null_h", NULL), ("fwd_null_out", NULL), ("fwd_B_neg", SHAPE),
    ("fwd_K0", SHAPE), ("fwd_SH2_not4", SHAPE), ("fwd_SH2_small", SHAPE), ("fwd_D0", SHAPE),
    ("fwd_misaligned_h", ALIGN), ("fwd_misaligned_out", ALIGN), ("fwd_alias_out_h", ALIAS),
    ("fwd_alias_out_WO", ALIAS), ("fwd_B0_ok", 0), ("fwd_launches_B0", 0),
    ("fwdex_misaligned_gs", ALIGN), ("fwdex_alias_gs_out", ALIAS), ("bwdex_alias_gs_dWA", ALIAS),
    ("bwd_null_ws", WORKSPACE), ("bwd_short_ws", WORKSPACE), ("bwd_null_dWO", NULL),
    ("bwd_null_g", NULL), ("bwd_shape", SHAPE), ("bwd_misaligned_ws", ALIGN),
    ("bwd_alias_out_out", ALIAS), ("bwd_alias_ws_in", ALIAS), ("bwd_alias_dh_g", ALIAS),
    ("bg_null_db", NULL), ("bg_null_dy", NULL), ("bg_C0", SHAPE), ("bg_N_neg", SHAPE),
    ("bg_misaligned_dy", ALIGN), ("bg_misaligned_db", ALIGN), ("bg_null_ws", WORKSPACE),
    ("bg_short_ws", WORKSPACE), ("bg_misaligned_ws", ALIGN), ("bg_alias_db_dy", ALIAS),
    ("bg_alias_ws_dy", ALIAS), ("bg_alias_db_ws", ALIAS),
    ("bl_fwd_null_ws", WORKSPACE), ("bl_fwd_misaligned_w", ALIGN), ("bl_fwd_alias_ws_out", ALIAS),
    ("bl_bwd_short_ws", WORKSPACE), ("bl_bwd_alias_dw_ws", ALIAS),
    ("bf16_B0_ok", 0), ("bf16_sh2_96", 6), ("bf16_d8", 6), ("bf16_misaligned", ALIGN),
    ("bf16_alias", ALIAS),
    ("bf16b_null_ws", WORKSPACE), ("bf16b_short_ws", WORKSPACE), ("bf16b_null_dWC", NULL),
    ("bf16b_null_g", NULL), ("bf16b_shape", SHAPE), ("bf16b_misaligned_h", ALIGN),
    ("bf16b_misaligned_gs", ALIGN), ("bf16b_alias_dhs2_hs2", ALIAS), ("bf16b_alias_ws_dWA", ALIAS),
    ("bf16b_alias_gs_dh", ALIAS),
])
def test_host_validation(probe, key, expect):
    assert probe[key] == expect, (key, probe[key])


def test_workspace_query(probe):
    assert probe["ws_bytes_pages"] == 152 * 4 * 256 * 16 * 4
    assert probe["ws_bytes_small_B"] == 3 * 4 * 256 * 16 * 4
    assert probe["ws_bytes_B0"] == 0
    assert probe["ws_bytes_bad"] == 0
    # wide states: 152 sample-range slots, dA|dB [B*K][128], [dC | ctx] [B][128]
    # and the split weights (tf32 parts and remainders of W_A and W_B)
    assert probe["ws_bytes_wide"] == (152 * 4 * 512 * 64 + 16384 * 16 * 128 + 16384 * 128 + 4 * 512 * 64) * 4


def test_bias_grad_workspace_query(probe):
    # one partial per column for each range of about 16 rows, at most 152 ranges
    assert probe["bg_ws_pages"] == 152 * 256 * 4
    assert probe["bg_ws_one"] == 1 * 3 * 4
    assert probe["bg_ws_N0"] == 0
    assert probe["bg_ws_big"] == 152 * 7 * 4
    assert probe["bg_ws_bad"] == 0


def test_blend_workspace_query(probe):
    # W_O = w / D broadcast to [D, SH2]; the backward adds it and dW_O to its own workspace
    assert probe["bl_ws_fwd"] == 16 * 256 * 4
    assert probe["bl_ws_bwd"] == probe["ws_bytes_pages"] + 2 * 16 * 256 * 4


def test_path_choice(probe):
    assert probe["path_pages"] == 1
    assert probe["path_long"] == 1
    assert probe["path_tiny"] == 1
    assert probe["path_wide"] == 3
    assert probe["path_K129"] == 2
    assert probe["path_huge"] == 0
    assert probe["fwd_path_pages"] == 1
    assert probe["fwd_path_wide"] == 3
    assert probe["fwd_path_K129"] == 2
    assert probe["fwd_path_huge"] == 0


def test_fused_range_has_tensor_core_plans_in_both_directions(probe):
    # every shape the fused kernels take has a tensor-core plan that fits in
    # 227 KB of shared memory, forward and backward (the library keeps no
    # other kernel for these shapes)
    assert probe["fused_range"] == [[1, 1]]
    assert probe["status_str_ok"] == "ok"
