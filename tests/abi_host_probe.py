"""Host-only checks of the C ABI, run in a child process with no visible GPU.

Every call below must be rejected by the host-side argument checks before the
library touches CUDA. The child hides all GPUs (CUDA_VISIBLE_DEVICES=""), so
even a check that wrongly passed could not launch a kernel on the fake
addresses used here. Prints one JSON object with the observed results.
"""
import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import gated_ssm_temporal_gb300 as g  # noqa: E402

A = 1 << 32  # fake, 16-byte aligned device addresses far apart
W = [A + i * (1 << 24) for i in range(20)]
B, K, SH2, D = 8, 8, 32, 4
res = {}


def fwd(**kw):
    args = dict(h_history=W[0], h_s2=W[1], W_A=W[2], W_B=W[3], W_C=W[4], W_O=W[5], tw=0.5,
                B=B, K=K, SH2=SH2, D=D, h_enriched=W[6], stream=0)
    args.update(kw)
    return g.m2scan_fwd(**args)


def bwd(**kw):
    ws = g.m2scan_bwd_workspace_bytes(B, K, SH2, D)
    args = dict(h_history=W[0], h_s2=W[1], W_A=W[2], W_B=W[3], W_C=W[4], W_O=W[5], tw=0.5,
                d_h_enriched=W[7], B=B, K=K, SH2=SH2, D=D, d_h_history=W[8], d_h_s2=W[9],
                dW_A=W[10], dW_B=W[11], dW_C=W[12], dW_O=W[13], workspace=W[14],
                workspace_bytes=ws, stream=0)
    args.update(kw)
    return g.m2scan_bwd(**args)


res["fwd_null_WA"] = fwd(W_A=0)
res["fwd_null_h"] = fwd(h_history=0)
res["fwd_null_out"] = fwd(h_enriched=0)
res["fwd_B_neg"] = fwd(B=-1)
res["fwd_K0"] = fwd(K=0)
res["fwd_SH2_not4"] = fwd(SH2=30)
res["fwd_SH2_small"] = fwd(SH2=0)
res["fwd_D0"] = fwd(D=0)
res["fwd_misaligned_h"] = fwd(h_history=W[0] + 4)
res["fwd_misaligned_out"] = fwd(h_enriched=W[6] + 8)
res["fwd_alias_out_h"] = fwd(h_enriched=W[0] + 64)
res["fwd_alias_out_WO"] = fwd(h_enriched=W[5])
res["fwdex_misaligned_gs"] = g.m2scan_fwd_ex(W[0], W[1], W[2], W[3], W[4], W[5], 0.5, W[18] + 2,
                                          B, K, SH2, D, W[6], 0)
res["fwdex_alias_gs_out"] = g.m2scan_fwd_ex(W[0], W[1], W[2], W[3], W[4], W[5], 0.5, W[6] + 8,
                                         B, K, SH2, D, W[6], 0)
res["fwd_B0_ok"] = fwd(B=0, h_history=0, h_s2=0, h_enriched=0)
res["fwd_launches_B0"] = g.m2scan_last_launch_count()
res["bwdex_alias_gs_dWA"] = g.m2scan_bwd_ex(
    W[0], W[1], W[2], W[3], W[4], W[5], 0.5, W[10] + 4, W[7], B, K, SH2, D, W[8], W[9], W[10],
    W[11], W[12], W[13], W[14], g.m2scan_bwd_workspace_bytes(B, K, SH2, D), 0)
res["bwd_null_ws"] = bwd(workspace=0)
res["bwd_short_ws"] = bwd(workspace_bytes=g.m2scan_bwd_workspace_bytes(B, K, SH2, D) - 16)
res["bwd_null_dWO"] = bwd(dW_O=0)
res["bwd_null_g"] = bwd(d_h_enriched=0)
res["bwd_shape"] = bwd(K=-3)
res["bwd_misaligned_ws"] = bwd(workspace=W[14] + 4)
res["bwd_alias_out_out"] = bwd(dW_B=W[10] + 16)
res["bwd_alias_ws_in"] = bwd(workspace=W[0])
res["bwd_alias_dh_g"] = bwd(d_h_history=W[7])
res["ws_bytes_pages"] = g.m2scan_bwd_workspace_bytes(8192, 8, 256, 16)
res["ws_bytes_small_B"] = g.m2scan_bwd_workspace_bytes(3, 8, 256, 16)
res["ws_bytes_B0"] = g.m2scan_bwd_workspace_bytes(0, 8, 256, 16)
res["ws_bytes_wide"] = g.m2scan_bwd_workspace_bytes(16384, 16, 512, 64)
res["ws_bytes_bad"] = g.m2scan_bwd_workspace_bytes(5, 0, 256, 16)
res["path_pages"] = g.m2scan_path_for(8, 256, 16)
res["path_long"] = g.m2scan_path_for(64, 256, 16)
res["path_tiny"] = g.m2scan_path_for(8, 32, 4)
res["path_wide"] = g.m2scan_path_for(16, 512, 64)
res["path_K129"] = g.m2scan_path_for(129, 256, 16)
res["path_huge"] = g.m2scan_path_for(100000, 256, 64)
res["fwd_path_pages"] = g.m2scan_fwd_path_for(8, 256, 16)
res["fwd_path_wide"] = g.m2scan_fwd_path_for(16, 512, 64)
res["fwd_path_K129"] = g.m2scan_fwd_path_for(129, 256, 16)
res["fwd_path_huge"] = g.m2scan_fwd_path_for(100000, 256, 64)
# every shape of the fused kernels' range (D in {4, 8, 16}, SH2 a multiple of
# 32 up to 256, K up to 128): the family each direction takes
res["fused_range"] = sorted({(g.m2scan_fwd_path_for(k, s, d), g.m2scan_path_for(k, s, d))
                             for k in range(1, 129) for s in range(32, 257, 32) for d in (4, 8, 16)})


def bias(**kw):
    N, C = kw.pop("N", 100), kw.pop("C", 7)
    args = dict(dy=W[15], N=N, C=C, db=W[16], accumulate=0, workspace=W[17],
                workspace_bytes=g.m2scan_bias_grad_workspace_bytes(N, C), stream=0)
    args.update(kw)
    return g.m2scan_bias_grad(**args)


res["bg_null_db"] = bias(db=0)
res["bg_null_dy"] = bias(dy=0)
res["bg_C0"] = bias(C=0)
res["bg_N_neg"] = bias(N=-1)
res["bg_misaligned_dy"] = bias(dy=W[15] + 4)
res["bg_misaligned_db"] = bias(db=W[16] + 8)
res["bg_null_ws"] = bias(workspace=0)
res["bg_short_ws"] = bias(workspace_bytes=g.m2scan_bias_grad_workspace_bytes(100, 7) - 4)
res["bg_misaligned_ws"] = bias(workspace=W[17] + 4)
res["bg_alias_db_dy"] = bias(db=W[15] + 32)
res["bg_alias_ws_dy"] = bias(workspace=W[15] + 16)
res["bg_alias_db_ws"] = bias(db=W[17])
res["bg_ws_pages"] = g.m2scan_bias_grad_workspace_bytes(8192, 256)
res["bg_ws_one"] = g.m2scan_bias_grad_workspace_bytes(1, 3)
res["bg_ws_N0"] = g.m2scan_bias_grad_workspace_bytes(0, 5)
res["bg_ws_big"] = g.m2scan_bias_grad_workspace_bytes(100000, 7)
res["bg_ws_bad"] = g.m2scan_bias_grad_workspace_bytes(10, 0)
res["bl_fwd_null_ws"] = g.m2scan_fwd_blend(W[0], W[1], W[2], W[3], W[4], W[18], 0, B, K, SH2, D,
                                          W[6], 0, 0, 0)
res["bl_fwd_misaligned_w"] = g.m2scan_fwd_blend(W[0], W[1], W[2], W[3], W[4], W[18] + 4, 0, B, K,
                                               SH2, D, W[6], W[19], 1 << 20, 0)
res["bl_fwd_alias_ws_out"] = g.m2scan_fwd_blend(W[0], W[1], W[2], W[3], W[4], W[18], 0, B, K, SH2,
                                               D, W[6], W[6], 1 << 20, 0)
res["bl_bwd_short_ws"] = g.m2scan_bwd_blend(
    W[0], W[1], W[2], W[3], W[4], W[18], 0, W[7], B, K, SH2, D, W[8], W[9], W[10], W[11], W[12],
    W[13], W[14], g.m2scan_blend_bwd_workspace_bytes(B, K, SH2, D) - 16, 0)
res["bl_bwd_alias_dw_ws"] = g.m2scan_bwd_blend(
    W[0], W[1], W[2], W[3], W[4], W[18], 0, W[7], B, K, SH2, D, W[8], W[9], W[10], W[11], W[12],
    W[14] + 64, W[14], g.m2scan_blend_bwd_workspace_bytes(B, K, SH2, D), 0)
res["bl_ws_fwd"] = g.m2scan_blend_fwd_workspace_bytes(256, 16)
res["bl_ws_bwd"] = g.m2scan_blend_bwd_workspace_bytes(8192, 8, 256, 16)
res["bf16_B0_ok"] = g.m2scan_fwd_bf16(0, 0, W[2], W[3], W[4], W[5], 0.1, 0, 0, 8, 256, 16, 0, 0)
res["bf16_sh2_96"] = g.m2scan_fwd_bf16(W[0], W[1], W[2], W[3], W[4], W[5], 0.1, 0, 8, 8, 96, 16,
                                       W[6], 0)
res["bf16_d8"] = g.m2scan_fwd_bf16(W[0], W[1], W[2], W[3], W[4], W[5], 0.1, 0, 8, 8, 256, 8, W[6], 0)
res["bf16_misaligned"] = g.m2scan_fwd_bf16(W[0] + 2, W[1], W[2], W[3], W[4], W[5], 0.1, 0, 8, 8,
                                           256, 16, W[6], 0)
res["bf16_alias"] = g.m2scan_fwd_bf16(W[0], W[1], W[2], W[3], W[4], W[5], 0.1, 0, 8, 8, 256, 16,
                                      W[0] + 1024, 0)
def bwd_bf16(**kw):
    ws = g.m2scan_bwd_workspace_bytes(B, K, SH2, D)
    args = dict(h_history=W[0], h_s2=W[1], W_A=W[2], W_B=W[3], W_C=W[4], W_O=W[5], tw=0.5,
                gate_scale=0, d_h_enriched=W[7], B=B, K=K, SH2=SH2, D=D, d_h_history=W[8],
                d_h_s2=W[9], dW_A=W[10], dW_B=W[11], dW_C=W[12], dW_O=W[13], workspace=W[14],
                workspace_bytes=ws, stream=0)
    args.update(kw)
    return g.m2scan_bwd_bf16(**args)


res["bf16b_null_ws"] = bwd_bf16(workspace=0)
res["bf16b_short_ws"] = bwd_bf16(workspace_bytes=g.m2scan_bwd_workspace_bytes(B, K, SH2, D) - 16)
res["bf16b_null_dWC"] = bwd_bf16(dW_C=0)
res["bf16b_null_g"] = bwd_bf16(d_h_enriched=0)
res["bf16b_shape"] = bwd_bf16(SH2=6)
res["bf16b_misaligned_h"] = bwd_bf16(h_history=W[0] + 2)
res["bf16b_misaligned_gs"] = bwd_bf16(gate_scale=W[18] + 2)
res["bf16b_alias_dhs2_hs2"] = bwd_bf16(d_h_s2=W[1] + 16)
res["bf16b_alias_ws_dWA"] = bwd_bf16(workspace=W[10])
res["bf16b_alias_gs_dh"] = bwd_bf16(gate_scale=W[8] + 4)

res["status_str_ok"] = g.m2scan_status_str(0)
print(json.dumps(res))
