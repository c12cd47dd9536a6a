"""Plant plausible mistakes in copies of the oracle and check the pins catch each.

Each mutant is a one-line textual change to ``oracle/m2scan_oracle.c`` (a
dropped term, a wrong sign, an index off by one step, a transposed operand,
the errors the pages' own backward listing makes). The mutant is compiled
into a temporary library on the CPU; at least one pin must fail on it.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "m2scan_oracle.c")

MUTANTS = {
    "gate_complement": ("xs = gs * g * xs + Bv[t * D + s];",
                        "xs = gs * (1.0 - g) * xs + Bv[t * D + s];"),
    "state_init_one": ("double xs = 0.0; /* x_{-1} = 0 */", "double xs = 1.0;"),
    "drop_B_term": ("xs = gs * g * xs + Bv[t * D + s];",
                    "xs = gs * g * xs + 0.0 * Bv[t * D + s];"),
    "ctx_without_C": ("ctx[s] = C[s] * xs;", "ctx[s] = xs;"),
    "output_no_residual": ("h_enriched[b * SH2 + j] = hs[j] + tw * o;",
                           "h_enriched[b * SH2 + j] = tw * o;"),
    "output_transposed_WO": ("o += ctx[s] * W_O[(int64_t)s * SH2 + j];",
                             "o += ctx[s] * W_O[(int64_t)(j % D) * SH2 + (s % SH2)];"),
    "dctx_without_tw": ("dctx[s] = tw * acc;", "dctx[s] = acc;"),
    "dC_without_x": ("dC[s] = dctx[s] * x[(K - 1) * D + s];", "dC[s] = dctx[s];"),
    "dx_without_C": ("double dx = dctx[s] * C[s];", "double dx = dctx[s];"),
    "dx_complement_gate": ("dx = dx * gs * gt;", "dx = dx * gs * (1.0 - gt);"),
    "sigmoid_derivative_dropped": ("dA[t * D + s] = dx * xprev * gs * gt * (1.0 - gt);",
                                   "dA[t * D + s] = dx * xprev * gs * gt;"),
    "gate_scale_dropped_forward": ("xs = gs * g * xs + Bv[t * D + s];",
                                   "xs = g * xs + Bv[t * D + s];"),
    "gate_scale_dropped_in_dA": ("dA[t * D + s] = dx * xprev * gs * gt * (1.0 - gt);",
                                 "dA[t * D + s] = dx * xprev * gt * (1.0 - gt);"),
    "gate_scale_dropped_in_dx": ("dx = dx * gs * gt;", "dx = dx * gt;"),
    "blend_without_1_over_D": ("h_enriched[b * SH2 + j] = hs[j] + w * context / D;",
                               "h_enriched[b * SH2 + j] = hs[j] + w * context;"),
    "blend_dcontext_without_w": ("dcontext += g[j] * w / D;", "dcontext += g[j] / D;"),
    "blend_dw_without_context": ("pO[j] += g[j] * context / D;", "pO[j] += g[j] / D;"),
    "blend_dC_uses_C": ("dC[s] = dcontext * x[(K - 1) * D + s];", "dC[s] = dcontext * C[s];"),
    "gate_scale_squared_in_dA": ("dA[t * D + s] = dx * xprev * gs * gt * (1.0 - gt);",
                                 "dA[t * D + s] = dx * xprev * gs * gs * gt * (1.0 - gt);"),
    "xprev_off_by_one": ("double xprev = (t > 0) ? x[(t - 1) * D + s] : 0.0;",
                         "double xprev = x[t * D + s];"),
    "dWB_uses_dA": ("sb += h[(int64_t)t * SH2 + j] * dBv[t * D + s];",
                    "sb += h[(int64_t)t * SH2 + j] * dA[t * D + s];"),
    "dWO_missing_tw": ("pO[(int64_t)s * SH2 + j] += tw * ctx[s] * g[j];",
                       "pO[(int64_t)s * SH2 + j] += ctx[s] * g[j];"),
    "dhist_swapped_weights": ("acc += dA[t * D + s] * W_A[(int64_t)j * D + s] +",
                              "acc += dA[t * D + s] * W_B[(int64_t)j * D + s] +"),
    "dhs2_no_residual": ("double acc = g[j], aacc", "double acc = 0.0, aacc"),
    "dWC_uses_dctx": ("pC[(int64_t)j * D + s] += hs[j] * dC[s];",
                      "pC[(int64_t)j * D + s] += hs[j] * dctx[s];"),
    "combine_drops_last_block": ("for (int blk = 0; blk < M2O_BLOCKS; blk++) {\n      const",
                                 "for (int blk = 0; blk < M2O_BLOCKS - 1; blk++) {\n      const"),
    # the per-element error scales (sums of |terms|)
    "abs_of_sum_over_t": ("ua += fabs(h[(int64_t)t * SH2 + j] * dA[t * D + s]);",
                          "ua = fabs(sa);"),
    "abs_dWB_uses_dA": ("ub += fabs(h[(int64_t)t * SH2 + j] * dBv[t * D + s]);",
                        "ub += fabs(h[(int64_t)t * SH2 + j] * dA[t * D + s]);"),
    "abs_dWO_missing_tw": ("qO[(int64_t)s * SH2 + j] += fabs(tw * ctx[s] * g[j]);",
                           "qO[(int64_t)s * SH2 + j] += fabs(ctx[s] * g[j]);"),
    "abs_dWC_signed": ("qC[(int64_t)j * D + s] += fabs(hs[j] * dC[s]);",
                       "qC[(int64_t)j * D + s] += hs[j] * dC[s];"),
    "abs_dh_drops_B_term": ("fabs(dBv[t * D + s] * W_B[(int64_t)j * D + s]);",
                            "0.0 * fabs(dBv[t * D + s] * W_B[(int64_t)j * D + s]);"),
    "abs_dhs2_no_residual": ("double acc = g[j], aacc = fabs(g[j]);",
                             "double acc = g[j], aacc = 0.0;"),
    "abs_out_no_residual": ("abs_out[b * SH2 + j] = fabs(hs[j]) + fabs(tw) * ao;",
                            "abs_out[b * SH2 + j] = fabs(tw) * ao;"),
    "abs_combine_drops_last_block": ("ua += p[4 * nw + e];",
                                     "ua += (blk < M2O_BLOCKS - 1) ? p[4 * nw + e] : 0.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, "mutation site not unique/found: %s" % name
    path = tmp_path / ("mutant_%s.c" % name)
    path.write_text(src.replace(before, after))
    lib = oracle.open_library(oracle.compile_source(str(path), str(tmp_path / "lib.so")))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError as e:
            caught.append("%s: %s" % (pin.__name__, str(e)[:80]))
    assert caught, "mutant %s passed every pin" % name
